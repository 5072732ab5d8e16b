"""Split-KV flash attention forward for GB300 (sm_103a).

Thin ctypes binding over the C ABI in include/sk_attn.h (libskattn.so, built
in-tree by split_kv_flash_gb300/build.py).  The functions named like the C
entry points (sk_attn_plan, sk_attn_fwd, ...) only marshal arguments; every
step of the computation runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams only.  There is no CPU fallback: any entry point
called without the built library raises ImportError, and sk_attn_fwd on a
machine without an sm_103 GPU returns an error status (raised as SKError).
"""
import ctypes
import os

__all__ = [
    "SKError", "Opts", "PlanInfo", "lib", "sk_attn_plan", "sk_attn_plan_ranges", "sk_attn_fwd",
    "sk_attn_read_plan_echo", "sk_attn_workspace_status", "sk_attn_status_string",
    "sk_attn_fwd_noalloc", "sk_attn_noalloc_status", "NOALLOC_SCRATCH_BYTES",
    "sk_attn_last_error", "sk_attn_version", "attn_fwd", "SK_OK", "SK_PATH_DECODE",
    "SK_PATH_PREFILL", "SK_PATH_LATENT", "SK_PATH_LINEAR_RECURRENT", "SK_PATH_LINEAR_CHUNK", "sk_attn_plan_latent", "sk_attn_fwd_latent", "attn_fwd_latent",
    "LATENT_DQK", "LATENT_DV", "LinearAttnInfo", "sk_linear_attn_plan", "sk_linear_attn_fwd",
    "linear_attn_fwd", "LINEAR_ATTN_DIM", "SK_COMBINE_AUTO", "SK_COMBINE_KERNEL", "SK_COMBINE_IN_KERNEL", "SK_SCHEDULE_AUTO",
    "SK_SCHEDULE_ONE_TILE", "SK_SCHEDULE_PERSISTENT", "SK_TILE_MAP_AUTO", "SK_TILE_MAP_GRID", "SK_TILE_MAP_PACKED", "SK_POLICY_FILL", "SK_POLICY_FA_HEURISTIC", "SK_POLICY_FIXED_CHUNK",
    "SK_POLICY_MIN_CHUNK",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libskattn.so")

SK_OK, SK_ERR_INVALID_ARG, SK_ERR_UNSUPPORTED, SK_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3
SK_ERR_MISALIGNED, SK_ERR_CUDA, SK_ERR_DEVICE_TIMEOUT = 4, 5, 6
SK_POLICY_DEFAULT, SK_POLICY_FILL, SK_POLICY_FA_HEURISTIC = 0, 1, 2
SK_POLICY_FIXED_CHUNK, SK_POLICY_MIN_CHUNK = 3, 4
SK_PATH_AUTO, SK_PATH_DECODE, SK_PATH_PREFILL, SK_PATH_LATENT = 0, 1, 2, 3
SK_PATH_LINEAR_RECURRENT, SK_PATH_LINEAR_CHUNK = 4, 5
LATENT_DQK, LATENT_DV = 576, 512  # latent attention: 512 latent + 64 rotary key columns, 512 value columns
SK_COMBINE_AUTO, SK_COMBINE_KERNEL, SK_COMBINE_IN_KERNEL = 0, 1, 2
SK_SCHEDULE_AUTO, SK_SCHEDULE_ONE_TILE, SK_SCHEDULE_PERSISTENT = 0, 1, 2
SK_TILE_MAP_AUTO, SK_TILE_MAP_GRID, SK_TILE_MAP_PACKED = 0, 1, 2
NOALLOC_SCRATCH_BYTES = 16 << 20  # SK_NOALLOC_SCRATCH_BYTES in include/sk_attn.h


class Opts(ctypes.Structure):
    _fields_ = [
        ("policy", ctypes.c_int), ("force_num_splits", ctypes.c_int),
        ("force_pack_gqa", ctypes.c_int), ("force_path", ctypes.c_int),
        ("max_splits", ctypes.c_int), ("num_sms", ctypes.c_int),
        ("debug_echo_plan", ctypes.c_int), ("wait_timeout_us", ctypes.c_int),
        ("debug_inject_stall", ctypes.c_int),
        ("event_begin", ctypes.c_void_p), ("event_end", ctypes.c_void_p),
        ("combine_mode", ctypes.c_int), ("prefill_schedule", ctypes.c_int),
        ("tile_map", ctypes.c_int),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int), ("kBlockM", ctypes.c_int), ("kBlockN", ctypes.c_int),
        ("pack_gqa", ctypes.c_int), ("head_tiles", ctypes.c_int),
        ("rows_per_head_tile", ctypes.c_int), ("num_m_blocks", ctypes.c_int),
        ("num_splits", ctypes.c_int), ("num_splits_policy", ctypes.c_int),
        ("num_n_blocks_max", ctypes.c_int), ("grid_x", ctypes.c_int), ("grid_y", ctypes.c_int),
        ("grid_z", ctypes.c_int), ("num_ctas", ctypes.c_longlong),
        ("needs_combine", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
        ("echo_offset", ctypes.c_size_t), ("lse_part_offset", ctypes.c_size_t),
        ("o_part_offset", ctypes.c_size_t), ("combine_in_kernel", ctypes.c_int),
        ("counter_offset", ctypes.c_size_t), ("persistent", ctypes.c_int),
        ("persistent_ctas", ctypes.c_int), ("l2_section_heads", ctypes.c_int),
        ("tile_map", ctypes.c_int),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class LinearAttnInfo(ctypes.Structure):
    _fields_ = [("num_segments", ctypes.c_int), ("segment_len", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("launches", ctypes.c_int), ("path", ctypes.c_int)]


LINEAR_ATTN_DIM = 128  # dk = dv of the linear-attention entry points


class SKError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        msg = "%s%s" % (sk_attn_status_string(status), (": " + where) if where else "")
        super().__init__(msg)


_lib = None
_i32p = ctypes.POINTER(ctypes.c_int32)
_intp = ctypes.POINTER(ctypes.c_int)


def lib():
    """Load libskattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libskattn.so is not built; run split_kv_flash_gb300/build.py "
                              "(or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, ci, cf = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        L.sk_attn_plan.argtypes = [ci, ci, ci, ci, _intp, ci, ci, ci, ctypes.POINTER(Opts),
                                   ctypes.POINTER(PlanInfo)]
        L.sk_attn_plan_ranges.argtypes = [ci, ci, ci, ci, _intp, ci, ci, ci, ctypes.POINTER(Opts),
                                          _i32p, sz]
        L.sk_attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, _intp, ci, cf, ci, ci, vp, sz,
                                  vp, ctypes.POINTER(Opts)]
        L.sk_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, _intp, ci, cf, ci, ci,
                                          vp, ctypes.POINTER(Opts)]
        L.sk_attn_plan_latent.argtypes = [ci, ci, ci, _intp, ci, ci, ci, ci, ctypes.POINTER(Opts),
                                          ctypes.POINTER(PlanInfo)]
        L.sk_attn_fwd_latent.argtypes = [vp, vp, vp, vp, ci, ci, ci, _intp, ci, ci, cf, ci, ci, vp, sz,
                                         vp, ctypes.POINTER(Opts)]
        L.sk_linear_attn_plan.argtypes = [ci, ci, ci, ci, ci, ci, ctypes.POINTER(Opts),
                                          ctypes.POINTER(LinearAttnInfo)]
        L.sk_linear_attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, sz, vp,
                                         ctypes.POINTER(Opts)]
        L.sk_attn_read_plan_echo.argtypes = [vp, _i32p, sz, vp]
        L.sk_attn_workspace_status.argtypes = [vp, vp, _intp]
        L.sk_attn_noalloc_status.argtypes = [vp, _intp]
        for f in ("sk_attn_plan", "sk_attn_plan_ranges", "sk_attn_fwd", "sk_attn_fwd_noalloc",
                  "sk_attn_read_plan_echo", "sk_attn_workspace_status", "sk_attn_noalloc_status",
                  "sk_attn_plan_latent", "sk_attn_fwd_latent", "sk_linear_attn_plan",
                  "sk_linear_attn_fwd"):
            getattr(L, f).restype = ci
        L.sk_attn_status_string.argtypes = [ci]
        L.sk_attn_status_string.restype = ctypes.c_char_p
        L.sk_attn_last_error.argtypes = []
        L.sk_attn_last_error.restype = ctypes.c_char_p
        L.sk_attn_version.argtypes = []
        L.sk_attn_version.restype = ci
        _lib = L
    return _lib


def _kv_array(kv_len, B=None):
    """kv_len as a C int array; with B given, it must hold exactly B lengths
    (the library reads kv_len[0 .. B-1]; B <= 0 is left to the library to
    reject)."""
    vals = [int(x) for x in kv_len]
    if B is not None and int(B) > 0 and len(vals) != int(B):
        raise ValueError("kv_len holds %d lengths for B = %d sequences" % (len(vals), int(B)))
    return (ctypes.c_int * max(len(vals), 1))(*vals), len(vals)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(status):
    if status != SK_OK:
        raise SKError(status, sk_attn_last_error())


def sk_attn_status_string(status):
    return lib().sk_attn_status_string(int(status)).decode()


def sk_attn_last_error():
    return lib().sk_attn_last_error().decode()


def sk_attn_version():
    return lib().sk_attn_version()


def sk_attn_plan(B, Hq, Hkv, q_len, kv_len, d, causal=False, window_left=-1, opts=None):
    arr, _ = _kv_array(kv_len, B)
    info = PlanInfo()
    _check(lib().sk_attn_plan(B, Hq, Hkv, q_len, arr, d, int(causal), int(window_left),
                              ctypes.byref(opts) if opts is not None else None, ctypes.byref(info)))
    return info


def sk_attn_plan_ranges(B, Hq, Hkv, q_len, kv_len, d, causal=False, window_left=-1, opts=None):
    """Host plan's per-CTA table as a list of (n_block_min, n_block_max, word, has_work)."""
    info = sk_attn_plan(B, Hq, Hkv, q_len, kv_len, d, causal, window_left, opts)
    n = int(info.num_ctas) * 4
    buf = (ctypes.c_int32 * max(n, 1))()
    arr, _ = _kv_array(kv_len, B)
    _check(lib().sk_attn_plan_ranges(B, Hq, Hkv, q_len, arr, d, int(causal), int(window_left),
                                     ctypes.byref(opts) if opts is not None else None, buf, n))
    return [tuple(buf[i:i + 4]) for i in range(0, n, 4)]


def sk_attn_fwd(q, k, v, out, lse, B, Hq, Hkv, q_len, kv_len, d, scale, causal, window_left,
                workspace, ws_bytes, stream=None, opts=None):
    """Pointer-level call: q, k, v, out, lse, workspace are device pointers (ints)
    or tensors; stream is a cudaStream_t handle (int) or a torch.cuda.Stream."""
    arr, _ = _kv_array(kv_len, B)
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(lib().sk_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, q_len,
                             arr, d, float(scale), int(causal), int(window_left), _ptr(workspace),
                             int(ws_bytes), stream,
                             ctypes.byref(opts) if opts is not None else None))


def sk_attn_fwd_noalloc(q, k, v, out, lse, B, Hq, Hkv, q_len, kv_len, d, scale, causal,
                        window_left, stream=None, opts=None):
    """Like sk_attn_fwd, but with no workspace argument: for callers that cannot
    allocate device memory around the call.  The library's built-in scratch
    (NOALLOC_SCRATCH_BYTES per GPU) is used instead; larger problems raise
    SKError(SK_ERR_WORKSPACE_TOO_SMALL).  Calls that overlap on the GPU share
    that scratch and race: keep them ordered on one stream."""
    arr, _ = _kv_array(kv_len, B)
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(lib().sk_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                     q_len, arr, d, float(scale), int(causal), int(window_left),
                                     stream, ctypes.byref(opts) if opts is not None else None))


def sk_attn_plan_latent(B, Hq, q_len, kv_len, d_qk=LATENT_DQK, d_v=LATENT_DV, causal=False, window_left=-1,
                        opts=None):
    arr, _ = _kv_array(kv_len, B)
    info = PlanInfo()
    _check(lib().sk_attn_plan_latent(B, Hq, q_len, arr, d_qk, d_v, int(causal), int(window_left),
                                     ctypes.byref(opts) if opts is not None else None, ctypes.byref(info)))
    return info


def sk_attn_fwd_latent(q, kv, out, lse, B, Hq, q_len, kv_len, d_qk, d_v, scale, causal, window_left,
                       workspace, ws_bytes, stream=None, opts=None):
    """Pointer-level latent attention call (one latent KV head; the values are
    the first d_v columns of each kv row)."""
    arr, _ = _kv_array(kv_len, B)
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(lib().sk_attn_fwd_latent(_ptr(q), _ptr(kv), _ptr(out), _ptr(lse), B, Hq, q_len, arr, d_qk, d_v,
                                    float(scale), int(causal), int(window_left), _ptr(workspace),
                                    int(ws_bytes), stream,
                                    ctypes.byref(opts) if opts is not None else None))


def sk_attn_noalloc_status(stream=None):
    """Status word left by the last sk_attn_fwd_noalloc call on the current
    device: returns (status, where) like sk_attn_workspace_status."""
    where = ctypes.c_int(0)
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = lib().sk_attn_noalloc_status(stream, ctypes.byref(where))
    return st, where.value


def sk_attn_read_plan_echo(workspace, num_ctas, stream=None):
    n = int(num_ctas) * 4
    buf = (ctypes.c_int32 * max(n, 1))()
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(lib().sk_attn_read_plan_echo(_ptr(workspace), buf, n, stream))
    return [tuple(buf[i:i + 4]) for i in range(0, n, 4)]


def sk_attn_workspace_status(workspace, stream=None):
    """Returns (status, where)."""
    where = ctypes.c_int(0)
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    st = lib().sk_attn_workspace_status(_ptr(workspace), stream, ctypes.byref(where))
    return st, where.value


def attn_fwd(q, k, v, kv_len, scale=None, causal=False, window_left=-1, out=None, lse=None,
             workspace=None, opts=None, stream=None):
    """Convenience wrapper over sk_attn_fwd for torch CUDA tensors.

    q [B, q_len, Hq, d], k/v [sum(kv_len), Hkv, d] (bf16, contiguous, same device);
    kv_len: host list of B lengths.  Allocates out [B, q_len, Hq, d] bf16,
    lse [B, Hq, q_len] fp32 and a zeroed workspace when they are not given.
    Returns (out, lse, workspace).
    """
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k and v must be bfloat16")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise TypeError("q, k and v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k and v must be contiguous")
    B, sq, Hq, d = q.shape
    T, Hkv, d2 = k.shape
    kv_len = [int(x) for x in kv_len]
    if d2 != d or tuple(v.shape) != tuple(k.shape) or len(kv_len) != B or sum(kv_len) != T:
        raise ValueError("shape mismatch between q, k, v and kv_len")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    info = sk_attn_plan(B, Hq, Hkv, sq, kv_len, d, causal, window_left, opts)
    if out is None:
        out = torch.empty((B, sq, Hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, sq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sk_attn_fwd(q, k, v, out, lse, B, Hq, Hkv, sq, kv_len, d, scale, causal, window_left,
                workspace, workspace.numel(), stream, opts)
    return out, lse, workspace


def attn_fwd_latent(q, kv, kv_len, scale=None, causal=False, window_left=-1, out=None, lse=None,
                    workspace=None, opts=None, stream=None):
    """Convenience wrapper over sk_attn_fwd_latent for torch CUDA tensors.

    q [B, q_len, Hq, 576], kv [sum(kv_len), 576] (bf16, contiguous): one latent
    head whose rows are the keys and whose first 512 columns are the values.
    Allocates out [B, q_len, Hq, 512] bf16, lse [B, Hq, q_len] fp32 and a
    zeroed workspace when they are not given.  Returns (out, lse, workspace).
    """
    import torch
    if q.dtype != torch.bfloat16 or kv.dtype != torch.bfloat16:
        raise TypeError("q and kv must be bfloat16")
    if not (q.is_cuda and kv.is_cuda):
        raise TypeError("q and kv must be CUDA tensors")
    if not (q.is_contiguous() and kv.is_contiguous()):
        raise ValueError("q and kv must be contiguous")
    B, sq, Hq, d = q.shape
    T, d2 = kv.shape
    kv_len = [int(x) for x in kv_len]
    if d != LATENT_DQK or d2 != d or len(kv_len) != B or sum(kv_len) != T:
        raise ValueError("shape mismatch between q, kv and kv_len (q [B, q_len, Hq, 576], kv [sum(kv_len), 576])")
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    info = sk_attn_plan_latent(B, Hq, sq, kv_len, LATENT_DQK, LATENT_DV, causal, window_left, opts)
    if out is None:
        out = torch.empty((B, sq, Hq, LATENT_DV), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, sq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sk_attn_fwd_latent(q, kv, out, lse, B, Hq, sq, kv_len, LATENT_DQK, LATENT_DV, scale, causal, window_left,
                       workspace, workspace.numel(), stream, opts)
    return out, lse, workspace


def sk_linear_attn_plan(B, T, H, dk=LINEAR_ATTN_DIM, dv=LINEAR_ATTN_DIM, num_segments=0, opts=None):
    info = LinearAttnInfo()
    _check(lib().sk_linear_attn_plan(B, T, H, dk, dv, num_segments,
                                     ctypes.byref(opts) if opts is not None else None, ctypes.byref(info)))
    return info


def sk_linear_attn_fwd(q, k, v, g, out, B, T, H, dk, dv, scale, num_segments, workspace, ws_bytes, stream=None,
                       opts=None):
    """Pointer-level chunk-parallel gated linear attention call."""
    if stream is not None and not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(lib().sk_linear_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), B, T, H, dk, dv, float(scale),
                                    int(num_segments), _ptr(workspace), int(ws_bytes), stream,
                                    ctypes.byref(opts) if opts is not None else None))


def linear_attn_fwd(q, k, v, g, scale=None, num_segments=0, out=None, workspace=None, opts=None, stream=None):
    """Convenience wrapper over sk_linear_attn_fwd for torch CUDA tensors.

    q, k [B, T, H, 128], v [B, T, H, 128] bf16; g [B, T, H, 128] fp32 log decays.
    Returns (out [B, T, H, 128] bf16, workspace)."""
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k and v must be bfloat16")
    if g.dtype != torch.float32:
        raise TypeError("g must be float32")
    for t in (q, k, v, g):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v and g must be contiguous CUDA tensors")
    B, T, H, dk = q.shape
    dv = v.shape[3]
    if tuple(k.shape) != (B, T, H, dk) or tuple(g.shape) != (B, T, H, dk) or tuple(v.shape[:3]) != (B, T, H):
        raise ValueError("shape mismatch between q, k, v and g")
    if scale is None:
        scale = 1.0 / float(dk) ** 0.5
    info = sk_linear_attn_plan(B, T, H, dk, dv, num_segments, opts)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sk_linear_attn_fwd(q, k, v, g, out, B, T, H, dk, dv, scale, num_segments, workspace, workspace.numel(),
                       stream, opts)
    return out, workspace
