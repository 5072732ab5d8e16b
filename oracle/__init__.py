"""fp64 CPU oracle for split-KV flash attention forward.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg may import this package.  It shares no code with
the CUDA path (split_kv_flash_gb300): the attention math lives in
attn_oracle.c, the scheduling formulas in plan_oracle.py, both written from
the pages' definitions.

Parity status: every function here is pinned by tests/test_oracle_pins.py and
tests/test_plan_oracle.py (closed forms, invariances, library special cases and
the pages' worked examples); none is "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int)
        f64p = ctypes.POINTER(ctypes.c_double)
        L.oracle_attn_rows.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, i32p, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_int, ctypes.c_int, i32p, ctypes.c_long, f64p,
                                       f64p, ctypes.c_int]
        L.oracle_attn_rows.restype = ctypes.c_int
        L.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, i32p, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_int, ctypes.c_int, f64p, f64p, ctypes.c_int]
        L.oracle_attn_fwd.restype = ctypes.c_int
        L.oracle_attn_fwd_split.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, i32p, f64p, f64p, ctypes.c_int]
        L.oracle_attn_fwd_split.restype = ctypes.c_int
        L.oracle_attn_rows_v.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                         ctypes.c_int, ctypes.c_int, i32p, ctypes.c_long, f64p,
                                         f64p, ctypes.c_int]
        L.oracle_attn_rows_v.restype = ctypes.c_int
        L.oracle_attn_fwd_v.argtypes = [u16p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                        ctypes.c_int, ctypes.c_int, f64p, f64p, ctypes.c_int]
        L.oracle_attn_fwd_v.restype = ctypes.c_int
        f32p = ctypes.POINTER(ctypes.c_float)
        L.oracle_gla_fwd.argtypes = [u16p, u16p, u16p, f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_double, f64p, f64p, ctypes.c_int]
        L.oracle_gla_fwd.restype = ctypes.c_int
        L.oracle_gla_fwd_segments.argtypes = [u16p, u16p, u16p, f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, f64p,
                                              ctypes.c_int]
        L.oracle_gla_fwd_segments.restype = ctypes.c_int
        L.oracle_count_visible.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oracle_count_visible.restype = ctypes.c_longlong
        _lib = L
    return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are raw bf16 bit patterns (uint16), got %s" % a.dtype)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _f64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attn_fwd(q, k, v, kv_len, scale, causal=False, window_left=-1, nthreads=0):
    """Full fp64 attention.

    q: uint16 bf16 bits [B, sq, Hq, d]; k, v: uint16 [sum(kv_len), Hkv, d].
    Returns (out [B, sq, Hq, d] float64, lse [B, Hq, sq] float64).
    """
    B, sq, Hq, d = q.shape
    Hkv = k.shape[1]
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    kl, klp = _i32(kv_len)
    out = np.zeros((B, sq, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, sq), dtype=np.float64)
    rc = lib().oracle_attn_fwd(qp, kp, vp, B, Hq, Hkv, sq, klp, d, float(scale), int(causal),
                               int(window_left), _f64p(out), _f64p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return out, lse


def attn_rows(q, k, v, kv_len, scale, rows, causal=False, window_left=-1, nthreads=0):
    """Selected rows: rows is an int array [n, 3] of (b, h, i).
    Returns (out [n, d] float64, lse [n] float64)."""
    B, sq, Hq, d = q.shape
    Hkv = k.shape[1]
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    kl, klp = _i32(kv_len)
    rows, rp = _i32(np.asarray(rows).reshape(-1, 3))
    n = rows.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib().oracle_attn_rows(qp, kp, vp, B, Hq, Hkv, sq, klp, d, float(scale), int(causal),
                                int(window_left), rp, n, _f64p(out), _f64p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return out, lse


def attn_fwd_split(q, k, v, kv_len, scale, bounds, causal=False, window_left=-1, nthreads=0):
    """Split reference: bounds int [B, S+1] key boundaries per sequence."""
    B, sq, Hq, d = q.shape
    Hkv = k.shape[1]
    bounds = np.asarray(bounds, dtype=np.int32).reshape(B, -1)
    S = bounds.shape[1] - 1
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    kl, klp = _i32(kv_len)
    bd, bdp = _i32(bounds)
    out = np.zeros((B, sq, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, sq), dtype=np.float64)
    rc = lib().oracle_attn_fwd_split(qp, kp, vp, B, Hq, Hkv, sq, klp, d, float(scale),
                                     int(causal), int(window_left), S, bdp, _f64p(out),
                                     _f64p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_split rejected its arguments")
    return out, lse


def attn_fwd_v(q, k, v, kv_len, scale, causal=False, window_left=-1, nthreads=0):
    """Full fp64 attention with value width dv (the last dimension of v) that may
    differ from the query/key width d.  q [B, sq, Hq, d]; k [sum(kv_len), Hkv, d];
    v [sum(kv_len), Hkv, dv], all uint16 bf16 bits.  Returns (out [B, sq, Hq, dv],
    lse [B, Hq, sq]) as float64."""
    B, sq, Hq, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[2]
    if k.shape[2] != d or v.shape[:2] != k.shape[:2]:
        raise ValueError("shape mismatch")
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    kl, klp = _i32(kv_len)
    out = np.zeros((B, sq, Hq, dv), dtype=np.float64)
    lse = np.zeros((B, Hq, sq), dtype=np.float64)
    rc = lib().oracle_attn_fwd_v(qp, kp, vp, B, Hq, Hkv, sq, klp, d, dv, float(scale), int(causal),
                                 int(window_left), _f64p(out), _f64p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_v rejected its arguments")
    return out, lse


def attn_rows_v(q, k, v, kv_len, scale, rows, causal=False, window_left=-1, nthreads=0):
    """Selected rows (int array [n, 3] of (b, h, i)) with value width dv = v.shape[2].
    Returns (out [n, dv] float64, lse [n] float64)."""
    B, sq, Hq, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[2]
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    kl, klp = _i32(kv_len)
    rows, rp = _i32(np.asarray(rows).reshape(-1, 3))
    n = rows.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib().oracle_attn_rows_v(qp, kp, vp, B, Hq, Hkv, sq, klp, d, dv, float(scale), int(causal),
                                  int(window_left), rp, n, _f64p(out), _f64p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_rows_v rejected its arguments")
    return out, lse


def count_visible(sq, sk, causal, window_left=-1):
    return int(lib().oracle_count_visible(int(sq), int(sk), int(causal), int(window_left)))


# ------------------------------------------------------------ linear attention
# Gated linear attention with a decay per key channel (linear_attn_oracle.c):
#   S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T,  o_t = scale * S_t^T q_t,  S_0 = 0.

def _f32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def gla_fwd(q, k, v, g, scale, nthreads=0):
    """Token-by-token recurrence.  q, k [B, T, H, dk] and v [B, T, H, dv] as bf16
    bits (uint16); g [B, T, H, dk] float32.  Returns (out [B, T, H, dv],
    final state [B, H, dk, dv]) as float64."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    g, gp = _f32(g)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    state = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = lib().oracle_gla_fwd(qp, kp, vp, gp, B, T, H, dk, dv, float(scale), _f64p(out), _f64p(state),
                              int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gla_fwd rejected its arguments")
    return out, state


def gla_fwd_segments(q, k, v, g, scale, nseg, nthreads=0):
    """The segment method (per-segment (M, h_ext), affine combine, re-run from
    each segment's incoming state).  Returns out [B, T, H, dv] float64."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    g, gp = _f32(g)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    rc = lib().oracle_gla_fwd_segments(qp, kp, vp, gp, B, T, H, dk, dv, float(scale), int(nseg), _f64p(out),
                                       int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gla_fwd_segments rejected its arguments")
    return out
