"""CPU checks of the C ABI: the library builds and loads, exports every entry
point that include/sk_attn.h declares, and rejects bad arguments in the host
scheduler without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sk():
    from split_kv_flash_gb300 import build as b
    b.build()
    import split_kv_flash_gb300 as sk
    sk.lib()
    return sk


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(sk_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(sk):
    names = _declared_symbols()
    assert {"sk_attn_plan", "sk_attn_plan_ranges", "sk_attn_fwd", "sk_attn_read_plan_echo",
            "sk_attn_workspace_status", "sk_attn_status_string", "sk_attn_last_error",
            "sk_attn_version"} <= names
    lib = ctypes.CDLL(sk.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), "symbol %s declared but not exported" % n


def test_version_and_status_strings(sk):
    assert sk.sk_attn_version() == 104
    assert sk.sk_attn_status_string(0) == "SK_OK"
    assert sk.sk_attn_status_string(6) == "SK_ERR_DEVICE_TIMEOUT"
    assert sk.sk_attn_status_string(99) == "SK_ERR_UNKNOWN"


def _opts(sk, **kw):
    o = sk.Opts()
    o.num_sms = kw.pop("num_sms", 148)
    for k, v in kw.items():
        setattr(o, k, v)
    return o


@pytest.mark.parametrize("args,status", [
    (dict(B=0), 1), (dict(Hq=6, Hkv=4), 1), (dict(d=96), 2), (dict(kv=[-1]), 1),
    (dict(q_len=-1), 1), (dict(Hq=0), 1), (dict(kv=[1 << 30]), 1),
])
def test_plan_rejects_bad_arguments(sk, args, status):
    a = dict(B=1, Hq=8, Hkv=2, q_len=1, kv=[100], d=128)
    a.update(args)
    kv = a["kv"] if len(a["kv"]) == max(a["B"], 1) else a["kv"] * max(a["B"], 1)
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_plan(a["B"], a["Hq"], a["Hkv"], a["q_len"], kv, a["d"], opts=_opts(sk))
    assert ei.value.status == status
    assert sk.sk_attn_last_error() != ""


def test_plan_rejects_bad_options(sk):
    for kw in (dict(policy=9), dict(force_path=7), dict(force_pack_gqa=2), dict(max_splits=-3)):
        with pytest.raises(sk.SKError) as ei:
            sk.sk_attn_plan(1, 8, 2, 1, [100], 128, opts=_opts(sk, **kw))
        assert ei.value.status == 1


def test_decode_path_needs_small_tiles(sk):
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_plan(1, 16, 16, 100, [500], 128, opts=_opts(sk, force_path=sk.SK_PATH_DECODE))
    assert ei.value.status == 2


def test_workspace_layout_is_aligned_and_sized(sk):
    info = sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=_opts(sk, num_sms=152))
    assert info.needs_combine == 1
    S = info.num_splits
    assert info.echo_offset == 256
    for off in (info.lse_part_offset, info.o_part_offset, info.workspace_bytes):
        assert off % 256 == 0
    assert info.o_part_offset - info.lse_part_offset >= S * 32 * 4
    assert info.workspace_bytes - info.o_part_offset >= S * 32 * 128 * 4
    # no split -> no partial buffers
    info1 = sk.sk_attn_plan(4, 32, 8, 8192, [8192] * 4, 128, causal=True, opts=_opts(sk))
    assert info1.needs_combine == 0
    assert info1.workspace_bytes == info1.o_part_offset


def test_fwd_without_gpu_fails_cleanly(sk):
    """No GPU here: the call must return an error status, never compute on the CPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_fwd(16, 16, 16, 16, 16, 1, 4, 4, 1, [256], 64, 0.125, 0, -1, 256, 1 << 20)
    assert ei.value.status in (2, 5)


def test_binding_checks_kv_len_length(sk):
    """The C side reads kv_len[0 .. B-1]; the binding refuses a list of another
    length before any call reaches the library."""
    o = _opts(sk)
    with pytest.raises(ValueError):
        sk.sk_attn_plan(3, 4, 4, 1, [100, 200], 128, opts=o)
    with pytest.raises(ValueError):
        sk.sk_attn_plan_ranges(1, 4, 4, 1, [100, 200], 128, opts=o)
    with pytest.raises(ValueError):
        sk.sk_attn_fwd(0, 0, 0, 0, 0, 2, 4, 4, 1, [100], 128, 0.1, 0, -1, 0, 0)
    with pytest.raises(ValueError):
        sk.sk_attn_fwd_noalloc(0, 0, 0, 0, 0, 2, 4, 4, 1, [100, 1, 2], 128, 0.1, 0, -1)
    assert sk.sk_attn_plan(2, 4, 4, 1, [100, 200], 128, opts=o).num_ctas >= 2


def test_combine_mode_in_plan(sk):
    """In-kernel merge: on request (mode 2), on the decode path when the tile's
    staged partials fit the decode kernel's K/V rings; never on the prefill
    path; the default and mode 1 keep the separate kernel; an unknown mode is
    rejected."""
    o = _opts(sk, num_sms=152)
    assert sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=o).combine_in_kernel == 0  # default
    o = _opts(sk, num_sms=152, combine_mode=2)
    info = sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=o)
    assert info.needs_combine == 1 and info.combine_in_kernel == 1
    assert info.counter_offset % 256 == 0 and info.lse_part_offset >= info.counter_offset + 4 * 4
    o1 = _opts(sk, num_sms=152, combine_mode=1)
    assert sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=o1).combine_in_kernel == 0
    op = _opts(sk, num_sms=152, force_num_splits=4, force_path=2, combine_mode=2)
    assert sk.sk_attn_plan(1, 4, 2, 300, [4000], 128, True, opts=op).combine_in_kernel == 0
    # 64 rows x 128 splits x 512 B = 4 MB of partials cannot be staged
    big = _opts(sk, num_sms=152, force_num_splits=128, combine_mode=2)
    info = sk.sk_attn_plan(1, 64, 1, 1, [1 << 17], 128, opts=big)
    assert info.needs_combine == 1 and info.combine_in_kernel == 0
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_plan(1, 32, 4, 1, [4096], 128, opts=_opts(sk, combine_mode=5))
    assert ei.value.status == 1
    assert sk.sk_attn_version() == 104


def test_persistent_prefill_plan(sk):
    """Prefill plans run persistent CTAs (at most one per SM) on request; the L2
    section follows the 32 MB rule; G = 3 (a 128-row box is not whole head
    groups) keeps one CTA per tile."""
    assert sk.sk_attn_plan(4, 32, 8, 8192, [8192] * 4, 128, True, opts=_opts(sk, num_sms=152)).persistent == 0
    o = _opts(sk, num_sms=152, prefill_schedule=2)
    info = sk.sk_attn_plan(4, 32, 8, 8192, [8192] * 4, 128, True, opts=o)
    assert info.persistent == 1 and info.persistent_ctas == 152
    # one KV head of 8192 keys = 8192 * 256 * 2 B = 4 MB -> 8 KV heads, x G = 4 query heads
    assert info.l2_section_heads == 32
    assert info.counter_offset % 256 == 0 and info.lse_part_offset >= info.counter_offset + 8
    assert sk.sk_attn_plan(4, 32, 8, 8192, [8192] * 4, 128, True,
                           opts=_opts(sk, num_sms=152, prefill_schedule=1)).persistent == 0
    assert sk.sk_attn_plan(1, 6, 2, 300, [500], 128, True, opts=o).persistent == 0  # G = 3
    small = sk.sk_attn_plan(1, 2, 2, 300, [300], 128, True, opts=o)
    assert small.persistent == 1 and small.persistent_ctas == small.num_ctas  # fewer tiles than SMs
    assert sk.sk_attn_plan(1, 32, 4, 1, [4096], 128, opts=o).persistent == 0  # decode path
    with pytest.raises(sk.SKError):
        sk.sk_attn_plan(1, 2, 2, 300, [300], 128, True, opts=_opts(sk, prefill_schedule=7))


def test_latent_plan(sk):
    """Latent attention plans: the latent path, every query head packed into
    16- or 32-row tiles of the one latent head, partials 512 columns wide;
    other widths are refused."""
    o = _opts(sk, num_sms=152)
    info = sk.sk_attn_plan_latent(2, 64, 9, [2065, 2065], 576, 512, True, opts=o)
    assert info.path == sk.SK_PATH_LATENT
    assert info.pack_gqa == 1 and info.head_tiles == 1
    assert info.rows_per_head_tile == 9 * 64 and info.kBlockM == 32
    assert info.num_m_blocks == 18
    assert info.grid_x == 18 and info.grid_y == info.num_splits and info.grid_z == 2
    # at most 8 KV blocks: 16-row tiles
    short = sk.sk_attn_plan_latent(2, 64, 9, [521, 521], 576, 512, True, opts=o)
    assert short.kBlockM == 16 and short.num_m_blocks == 36
    if info.needs_combine:
        rows = info.num_splits * 2 * 64 * 9
        assert info.o_part_offset - info.lse_part_offset >= rows * 4
        assert info.workspace_bytes - info.o_part_offset >= rows * 512 * 4
    assert sk.sk_attn_plan_latent(1, 8, 2, [4096], opts=o).kBlockM == 16
    assert sk.sk_attn_plan_latent(1, 16, 2, [4096], opts=o).kBlockM == 32
    # one query head: nothing to pack, one head tile of q_len rows
    one = sk.sk_attn_plan_latent(1, 1, 5, [300], opts=o)
    assert one.pack_gqa == 0 and one.rows_per_head_tile == 5 and one.path == sk.SK_PATH_LATENT
    for d_qk, d_v in ((128, 128), (576, 576), (512, 512), (576, 128)):
        with pytest.raises(sk.SKError) as ei:
            sk.sk_attn_plan_latent(1, 16, 2, [100], d_qk, d_v, opts=o)
        assert ei.value.status == 2
    # the standard entry point does not accept the latent path or width
    with pytest.raises(sk.SKError):
        sk.sk_attn_plan(1, 16, 1, 2, [100], 576, opts=o)
    with pytest.raises(sk.SKError):
        sk.sk_attn_plan(1, 16, 1, 2, [100], 128, opts=_opts(sk, num_sms=152, force_path=3))


def test_latent_fwd_without_gpu_fails_cleanly(sk):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_fwd_latent(16, 16, 16, 16, 1, 16, 2, [256], 576, 512, 0.07, 1, -1, 256, 1 << 20)
    assert ei.value.status in (2, 5)


def test_linear_plan_paths_without_gpu(sk):
    """The linear-attention planner picks the window path by default, the
    recurrent path on request, and rejects attention paths; the window path asks
    for at least 128 tokens per segment, the recurrent one for 64."""
    o = _opts(sk, num_sms=152)
    info = sk.sk_linear_attn_plan(1, 8192, 4, opts=o)
    assert info.path == sk.SK_PATH_LINEAR_CHUNK and info.num_segments == 38 and info.launches == 3
    o = _opts(sk, num_sms=152, force_path=sk.SK_PATH_LINEAR_RECURRENT)
    info = sk.sk_linear_attn_plan(1, 8192, 4, opts=o)
    assert info.path == sk.SK_PATH_LINEAR_RECURRENT and info.num_segments == 38
    # short sequence: the minimum segment length decides the count
    short = {}
    for path in (sk.SK_PATH_LINEAR_CHUNK, sk.SK_PATH_LINEAR_RECURRENT):
        short[path] = sk.sk_linear_attn_plan(1, 1000, 4, opts=_opts(sk, num_sms=152, force_path=path))
    assert short[sk.SK_PATH_LINEAR_CHUNK].num_segments == 8      # ceil(1000 / 128)
    assert short[sk.SK_PATH_LINEAR_RECURRENT].num_segments == 16  # ceil(1000 / 64)
    with pytest.raises(sk.SKError) as ei:
        sk.sk_linear_attn_plan(1, 64, 1, opts=_opts(sk, num_sms=152, force_path=sk.SK_PATH_PREFILL))
    assert ei.value.status == 1
