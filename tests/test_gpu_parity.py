"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs.  Tolerances: max-abs 8e-3 on O, 1e-3 on LSE."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return H.sk_mod()


def _check_full(sk, w, opts=None, tag=None):
    q, k, v = wl.make_inputs(w)
    out, lse = H.run_gpu(sk, w, q, k, v, opts)
    ref_o, ref_l = H.oracle_full(w, q, k, v)
    return H.compare_full(out, lse, ref_o, ref_l, tag or w.name)


def _check_sampled(sk, w, n_rows, opts=None, full_heads=None):
    """Sampled rows, plus every query row of the (b, h) heads in full_heads."""
    q, k, v = wl.make_inputs(w)
    out, lse = H.run_gpu(sk, w, q, k, v, opts)
    rows = H.sample_rows(w, n_rows)
    if full_heads:
        extra = np.array([(b, h, i) for b, h in full_heads for i in range(w.q_len)], dtype=np.int32)
        rows = np.unique(np.concatenate([rows, extra]), axis=0)
    ref_o, ref_l = oracle.attn_rows(wl.bits(q), wl.bits(k), wl.bits(v), w.kv_len, w.scale, rows,
                                    w.causal, w.window_left)
    return H.compare_rows(out, lse, rows, ref_o, ref_l, w.name)


# ------------------------------------------------------------ the workloads

def test_tiny_decode(sk):
    _check_full(sk, wl.tiny_decode())


@pytest.mark.parametrize("kv", [4096, 16384, 32768, 131072])
def test_gqa_decode(sk, kv):
    _check_full(sk, wl.gqa_decode(kv))


@pytest.mark.parametrize("q_len", [9, 17, 33])
@pytest.mark.parametrize("prefix", [128, 512, 2048, 8192])
def test_spec_verify(sk, q_len, prefix):
    _check_full(sk, wl.spec_verify(q_len, prefix))


@pytest.mark.parametrize("B", [1, 2, 4, 8])
def test_varlen_decode(sk, B):
    _check_full(sk, wl.varlen_decode(B))


@pytest.mark.parametrize("B", [16, 32])
def test_varlen_decode_large(sk, B):
    _check_full(sk, wl.varlen_decode(B))


@pytest.mark.parametrize("combine", [0, 2])
@pytest.mark.parametrize("B", [2, 8, 32])
def test_varlen_decode_packed_tile_map(sk, B, combine):
    """The packed tile map (one-dimensional grid over the CTAs with work, each
    finding its sequence by a warp prefix sum), with the combine kernel and with
    the in-kernel merge: same results as the oracle."""
    o = sk.Opts()
    o.tile_map = sk.SK_TILE_MAP_PACKED
    o.combine_mode = combine
    w = wl.varlen_decode(B)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left, o)
    assert info.tile_map == sk.SK_TILE_MAP_PACKED
    _check_full(sk, w, opts=o, tag=w.name + "_packed")


@pytest.mark.parametrize("local", [False, True])
def test_prefill_8192(sk, local):
    """Sampled rows over every head, plus one whole head of every sequence: all
    32 m blocks of it, both 128-row halves of each, every LPT launch position."""
    w = wl.prefill(local)
    _check_sampled(sk, w, 384, full_heads=[(b, (7 * b + 3) % w.Hq) for b in range(w.B)])


# ----------------------------------------------------------- shapes and edges

EDGE = [
    # name, B, Hq, Hkv, d, q_len, kv_len, causal, window
    ("prefill_ragged_d128", 2, 4, 2, 128, 200, [333, 200], True, -1),
    ("prefill_ragged_d64", 1, 2, 1, 64, 300, [300], True, -1),
    ("prefill_packed_gqa", 1, 16, 2, 128, 33, [1000], True, -1),
    # G = 3: a 128-row half is not whole groups of 3 heads, so Q is loaded by the
    # softmax warps and O stored directly instead of through the TMA maps
    ("prefill_packed_g3", 1, 6, 2, 128, 40, [500], True, -1),
    ("prefill_local", 1, 4, 4, 128, 520, [520], True, 100),
    ("prefill_window_no_causal", 1, 2, 2, 128, 150, [400], False, 60),
    ("prefill_sk_lt_sq", 1, 2, 2, 128, 260, [100], True, -1),
    ("decode_d64_gqa", 3, 8, 2, 64, 1, [1, 129, 1000], False, -1),
    ("decode_empty_seq", 3, 4, 4, 128, 1, [0, 5, 256], False, -1),
    ("decode_window", 2, 8, 8, 128, 3, [700, 90], False, 33),
    ("decode_causal_window", 1, 8, 2, 128, 8, [1000], True, 0),
    ("decode_unpacked_gqa", 1, 8, 4, 128, 30, [500], True, -1),
    ("verify_sk_lt_sq", 1, 4, 4, 128, 40, [20], True, -1),
    ("decode_kv_not_multiple", 1, 4, 1, 128, 1, [127], False, -1),
    ("decode_rows_64", 1, 64, 1, 128, 1, [3000], False, -1),
    ("decode_rows_48", 1, 16, 1, 128, 3, [3000], False, -1),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_shapes(sk, case):
    name, B, Hq, Hkv, d, sq, kv, causal, window = case
    w = wl.Workload(name, B, Hq, Hkv, d, sq, kv, causal=causal, window_left=window, seed=77)
    opts = None
    if name == "decode_unpacked_gqa":
        opts = sk.Opts()
        opts.force_pack_gqa = -1
    _check_full(sk, w, opts)


def test_q_len_zero_is_a_no_op(sk):
    q = torch.empty((1, 0, 4, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((64, 4, 128), device="cuda").to(torch.bfloat16)
    out, lse, _ = sk.attn_fwd(q, k, k.clone(), [64])
    assert out.numel() == 0 and lse.numel() == 0


# ------------------------------------------------------- split invariance

@pytest.mark.parametrize("S", [1, 2, 3, 7, 32, 128])
def test_forced_splits(sk, S):
    w = wl.gqa_decode(16384)
    opts = sk.Opts()
    opts.force_num_splits = S
    _check_full(sk, w, opts, "%s_S%d" % (w.name, S))


@pytest.mark.parametrize("policy", [1, 2, 3, 4])
def test_policies(sk, policy):
    w = wl.gqa_decode(32768)
    opts = sk.Opts()
    opts.policy = policy
    _check_full(sk, w, opts, "%s_policy%d" % (w.name, policy))


def test_prefill_path_with_splits(sk):
    w = wl.Workload("prefill_split", 1, 4, 2, 128, 256, [2048], causal=True, seed=5)
    opts = sk.Opts()
    opts.force_num_splits = 5
    _check_full(sk, w, opts)


def test_decode_forced_onto_prefill_kernel(sk):
    w = wl.gqa_decode(4096)
    opts = sk.Opts()
    opts.force_path = sk.SK_PATH_PREFILL
    _check_full(sk, w, opts, "gqa_decode_on_prefill_kernel")


# ------------------------------------------------ rows outside a sequence

NEIGHBOUR = [
    # name, B, Hq, Hkv, q_len, kv_len, causal
    ("decode_varlen", 3, 8, 2, 1, [300, 200, 129], False),
    ("verify_uniform", 2, 4, 4, 9, [300, 300], True),
    ("prefill_uniform", 2, 4, 2, 300, [300, 300], True),
]


@pytest.mark.parametrize("case", NEIGHBOUR, ids=[c[0] for c in NEIGHBOUR])
def test_rows_past_a_sequence_never_leak(sk, case):
    """The 128-row block holding the end of a sequence also holds the first
    rows of the next one.  Here those rows carry +Inf, -Inf and NaN in K and V;
    every sequence whose own keys are finite must still match the oracle."""
    name, B, Hq, Hkv, sq, kv, causal = case
    w = wl.Workload(name, B, Hq, Hkv, 128, sq, kv, causal=causal, seed=31)
    q, k, v = wl.make_inputs(w)
    off = np.concatenate([[0], np.cumsum(kv)])
    bad = {1}  # sequence 1's first rows are poisoned; its own result is not checked
    r0 = int(off[1])
    k[r0:r0 + 3] = float("nan")
    k[r0 + 3:r0 + 6] = float("inf")
    v[r0:r0 + 3] = float("inf")
    v[r0 + 3:r0 + 6] = float("nan")
    v[r0 + 6:r0 + 9] = -float("inf")
    out, lse = H.run_gpu(sk, w, q, k, v)
    for b in range(B):
        if b in bad:
            continue
        wb = wl.Workload(name, 1, Hq, Hkv, 128, sq, [kv[b]], causal=causal)
        qb = q[b:b + 1]
        kb = k[int(off[b]):int(off[b + 1])]
        vb = v[int(off[b]):int(off[b + 1])]
        ref_o, ref_l = oracle.attn_fwd(wl.bits(qb), wl.bits(kb), wl.bits(vb), wb.kv_len, wb.scale,
                                       wb.causal, wb.window_left)
        H.compare_full(out[b:b + 1], lse[b:b + 1], ref_o, ref_l, "%s_seq%d" % (name, b))


# ------------------------------------------------------- how splits are merged

MERGE_CASES = [
    wl.tiny_decode(),
    wl.gqa_decode(16384),
    wl.gqa_decode(131072),
    wl.spec_verify(33, 2048),
    wl.varlen_decode(8),
    wl.Workload("decode_d64_gqa_empty", 3, 8, 2, 64, 1, [0, 129, 1000], seed=78),
]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("w", MERGE_CASES, ids=[w.name for w in MERGE_CASES])
def test_split_merge_modes(sk, w, mode):
    """The separate combine kernel (mode 1) and the in-kernel merge by the last
    split CTA of each tile (mode 2) both match the oracle, on two calls in a
    row over one workspace (the per-tile arrival counters reset themselves)."""
    opts = sk.Opts()
    opts.combine_mode = mode
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left, opts)
    if mode == 2:
        assert info.combine_in_kernel == int(info.needs_combine == 1)
    else:
        assert info.combine_in_kernel == 0
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    ref_o, ref_l = H.oracle_full(w, q, k, v)
    out, lse, ws = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left, opts=opts)
    for call in range(2):
        if call:
            out.zero_()
            lse.zero_()
            sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left, out=out, lse=lse,
                        workspace=ws, opts=opts)
        torch.cuda.synchronize()
        assert sk.sk_attn_workspace_status(ws)[0] == 0
        H.compare_full(out.float().cpu().numpy().astype(np.float64),
                       lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
                       "%s_mode%d_call%d" % (w.name, mode, call))


# --------------------------------------------------- prefill tile schedules

SCHED_CASES = [
    # name, B, Hq, Hkv, d, q_len, kv_len, causal, window, forced splits
    ("causal_multi_tile", 2, 4, 2, 128, 700, [700, 700], True, -1, 0),
    ("local_window", 1, 8, 2, 128, 1100, [1100], True, 130, 0),
    ("varlen_splits", 3, 4, 2, 128, 300, [2000, 300, 900], True, -1, 3),
    ("packed_gqa_d64", 1, 16, 2, 64, 40, [3000], False, -1, 0),
    ("sk_lt_sq", 1, 2, 2, 128, 600, [150], True, -1, 0),
    ("window_no_causal", 1, 2, 2, 128, 400, [900], False, 60, 2),
]


@pytest.mark.parametrize("schedule", [1, 2])
@pytest.mark.parametrize("case", SCHED_CASES, ids=[c[0] for c in SCHED_CASES])
def test_prefill_schedules(sk, case, schedule):
    """One CTA per tile (1) and persistent CTAs taking tiles from the atomic
    counter (2) give the oracle's result, twice in a row on one workspace (the
    persistent counters re-arm themselves), and echo the host plan's ranges."""
    name, B, Hq, Hkv, d, sq, kv, causal, window, S = case
    w = wl.Workload(name, B, Hq, Hkv, d, sq, kv, causal=causal, window_left=window, seed=41)
    opts = sk.Opts()
    opts.prefill_schedule = schedule
    opts.force_path = sk.SK_PATH_PREFILL
    opts.debug_echo_plan = 1
    if S:
        opts.force_num_splits = S
    info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, opts)
    assert info.persistent == (1 if schedule == 2 else 0)
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    ref_o, ref_l = H.oracle_full(w, q, k, v)
    out, lse, ws = sk.attn_fwd(qg, kg, vg, kv, w.scale, causal, window, opts=opts)
    for call in range(2):
        if call:
            out.zero_()
            sk.attn_fwd(qg, kg, vg, kv, w.scale, causal, window, out=out, lse=lse, workspace=ws, opts=opts)
        torch.cuda.synchronize()
        assert sk.sk_attn_workspace_status(ws)[0] == 0
        H.compare_full(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                       ref_o, ref_l, "%s_sched%d_call%d" % (name, schedule, call))
    echo = sk.sk_attn_read_plan_echo(ws, info.num_ctas)
    host = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, opts)
    assert np.array_equal(np.array(echo, dtype=np.int32), np.array(host, dtype=np.int32))
