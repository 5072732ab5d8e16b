"""GPU parity of latent attention (absorbed MLA: one latent KV head, 576 key
columns, the first 512 of them the values) through the C ABI against the fp64
oracle, on the verify shapes of "The Occupancy Awakening" and on edge cases.
Tolerances: those of the other parity tests (max-abs 8e-3 on O, 1e-3 on LSE),
on latent rows scaled by 0.5 so that |O| stays near or below 2.  One test runs
unit-variance rows, where a row that sees one to three keys has |O| up to ~4:
there the bf16 output's own rounding (half a unit in the last place, up to
2^-8 |O|) is added to the 8e-3 bound."""
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


def _oracle_kv(kv):
    """Keys [T, 1, 576] and values [T, 1, 512] (bit patterns) of the latent rows."""
    k = wl.bits(kv)[:, None, :]
    v = np.ascontiguousarray(k[:, :, :512])
    return k, v


def _run(sk, w, q, kv, opts=None):
    out, lse, ws = sk.attn_fwd_latent(q.cuda(), kv.cuda(), w.kv_len, w.scale, w.causal, w.window_left, opts=opts)
    torch.cuda.synchronize()
    st, where = sk.sk_attn_workspace_status(ws)
    assert st == 0, "device status %d at %d" % (st, where)
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(sk, w, opts=None, tag=None):
    q, kv = wl.make_latent_inputs(w)
    out, lse = _run(sk, w, q, kv, opts)
    k, v = _oracle_kv(kv)
    ref_o, ref_l = oracle.attn_fwd_v(wl.bits(q), k, v, w.kv_len, w.scale, w.causal, w.window_left)
    return H.compare_full(out, lse, ref_o, ref_l, tag or w.name)


# The verify shapes the page reports parity on (B, H, q_len, kv_len), causal
# (the draft rows see the prefix and the drafts before them) and unmasked.
PAGE_SHAPES = [(2, 16, 17, 2065), (1, 64, 33, 161), (2, 64, 9, 521), (2, 8, 9, 9)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,q_len,kv", PAGE_SHAPES)
def test_latent_verify_page_shapes(sk, B, Hq, q_len, kv, causal):
    _check(sk, wl.latent_verify(B, Hq, q_len, kv, causal, seed=1500 + Hq + q_len))


@pytest.mark.parametrize("splits", [1, 2, 5, 16, 40])
def test_latent_forced_splits(sk, splits):
    """Every split count merges to the same result (combine at 512 columns,
    both combine shapes: <= 16 and > 16 splits)."""
    o = sk.Opts()
    o.force_num_splits = splits
    w = wl.latent_verify(2, 16, 17, [5200, 3001], True, seed=1550)
    _check(sk, w, o, "%s_S%d" % (w.name, splits))


@pytest.mark.parametrize("B,Hq,q_len,kv,causal,window", [
    (1, 1, 1, [1], False, -1),          # one head, one key
    (1, 3, 5, [130], True, -1),         # odd head count, ragged tail block
    (3, 16, 2, [0, 300, 129], False, -1),   # an empty sequence: O = 0, LSE = -inf
    (2, 16, 4, [3, 700], True, -1),     # fewer keys than query rows: causal rows with no key
    (2, 32, 3, [1000, 2048], True, 100),  # local window
    (1, 128, 1, [4096], False, -1),     # 128 heads: four 32-row tiles
    (4, 16, 1, [8192, 1, 777, 4000], False, -1),  # varlen decode
])
def test_latent_edges(sk, B, Hq, q_len, kv, causal, window):
    w = wl.LatentWorkload("latent_edge_b%d_h%d_q%d" % (B, Hq, q_len), B, Hq, q_len, kv, causal, window,
                          seed=1560 + B + Hq + q_len)
    _check(sk, w)


@pytest.mark.parametrize("B,Hq,q_len,kv", [(2, 8, 9, 9), (2, 16, 17, 2065)])
def test_latent_unit_variance_rows(sk, B, Hq, q_len, kv):
    w = wl.latent_verify(B, Hq, q_len, kv, True, seed=1540 + Hq)
    w.kv_scale = 1.0
    q, kv_t = wl.make_latent_inputs(w)
    out, lse = _run(sk, w, q, kv_t)
    k, v = _oracle_kv(kv_t)
    ref_o, ref_l = oracle.attn_fwd_v(wl.bits(q), k, v, w.kv_len, w.scale, True, -1)
    assert np.all(np.isfinite(out))
    assert np.array_equal(np.isfinite(lse), np.isfinite(ref_l))
    fin = np.isfinite(ref_l)
    assert float(np.max(np.abs(lse[fin] - ref_l[fin]))) <= H.TOL_LSE
    excess = np.abs(out - ref_o) - (H.TOL_O + np.abs(ref_o) * 2.0 ** -8)
    assert float(np.max(excess)) <= 0.0, "max|dO| = %.3e" % float(np.max(np.abs(out - ref_o)))


def test_latent_neighbour_rows_do_not_leak(sk):
    """Inf / NaN in the first rows of sequence 1 (read by the last block of
    sequence 0) must not reach sequence 0's output."""
    w = wl.latent_verify(2, 16, 9, [200, 300], True, seed=1580)
    q, kv = wl.make_latent_inputs(w)
    poisoned = kv.clone()
    poisoned[200:256] = float("inf")
    poisoned[201] = float("nan")
    out, lse = _run(sk, w, q, poisoned)
    k, v = _oracle_kv(kv[:200].contiguous())
    ref_o, ref_l = oracle.attn_fwd_v(wl.bits(q[:1].contiguous()), k, v, [200], w.scale, True, -1)
    H.compare_full(out[:1], lse[:1], ref_o, ref_l, "latent_poisoned_neighbour")


def test_latent_long_prefix_sampled(sk):
    """Long prefix (64 Ki keys, many splits): sampled rows against the oracle."""
    w = wl.latent_verify(1, 16, 3, [65536], True, seed=1590)
    q, kv = wl.make_latent_inputs(w)
    out, lse = _run(sk, w, q, kv)
    rows = np.array([(0, h, i) for h in (0, 5, 15) for i in range(3)], dtype=np.int32)
    k, v = _oracle_kv(kv)
    ref_o, ref_l = oracle.attn_rows_v(wl.bits(q), k, v, w.kv_len, w.scale, rows, True, -1)
    H.compare_rows(out, lse, rows, ref_o, ref_l, w.name)


@pytest.mark.parametrize("causal,window", [(True, -1), (False, -1), (True, 300)])
def test_latent_plan_echo_matches_oracle_schedule(sk, causal, window):
    """The latent kernel's own KV block ranges (debug echo) are the scheduling
    oracle's table for the packed problem: one head tile of Hq packed rows."""
    from oracle import plan_oracle as po
    from tests.test_plan_vs_oracle import same_table
    w = wl.LatentWorkload("latent_echo", 2, 16, 17, [2065, 1000], causal, window, seed=1595)
    q, kv = wl.make_latent_inputs(w)
    o = sk.Opts()
    o.debug_echo_plan = 1
    info = sk.sk_attn_plan_latent(w.B, w.Hq, w.q_len, w.kv_len, causal=causal, window_left=window, opts=o)
    out, lse, ws = sk.attn_fwd_latent(q.cuda(), kv.cuda(), w.kv_len, w.scale, causal, window, opts=o)
    echo = sk.sk_attn_read_plan_echo(ws, info.num_ctas)
    splits_b = po.split_counts(w.kv_len, 128, info.num_splits_policy)
    assert max(splits_b) == info.num_splits
    exp = po.cta_table(w.q_len, w.kv_len, w.Hq, True, 1, info.kBlockM, 128, info.num_m_blocks,
                       info.num_splits, splits_b, causal, window)
    assert info.path == sk.SK_PATH_LATENT
    assert same_table(echo, exp)
