"""Pins for the fp64 attention oracle (oracle/attn_oracle.c).

Each test checks the oracle against something other than itself: a closed
form, an invariance of softmax attention, a library routine on a special case
(torch float64 softmax / logsumexp, which the oracle does not use), or counts
that the pages print.  Together they are chosen so that a dropped term, a sign
or index error, a transposed operand, a wrong GQA head map, a wrong causal
offset or a wrong window bound fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

from workloads import bits


def bf(x):
    """float array -> bf16 bits (values chosen exactly representable)."""
    t = torch.from_numpy(np.array(x, dtype=np.float32)).to(torch.bfloat16)
    return bits(t)


def as_f64(b):
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def rand_bits(shape, rng, scale=1.0):
    x = rng.standard_normal(shape).astype(np.float32) * scale
    return bf(x)


# ---------------------------------------------------------------- closed forms

def test_single_visible_key_returns_its_value_row(oracle_mod):
    """One key: O = V row exactly, LSE = s * q.k (the logit itself)."""
    rng = np.random.default_rng(1)
    q = rand_bits((1, 1, 2, 16), rng)
    k = rand_bits((1, 1, 16), rng)
    v = rand_bits((1, 1, 16), rng)
    s = 0.3
    out, lse = oracle_mod.attn_fwd(q, k, v, [1], s)
    V = as_f64(v)
    for h in range(2):
        np.testing.assert_array_equal(out[0, 0, h], V[0, 0])
        x = s * float(torch.dot(torch.from_numpy(as_f64(q)[0, 0, h]), torch.from_numpy(as_f64(k)[0, 0])))
        assert lse[0, h, 0] == pytest.approx(x, rel=1e-14, abs=1e-14)


def test_zero_query_gives_uniform_weights(oracle_mod):
    """q = 0: every visible logit is 0, LSE = ln n, O = mean of the V rows."""
    rng = np.random.default_rng(2)
    n = 37
    q = bf(np.zeros((1, 1, 1, 32)))
    k = rand_bits((n, 1, 32), rng)
    v = rand_bits((n, 1, 32), rng)
    out, lse = oracle_mod.attn_fwd(q, k, v, [n], 0.125)
    assert lse[0, 0, 0] == pytest.approx(math.log(n), rel=1e-15)
    np.testing.assert_allclose(out[0, 0, 0], as_f64(v)[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_value(oracle_mod):
    rng = np.random.default_rng(3)
    n, d = 19, 24
    q = rand_bits((1, 1, 1, d), rng)
    krow = rand_bits((1, 1, d), rng)
    k = np.repeat(krow, n, axis=0)
    v = rand_bits((n, 1, d), rng)
    s = 0.2
    out, lse = oracle_mod.attn_fwd(q, k, v, [n], s)
    x = s * float(np.dot(as_f64(q)[0, 0, 0], as_f64(krow)[0, 0]))
    assert lse[0, 0, 0] == pytest.approx(x + math.log(n), rel=1e-13, abs=1e-13)
    np.testing.assert_allclose(out[0, 0, 0], as_f64(v)[:, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_constant_value_rows_return_the_constant(oracle_mod):
    rng = np.random.default_rng(4)
    n, d = 50, 16
    q = rand_bits((2, 3, 2, d), rng)
    k = rand_bits((2 * n, 1, d), rng, scale=2.0)
    c = np.array([0.5, -1.25, 3.0, 0.0] * 4, dtype=np.float32)
    v = bf(np.broadcast_to(c, (2 * n, 1, d)))
    out, _ = oracle_mod.attn_fwd(q, k, v, [n, n], 0.25, causal=True)
    np.testing.assert_allclose(out, np.broadcast_to(c.astype(np.float64), out.shape), atol=1e-13)


def test_gqa_query_head_uses_kv_head_h_div_g(oracle_mod):
    """V constant per KV head: query head h must return the constant of KV
    head h // G (contiguous grouping), not h % Hkv."""
    rng = np.random.default_rng(5)
    Hq, Hkv, n, d = 8, 2, 9, 8
    q = rand_bits((1, 1, Hq, d), rng)
    k = rand_bits((n, Hkv, d), rng)
    vals = np.array([1.5, -2.0], dtype=np.float32)
    v = bf(np.broadcast_to(vals[None, :, None], (n, Hkv, d)))
    out, _ = oracle_mod.attn_fwd(q, k, v, [n], 0.3)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, 0, h], vals[h // (Hq // Hkv)], atol=1e-14)


def _one_hot_visibility(oracle_mod, sq, sk, causal, wl):
    """K = 0 makes the weights uniform over the visible keys; V = identity rows
    turns O into the indicator of the visible set divided by its size."""
    d = sk
    q = bf(np.ones((1, sq, 1, d)))
    k = bf(np.zeros((sk, 1, d)))
    v = bf(np.eye(sk, d)[:, None, :])
    out, lse = oracle_mod.attn_fwd(q, k, v, [sk], 1.0, causal=causal, window_left=wl)
    return out[0, :, 0, :], lse[0, 0]


def test_causal_alignment_is_bottom_right(oracle_mod):
    """sq=3, sk=7: query i sees keys 0 .. i + sk - sq (the key offset of the
    causal bound in the tiling chapter, section 3.1)."""
    sq, sk = 3, 7
    o, lse = _one_hot_visibility(oracle_mod, sq, sk, True, -1)
    for i in range(sq):
        last = i + sk - sq
        expect = np.zeros(sk)
        expect[: last + 1] = 1.0 / (last + 1)
        np.testing.assert_allclose(o[i], expect, atol=1e-15)
        assert lse[i] == pytest.approx(math.log(last + 1), rel=1e-15)


def test_local_window_is_inclusive_left_bound(oracle_mod):
    """window_left = 2, causal: query i sees keys i+sk-sq-2 .. i+sk-sq (three keys)."""
    sq, sk, wl = 4, 9, 2
    o, _ = _one_hot_visibility(oracle_mod, sq, sk, True, wl)
    for i in range(sq):
        diag = i + sk - sq
        expect = np.zeros(sk)
        expect[diag - wl: diag + 1] = 1.0 / (wl + 1)
        np.testing.assert_allclose(o[i], expect, atol=1e-15)


def test_window_without_causal_leaves_right_side_open(oracle_mod):
    sq, sk, wl = 2, 6, 1
    o, _ = _one_hot_visibility(oracle_mod, sq, sk, False, wl)
    for i in range(sq):
        lo = i + sk - sq - wl
        expect = np.zeros(sk)
        expect[lo:] = 1.0 / (sk - lo)
        np.testing.assert_allclose(o[i], expect, atol=1e-15)


def test_row_with_no_visible_key(oracle_mod):
    """sk < sq with causal: the first rows see nothing -> O = 0, LSE = -inf."""
    rng = np.random.default_rng(6)
    sq, sk, d = 5, 2, 8
    q = rand_bits((1, sq, 1, d), rng)
    k = rand_bits((sk, 1, d), rng)
    v = rand_bits((sk, 1, d), rng)
    out, lse = oracle_mod.attn_fwd(q, k, v, [sk], 0.5, causal=True)
    for i in range(sq):
        visible = i + sk - sq + 1
        if visible <= 0:
            assert lse[0, 0, i] == -math.inf
            assert np.all(out[0, i, 0] == 0.0)
        else:
            assert np.isfinite(lse[0, 0, i])


# ----------------------------------------------------------------- invariances

def test_permuting_keys_and_values_together_changes_nothing(oracle_mod):
    rng = np.random.default_rng(7)
    n, d = 64, 32
    q = rand_bits((1, 2, 4, d), rng)
    k = rand_bits((n, 2, d), rng)
    v = rand_bits((n, 2, d), rng)
    out0, lse0 = oracle_mod.attn_fwd(q, k, v, [n], 0.17)
    perm = rng.permutation(n)
    out1, lse1 = oracle_mod.attn_fwd(q, k[perm], v[perm], [n], 0.17)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13)


def test_duplicating_every_pair_adds_ln2(oracle_mod):
    rng = np.random.default_rng(8)
    n, d = 40, 16
    q = rand_bits((1, 1, 2, d), rng)
    k = rand_bits((n, 1, d), rng)
    v = rand_bits((n, 1, d), rng)
    out0, lse0 = oracle_mod.attn_fwd(q, k, v, [n], 0.4)
    out1, lse1 = oracle_mod.attn_fwd(q, np.concatenate([k, k]), np.concatenate([v, v]), [2 * n], 0.4)
    np.testing.assert_allclose(lse1, lse0 + math.log(2.0), rtol=1e-13)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)


def test_shifting_every_key_shifts_lse_only(oracle_mod):
    """k_j -> k_j + c shifts every logit by s<q,c>: O unchanged, LSE + s<q,c>.
    Small integers keep k + c exact in bf16."""
    rng = np.random.default_rng(9)
    n, d = 30, 16
    qf = rng.integers(-3, 4, size=(1, 1, 1, d)).astype(np.float32)
    kf = rng.integers(-4, 5, size=(n, 1, d)).astype(np.float32)
    cf = rng.integers(-2, 3, size=(d,)).astype(np.float32)
    vf = rng.standard_normal((n, 1, d)).astype(np.float32)
    s = 0.0625
    out0, lse0 = oracle_mod.attn_fwd(bf(qf), bf(kf), bf(vf), [n], s)
    out1, lse1 = oracle_mod.attn_fwd(bf(qf), bf(kf + cf), bf(vf), [n], s)
    shift = s * float(np.dot(qf[0, 0, 0].astype(np.float64), cf.astype(np.float64)))
    assert lse1[0, 0, 0] == pytest.approx(lse0[0, 0, 0] + shift, rel=1e-13, abs=1e-12)
    np.testing.assert_allclose(out1, out0, rtol=1e-11, atol=1e-12)


# ----------------------------------------------- library routine special cases

@pytest.mark.parametrize("scale", [0.125, 40.0])
def test_unmasked_matches_torch_float64_softmax(oracle_mod, scale):
    """Unmasked attention is softmax(s Q K^T) V: compared with torch's float64
    softmax and logsumexp.  scale=40 gives logits near 1e3, where an exp()
    without max subtraction would overflow."""
    rng = np.random.default_rng(10)
    B, sq, Hq, Hkv, n, d = 2, 3, 4, 2, 23, 16
    q = rand_bits((B, sq, Hq, d), rng)
    k = rand_bits((B * n, Hkv, d), rng)
    v = rand_bits((B * n, Hkv, d), rng)
    out, lse = oracle_mod.attn_fwd(q, k, v, [n, n], scale)
    Q = torch.from_numpy(as_f64(q))
    K = torch.from_numpy(as_f64(k)).view(B, n, Hkv, d)
    V = torch.from_numpy(as_f64(v)).view(B, n, Hkv, d)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            logits = scale * Q[b, :, h, :] @ K[b, :, h // G, :].T
            ref_o = torch.softmax(logits, dim=-1) @ V[b, :, h // G, :]
            ref_l = torch.logsumexp(logits, dim=-1)
            np.testing.assert_allclose(out[b, :, h, :], ref_o.numpy(), rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse[b, h, :], ref_l.numpy(), rtol=1e-13)


def test_varlen_offsets_select_each_sequence(oracle_mod):
    """Packed varlen K/V must equal running each sequence on its own."""
    rng = np.random.default_rng(11)
    lens = [5, 17, 1, 9]
    d = 8
    q = rand_bits((4, 1, 2, d), rng)
    k = rand_bits((sum(lens), 1, d), rng)
    v = rand_bits((sum(lens), 1, d), rng)
    out, lse = oracle_mod.attn_fwd(q, k, v, lens, 0.5)
    off = 0
    for b, n in enumerate(lens):
        o1, l1 = oracle_mod.attn_fwd(q[b:b + 1], k[off:off + n], v[off:off + n], [n], 0.5)
        np.testing.assert_array_equal(out[b], o1[0])
        np.testing.assert_array_equal(lse[b], l1[0])
        off += n


def test_row_subset_matches_full_output(oracle_mod):
    rng = np.random.default_rng(12)
    q = rand_bits((2, 5, 4, 16), rng)
    k = rand_bits((2 * 33, 2, 16), rng)
    v = rand_bits((2 * 33, 2, 16), rng)
    out, lse = oracle_mod.attn_fwd(q, k, v, [33, 33], 0.25, causal=True, window_left=7)
    rows = np.array([[0, 0, 0], [1, 3, 4], [0, 2, 2], [1, 1, 0]])
    o, l = oracle_mod.attn_rows(q, k, v, [33, 33], 0.25, rows, causal=True, window_left=7)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o[r], out[b, i, h])
        assert l[r] == lse[b, h, i]


# ---------------------------------------------------------- split invariance

@pytest.mark.parametrize("causal,wl", [(False, -1), (True, -1), (True, 13)])
def test_split_merge_equals_unsplit(oracle_mod, causal, wl):
    """Any partition of the key axis, evaluated per split and merged by
    log-sum-exp weights, equals the unsplit result (the KV-split reduction of
    'The Occupancy Awakening'; the combine step of the tiling chapter, 5.1)."""
    rng = np.random.default_rng(13)
    B, sq, Hq, Hkv, d = 2, 4, 4, 2, 16
    lens = [61, 40]
    q = rand_bits((B, sq, Hq, d), rng)
    k = rand_bits((sum(lens), Hkv, d), rng)
    v = rand_bits((sum(lens), Hkv, d), rng)
    out0, lse0 = oracle_mod.attn_fwd(q, k, v, lens, 0.3, causal=causal, window_left=wl)
    for S in (1, 2, 3, 7, 40):
        bounds = []
        for n in lens:
            cuts = np.sort(rng.integers(0, n + 1, size=S - 1))
            bounds.append([0, *cuts.tolist(), n])
        out1, lse1 = oracle_mod.attn_fwd_split(q, k, v, lens, 0.3, bounds, causal=causal,
                                                window_left=wl)
        np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)
        fin = np.isfinite(lse0)
        np.testing.assert_array_equal(np.isfinite(lse1), fin)
        np.testing.assert_allclose(lse1[fin], lse0[fin], rtol=1e-12)


# ------------------------------------------------------------- mask counting

def test_causal_pair_count_closed_form(oracle_mod):
    for n in (1, 7, 128, 300):
        assert oracle_mod.count_visible(n, n, 1, -1) == n * (n + 1) // 2


def test_local_pair_count_closed_form(oracle_mod):
    """Square causal + left window wl: row i sees min(i + 1, wl + 1) keys."""
    for n, wl in ((64, 5), (300, 31), (1000, 128)):
        expect = sum(min(i + 1, wl + 1) for i in range(n))
        assert oracle_mod.count_visible(n, n, 1, wl) == expect
    # 8192 / 1024 per head, as in the long prefill workload
    assert oracle_mod.count_visible(8192, 8192, 1, 1024) == 7_872_000


def test_unmasked_pair_count(oracle_mod):
    assert oracle_mod.count_visible(9, 2065, 0, -1) == 9 * 2065


# ------------------------------------------ value width different from key width

def test_value_width_single_key_and_mean(oracle_mod):
    """dv != d: one visible key returns its dv-wide value row and LSE = s q.k;
    identical keys return the mean of the dv-wide value rows, LSE + ln n."""
    rng = np.random.default_rng(21)
    d, dv = 24, 40
    q = rand_bits((1, 1, 3, d), rng)
    k1 = rand_bits((1, 1, d), rng)
    v1 = rand_bits((1, 1, dv), rng)
    out, lse = oracle_mod.attn_fwd_v(q, k1, v1, [1], 0.3)
    qf, kf, vf = as_f64(q), as_f64(k1), as_f64(v1)
    for h in range(3):
        np.testing.assert_array_equal(out[0, 0, h], vf[0, 0])
        assert lse[0, h, 0] == pytest.approx(0.3 * float(qf[0, 0, h] @ kf[0, 0]), rel=1e-12, abs=1e-12)
    n = 5
    k = np.repeat(k1, n, axis=0)
    v = rand_bits((n, 1, dv), rng)
    out, lse = oracle_mod.attn_fwd_v(q, k, v, [n], 0.3)
    vf = as_f64(v)
    np.testing.assert_allclose(out[0, 0, 1], vf[:, 0].mean(axis=0), rtol=0, atol=1e-12)
    assert lse[0, 1, 0] == pytest.approx(0.3 * float(qf[0, 0, 1] @ kf[0, 0]) + math.log(n), abs=1e-12)


def test_latent_values_match_torch_float64(oracle_mod):
    """Absorbed-MLA form (one latent KV head shared by every query head; the
    value is the first dv columns of each latent row), causal, against torch
    float64 softmax on a small case."""
    rng = np.random.default_rng(22)
    B, sq, Hq, d, dv, sk = 1, 3, 4, 36, 32, 11
    q = rand_bits((B, sq, Hq, d), rng)
    kv = rand_bits((sk, 1, d), rng)
    v = np.ascontiguousarray(kv[:, :, :dv])
    out, lse = oracle_mod.attn_fwd_v(q, kv, v, [sk], 0.2, causal=True)
    qt, kt = torch.from_numpy(as_f64(q)), torch.from_numpy(as_f64(kv))
    for i in range(sq):
        n = i + sk - sq + 1
        for h in range(Hq):
            x = 0.2 * (kt[:n, 0] @ qt[0, i, h])
            wts = torch.softmax(x, dim=0)
            ref = (wts[:, None] * kt[:n, 0, :dv]).sum(dim=0)
            np.testing.assert_allclose(out[0, i, h], ref.numpy(), rtol=0, atol=1e-12)
            assert lse[0, h, i] == pytest.approx(float(torch.logsumexp(x, dim=0)), abs=1e-12)


def test_value_width_equal_matches_common_entry_point(oracle_mod):
    """With dv = d the value-width entry point and the common one agree bit for bit."""
    rng = np.random.default_rng(23)
    q = rand_bits((2, 4, 4, 16), rng)
    k = rand_bits((30, 2, 16), rng)
    v = rand_bits((30, 2, 16), rng)
    o1, l1 = oracle_mod.attn_fwd(q, k, v, [10, 20], 0.25, True, 5)
    o2, l2 = oracle_mod.attn_fwd_v(q, k, v, [10, 20], 0.25, True, 5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
