"""Pins for the fp64 linear-attention oracle (oracle/linear_attn_oracle.c).

The oracle runs the gated linear-attention recurrence
    S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T,  o_t = scale * S_t^T q_t,  S_0 = 0,
and the segment method of the cuLA issue (per-segment (M, h_ext) from a zero
state, affine combine, re-run from each segment's incoming state).  Each pin
checks it against something that is not the recurrence: the unrolled sum
    o_t = scale * sum_{s <= t} sum_i q_t[i] k_s[i] exp(sum_{s < u <= t} g_u[i]) v_s,
numpy's matrix product on the ungated special case (causal linear attention),
the one-token limit of full decay, and the closed-form final state.  Planted
mistakes in a copy of the C source must each fail a pin.
"""
import ctypes
import inspect
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import build as obuild


def bf(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def f64(b):
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def inputs(B, T, H, dk, dv, seed, gscale=0.3):
    rng = np.random.default_rng(seed)
    q = bf(rng.standard_normal((B, T, H, dk)))
    k = bf(rng.standard_normal((B, T, H, dk)) / np.sqrt(dk))
    v = bf(rng.standard_normal((B, T, H, dv)))
    g = (-gscale * rng.random((B, T, H, dk))).astype(np.float32)
    return q, k, v, g


def unrolled(q, k, v, g, scale):
    """o_t by the explicit double sum (no recurrence), float64."""
    qf, kf, vf = f64(q), f64(k), f64(v)
    gf = g.astype(np.float64)
    B, T, H, dk = qf.shape
    out = np.zeros(vf.shape)
    cg = np.cumsum(gf, axis=1)  # cg[t] = sum_{u <= t} g_u
    for t in range(T):
        # decay from s to t: exp(cg[t] - cg[s]) per key channel
        w = np.exp(cg[:, t:t + 1] - cg[:, : t + 1])                       # [B, t+1, H, dk]
        coef = np.einsum("bhi,bshi,bshi->bsh", qf[:, t], kf[:, : t + 1], w)  # [B, t+1, H]
        out[:, t] = scale * np.einsum("bsh,bshj->bhj", coef, vf[:, : t + 1])
    return out


def test_matches_unrolled_sum(oracle_mod):
    q, k, v, g = inputs(2, 23, 3, 16, 12, seed=1)
    out, _ = oracle_mod.gla_fwd(q, k, v, g, 0.7)
    np.testing.assert_allclose(out, unrolled(q, k, v, g, 0.7), rtol=1e-11, atol=1e-12)


def test_ungated_is_causal_linear_attention_by_matmul(oracle_mod):
    """g = 0: o = scale * tril(Q K^T) V per (sequence, head)."""
    q, k, v, _ = inputs(1, 31, 2, 8, 8, seed=2)
    g = np.zeros(q.shape, dtype=np.float32)
    out, _ = oracle_mod.gla_fwd(q, k, v, g, 0.5)
    qf, kf, vf = f64(q), f64(k), f64(v)
    for h in range(2):
        ref = 0.5 * np.tril(qf[0, :, h] @ kf[0, :, h].T) @ vf[0, :, h]
        np.testing.assert_allclose(out[0, :, h], ref, rtol=1e-11, atol=1e-12)


def test_full_decay_keeps_only_the_current_token(oracle_mod):
    """exp(g) = 0 (g = -1e4): S_t = k_t v_t^T, o_t = scale (q_t . k_t) v_t."""
    q, k, v, _ = inputs(1, 9, 2, 8, 6, seed=3)
    g = np.full(q.shape, -1e4, dtype=np.float32)
    out, _ = oracle_mod.gla_fwd(q, k, v, g, 1.3)
    qf, kf, vf = f64(q), f64(k), f64(v)
    ref = 1.3 * np.einsum("bthi,bthi->bth", qf, kf)[..., None] * vf
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_final_state_closed_form(oracle_mod):
    """S_T = sum_s Diag(exp(sum_{u > s} g_u)) k_s v_s^T."""
    q, k, v, g = inputs(1, 17, 2, 8, 5, seed=4)
    _, state = oracle_mod.gla_fwd(q, k, v, g, 1.0)
    kf, vf = f64(k), f64(v)
    gf = g.astype(np.float64)
    after = np.cumsum(gf[:, ::-1], axis=1)[:, ::-1] - gf  # sum over u > s
    ref = np.einsum("bshi,bshj->bhij", kf * np.exp(after), vf)
    np.testing.assert_allclose(state, ref, rtol=1e-11, atol=1e-12)


def test_decay_is_per_key_channel(oracle_mod):
    """Decaying only key channel 0 leaves the other channels' contributions as if
    ungated: with q = e_1 the output ignores channel 0's decay."""
    q, k, v, _ = inputs(1, 11, 1, 4, 3, seed=5)
    qe = np.zeros((1, 11, 1, 4), dtype=np.float32)
    qe[..., 1] = 1.0
    qb = bf(qe)
    g = np.zeros((1, 11, 1, 4), dtype=np.float32)
    g[..., 0] = -2.0
    out, _ = oracle_mod.gla_fwd(qb, k, v, g, 1.0)
    kf, vf = f64(k), f64(v)
    ref = np.cumsum(kf[0, :, 0, 1][:, None] * vf[0, :, 0], axis=0)
    np.testing.assert_allclose(out[0, :, 0], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("nseg", [1, 2, 3, 7, 23, 30])
def test_segments_equal_the_recurrence(oracle_mod, nseg):
    """The affine combine of per-segment (M, h_ext) reproduces the recurrence for
    any segment count, including more segments than tokens."""
    q, k, v, g = inputs(2, 23, 2, 8, 8, seed=6)
    ref, _ = oracle_mod.gla_fwd(q, k, v, g, 0.9)
    out = oracle_mod.gla_fwd_segments(q, k, v, g, 0.9, nseg)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out, unrolled(q, k, v, g, 0.9), rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------- planted mistakes

MUTATIONS = {
    "decay_after_update": ("for (int j = 0; j < dv; ++j) row[j] = a * row[j] + ki * la_bf16(v[j]);",
                           "for (int j = 0; j < dv; ++j) row[j] = a * (row[j] + ki * la_bf16(v[j]));"),
    "output_reads_key_not_query": ("const double qi = la_bf16(q[i]);", "const double qi = la_bf16(k[i]);"),
    "scale_dropped": ("for (int j = 0; j < dv; ++j) out[j] *= scale;", "for (int j = 0; j < dv; ++j) out[j] *= 1.0;"),
    "decay_not_exponentiated": ("const double a = exp((double)g[i]);", "const double a = 1.0 + (double)g[i];"),
    "segment_length_floor": ("const int L = T > 0 ? (T + nseg - 1) / nseg : 0;",
                             "const int L = T > 0 ? (T / nseg > 0 ? T / nseg : 1) : 0;"),
    "combine_wrong_segment": ("m * sin[SZ * s + (size_t)i * dv + j] + hext[SZ * s + (size_t)i * dv + j];",
                              "m * sin[SZ * s + (size_t)i * dv + j] + hext[SZ * (s + 1) + (size_t)i * dv + j];"),
    "combine_decay_dropped": ("const double m = exp(logm[(size_t)s * dk + i]);", "const double m = 1.0;"),
}


def _pin_tests():
    mod = sys.modules[__name__]
    return [(n, f) for n, f in inspect.getmembers(mod, inspect.isfunction)
            if n.startswith("test_") and "oracle_mod" in inspect.signature(f).parameters
            and "planted" not in n and "unmutated" not in n]


def _run_pins(oracle_mod):
    failed = []
    for name, fn in _pin_tests():
        arg_sets = [{}]
        for m in getattr(fn, "pytestmark", []):
            if m.name == "parametrize":
                arg_sets = [{m.args[0]: v} for v in m.args[1]]
        for args in arg_sets:
            try:
                fn(oracle_mod=oracle_mod, **args)
            except Exception:  # noqa: BLE001 - any failure counts as caught
                failed.append(name)
                break
    return failed


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, oracle_mod, mutation):
    old, new = MUTATIONS[mutation]
    src = open(obuild.SRC_LINEAR).read()
    assert src.count(old) == 1, old
    path = tmp_path / "linear_attn_oracle.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(path), "-o", str(lib), "-lm"],
                   check=True)
    real = oracle_mod.lib()
    mutant = ctypes.CDLL(str(lib))
    for fname in ("oracle_gla_fwd", "oracle_gla_fwd_segments"):
        getattr(mutant, fname).argtypes = getattr(real, fname).argtypes
        getattr(mutant, fname).restype = getattr(real, fname).restype
    oracle_mod._lib = mutant
    try:
        failed = _run_pins(oracle_mod)
    finally:
        oracle_mod._lib = real
    assert failed, "no pin caught mutation %s" % mutation


def test_unmutated_oracle_passes_every_pin(oracle_mod):
    assert _run_pins(oracle_mod) == []
