"""GPU parity of the chunk-parallel gated linear attention (cuLA issue #11:
T split into segments merged by an affine combine) through the C ABI against
the fp64 oracle's token-by-token recurrence.

Recurrent path (fp32 throughout), per element: |o - o_ref| <= 2^-8 |o_ref| +
1e-3.  The output is bf16 (half a unit in the last place is at most 2^-9 |o|);
the fp32 state adds a relative error of about 1e-6 over the few hundred tokens
a decay of at most e^-0.1 per token keeps in memory, well inside the absolute
term.

Chunk path (tensor-core windows): the products take bf16 operands (unit
roundoff u = 2^-9) and accumulate in fp32.  Along the longest chain an output
term meets four roundings (the decayed q and k, the intra-window score, or the
decayed key, the state copy and the decayed q), so the textbook bound for sums
of rounded products gives, per element,
    |o - o_ref| <= 2^-8 |o_ref| + 1e-3 + 4u * o_abs,
with o_abs the same recurrence run on |q|, |k|, |v| (the sum of the terms'
magnitudes).  That bound is loose where terms cancel, so the rounding errors,
unbiased and independent, are also held in aggregate: the relative RMS error
over all outputs is at most 4u = 2^-7."""
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


CHUNK, RECURRENT = 5, 4  # SK_PATH_LINEAR_CHUNK (tensor-core windows, the default), SK_PATH_LINEAR_RECURRENT
PATHS = [pytest.param(CHUNK, id="chunk"), pytest.param(RECURRENT, id="recurrent")]


def _opts(sk, path):
    o = sk.Opts()
    o.force_path = path
    return o


U_BF16 = 2.0 ** -9


def _abs_bits(t):
    return (wl.bits(t) & np.uint16(0x7FFF)).astype(np.uint16)


def _check(sk, w, num_segments=0, calls=1, path=CHUNK):
    q, k, v, g = wl.make_linear_inputs(w)
    ref, _ = oracle.gla_fwd(wl.bits(q), wl.bits(k), wl.bits(v), g.numpy(), w.scale)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3
    if path == CHUNK:
        o_abs, _ = oracle.gla_fwd(_abs_bits(q), _abs_bits(k), _abs_bits(v), g.numpy(), w.scale)
        bound = bound + 4 * U_BF16 * o_abs
    qg, kg, vg, gg = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    o_ = _opts(sk, path)
    out, ws = sk.linear_attn_fwd(qg, kg, vg, gg, w.scale, num_segments, opts=o_)
    for call in range(calls):
        if call:
            out.zero_()
            sk.linear_attn_fwd(qg, kg, vg, gg, w.scale, num_segments, out=out, workspace=ws, opts=o_)
        torch.cuda.synchronize()
        st, where = sk.sk_attn_workspace_status(ws)
        assert st == 0, "device wait gave up at site %d" % where
        o = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(o))
        err = np.abs(o - ref) - bound
        assert float(err.max()) <= 0.0, "%s N=%d path %d call %d: max|dO| %.3e (max|O| %.3e)" % (
            w.name, num_segments, path, call, float(np.abs(o - ref).max()), float(np.abs(ref).max()))
        if path == CHUNK and ref.size >= 4096:
            rel_rms = float(np.sqrt(np.mean((o - ref) ** 2) / max(np.mean(ref ** 2), 1e-30)))
            assert rel_rms <= 4 * U_BF16, "%s N=%d: relative RMS error %.3e" % (w.name, num_segments, rel_rms)
    info = sk.sk_linear_attn_plan(w.B, w.T, w.H, num_segments=num_segments, opts=o_)
    assert info.path == path
    return info


@pytest.mark.parametrize("path", PATHS)
def test_page_worst_case_shape_auto_segments(sk, path):
    """B=1, H=4, T=8192 (the issue's worst case): one wave of segments."""
    info = _check(sk, wl.linear_attn(1, 8192, 4), 0, calls=2, path=path)
    assert info.num_segments > 1 and info.launches == 3


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("nseg", [1, 2, 5, 16, 37])
def test_segment_counts(sk, nseg, path):
    """Any segment count gives the recurrence's result (1 = no split)."""
    info = _check(sk, wl.linear_attn(2, 1111, 3, seed=1710), nseg, path=path)
    L = -(-1111 // nseg)
    assert info.segment_len == L and info.num_segments == -(-1111 // L)  # empty trailing segments dropped


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("B,T,H,nseg", [
    (1, 1, 1, 0),        # one token
    (1, 33, 2, 0),       # one chunk and one token
    (1, 40, 1, 40),      # one token per segment
    (3, 517, 5, 0),      # ragged chunks, several sequences and heads
    (1, 300, 2, 7),      # segments that end inside a staged chunk
    (1, 385, 1, 1),      # three full windows and one token
])
def test_edges(sk, B, T, H, nseg, path):
    _check(sk, wl.LinearWorkload("gla_edge_b%d_t%d_h%d" % (B, T, H), B, T, H, seed=1720 + T), nseg, path=path)


def test_errors(sk):
    w = wl.linear_attn(1, 64, 1)
    q, k, v, g = [t.cuda() for t in wl.make_linear_inputs(w)]
    out = torch.empty_like(v)
    info = sk.sk_linear_attn_plan(1, 64, 1, num_segments=2)
    ws = torch.empty(int(info.workspace_bytes), dtype=torch.uint8, device="cuda")
    with pytest.raises(sk.SKError) as ei:  # workspace too small
        sk.sk_linear_attn_fwd(q, k, v, g, out, 1, 64, 1, 128, 128, w.scale, 2, ws, 16)
    assert ei.value.status == 3
    with pytest.raises(sk.SKError) as ei:  # head dim outside the supported set
        sk.sk_linear_attn_plan(1, 64, 1, 64, 64)
    assert ei.value.status == 2
    with pytest.raises(sk.SKError) as ei:  # misaligned output
        sk.sk_linear_attn_fwd(q, k, v, g, out.data_ptr() + 2, 1, 64, 1, 128, 128, w.scale, 2, ws, ws.numel())
    assert ei.value.status == 4


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("gmax", [0.01, 1.5, 8.0, 150.0])
def test_decay_strengths(sk, gmax, path):
    """Weak decays (full windows; rescaled chunks only on the recurrent path),
    decays whose sums cross the window / rescaling range in some chunks (mixed),
    strong decays (windows of a few tokens; every chunk on the plain update),
    and log decays below the clamp at -100 (one-token windows)."""
    w = wl.LinearWorkload("gla_gmax%g" % gmax, 2, 700, 3, seed=1730, gmax=gmax)
    _check(sk, w, 0, path=path)
    _check(sk, w, 5, path=path)


def test_force_path_rejects_attention_paths(sk):
    o = _opts(sk, 2)  # SK_PATH_PREFILL
    with pytest.raises(sk.SKError) as ei:
        sk.sk_linear_attn_plan(1, 64, 1, opts=o)
    assert ei.value.status == 1


def test_injected_stall_times_out_and_recovers(sk):
    """Failure detection of the window path without a GPU fault: one MMA-warp
    wait targets a barrier nothing signals; it gives up after half the 20 ms
    limit, the kernels finish, the status word names that wait, and a correct
    call on the same workspace follows."""
    w = wl.linear_attn(1, 512, 2)
    q, k, v, g = [t.cuda() for t in wl.make_linear_inputs(w)]
    o = _opts(sk, CHUNK)
    o.debug_inject_stall = 1
    o.wait_timeout_us = 20000
    out, ws = sk.linear_attn_fwd(q, k, v, g, w.scale, 2, opts=o)
    st, where = sk.sk_attn_workspace_status(ws)
    assert st == 6  # SK_ERR_DEVICE_TIMEOUT
    assert where == (3 << 8) | 8  # linear-attention kernel, the injected wait
    _check(sk, w, 2, path=CHUNK)


@pytest.mark.parametrize("nseg", [1, 3])
@pytest.mark.parametrize("path", PATHS)
def test_call_clears_stale_status_word(sk, nseg, path):
    """The workspace header word reports a wait that gave up during the call;
    whatever it held before (an earlier call's report, reused memory) the
    call's first launch clears it, on both paths and segment layouts."""
    w = wl.linear_attn(1, 384, 2)
    q, k, v, g = [t.cuda() for t in wl.make_linear_inputs(w)]
    o = _opts(sk, path)
    info = sk.sk_linear_attn_plan(w.B, w.T, w.H, num_segments=nseg, opts=o)
    ws = torch.full((max(int(info.workspace_bytes), 256),), 0xA5, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(v)
    sk.linear_attn_fwd(q, k, v, g, w.scale, nseg, out=out, workspace=ws, opts=o)
    st, where = sk.sk_attn_workspace_status(ws)
    assert (st, where) == (0, 0)
