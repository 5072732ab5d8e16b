"""The entry point for callers that cannot allocate device memory.

sk_attn_fwd_noalloc takes no workspace: it runs the same split and combine
kernels on the library's built-in scratch array, so code that must not call
cudaMalloc (it can synchronise the device) can still run split-KV attention.
These tests call it through the C ABI twice in a row, on problems that need
the split partials in the scratch, and compare with sk_attn_fwd (which uses a
caller workspace) within the parity tolerances.  The file sorts last so that a
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return H.sk_mod()


def _noalloc(sk, w, qg, kg, vg, stream):
    out = torch.empty((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device="cuda")
    sk.sk_attn_fwd_noalloc(qg, kg, vg, out, lse, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d,
                           w.scale, int(w.causal), w.window_left, stream)
    return out, lse


def test_noalloc_matches_workspace_entry_point_twice(sk):
    stream = torch.cuda.current_stream()
    cases = [wl.gqa_decode(16384), wl.spec_verify(17, 2048)]
    for w in cases:
        info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left)
        assert info.needs_combine == 1  # the partials live in the built-in scratch
        assert info.workspace_bytes <= sk.NOALLOC_SCRATCH_BYTES
        q, k, v = wl.make_inputs(w)
        qg, kg, vg = H.to_gpu(q, k, v)
        ref_out, ref_lse, _ = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left)
        for _ in range(2):  # two calls in a row share (and reuse) the scratch
            out, lse = _noalloc(sk, w, qg, kg, vg, stream)
            torch.cuda.synchronize()
            d_o = (out.float() - ref_out.float()).abs().max().item()
            d_l = (lse - ref_lse).abs().max().item()
            assert d_o <= H.TOL_O and d_l <= H.TOL_LSE, (w.name, d_o, d_l)
            assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_problems_larger_than_the_scratch(sk):
    # 64 query rows x 64 heads with 128 forced splits needs ~268 MB of partials.
    B, Hq, Hkv, sq, d, kv = 1, 64, 64, 64, 128, [20000]
    opts = sk.Opts()
    opts.force_num_splits = 128
    opts.force_path = sk.SK_PATH_PREFILL
    info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, False, -1, opts)
    assert info.workspace_bytes > sk.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, sq, Hq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((kv[0], Hkv, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, sq), dtype=torch.float32, device="cuda")
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_fwd_noalloc(q, k, k, out, lse, B, Hq, Hkv, sq, kv, d, 0.1, 0, -1, None, opts)
    assert ei.value.status == 3
    assert "scratch" in sk.sk_attn_last_error()


def test_noalloc_reports_a_device_timeout_and_recovers(sk):
    """A kernel wait that nothing signals gives up after the bounded wait; the
    code it leaves in the built-in scratch is read with sk_attn_noalloc_status,
    and the next call on the same scratch is correct again."""
    w = wl.gqa_decode(16384)
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    stream = torch.cuda.current_stream()
    opts = sk.Opts()
    opts.debug_inject_stall = 1
    opts.wait_timeout_us = 20000
    out = torch.empty((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device="cuda")
    sk.sk_attn_fwd_noalloc(qg, kg, vg, out, lse, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d,
                           w.scale, 0, -1, stream, opts)
    st, where = sk.sk_attn_noalloc_status(stream)
    assert st == 6 and (where & 0xFF) == 8, (st, where)
    assert sk.sk_attn_noalloc_status(stream)[0] == 0  # read once, then cleared
    ref_out, ref_lse, _ = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale)
    out, lse = _noalloc(sk, w, qg, kg, vg, stream)
    torch.cuda.synchronize()
    assert sk.sk_attn_noalloc_status(stream)[0] == 0
    assert (out.float() - ref_out.float()).abs().max().item() <= H.TOL_O
    assert (lse - ref_lse).abs().max().item() <= H.TOL_LSE
