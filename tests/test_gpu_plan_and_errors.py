"""GPU checks of the plan echo (the kernels' KV block ranges are the host plan's,
bit for bit), of buffer bounds (canaries around every output) and of the
bounded-wait error path (an injected wait on a barrier that nothing signals
ends with SK_ERR_DEVICE_TIMEOUT and leaves the context usable)."""
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


ECHO_CASES = [
    ("gqa_decode", 1, 32, 4, 128, 1, [131072], False, -1, 0),
    ("verify", 2, 16, 16, 128, 17, [2048 + 17] * 2, True, -1, 0),
    ("varlen", 8, 32, 8, 128, 1, wl.varlen_lengths(8, 1303), False, -1, 0),
    ("prefill_local", 2, 8, 2, 128, 1024, [1024, 1024], True, 200, 0),
    ("prefill_split", 1, 4, 2, 128, 300, [4000], True, -1, 3),
    ("fa_policy", 1, 32, 4, 128, 1, [65536], False, -1, -2),
    ("varlen_packed", 8, 32, 8, 128, 1, wl.varlen_lengths(8, 1303), False, -1, -3),
    ("varlen_packed_many", 37, 8, 2, 64, 1, wl.varlen_lengths(37, 1304), False, -1, -3),
]


@pytest.mark.parametrize("case", ECHO_CASES, ids=[c[0] for c in ECHO_CASES])
def test_plan_echo_bit_exact(sk, case):
    name, B, Hq, Hkv, d, sq, kv, causal, window, force = case
    w = wl.Workload(name, B, Hq, Hkv, d, sq, kv, causal=causal, window_left=window, seed=3)
    opts = sk.Opts()
    opts.debug_echo_plan = 1
    if force > 0:
        opts.force_num_splits = force
    if force == -2:
        opts.policy = sk.SK_POLICY_FA_HEURISTIC
    if force == -3:
        opts.tile_map = sk.SK_TILE_MAP_PACKED
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    out, lse, ws = sk.attn_fwd(qg, kg, vg, kv, w.scale, causal, window, opts=opts)
    info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, opts)
    echo = sk.sk_attn_read_plan_echo(ws, info.num_ctas)
    host = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, opts)
    assert np.array_equal(np.array(echo, dtype=np.int32), np.array(host, dtype=np.int32))
    if force == -3:
        assert info.tile_map == sk.SK_TILE_MAP_PACKED and info.grid_y == 1 and info.grid_z == 1


def test_outputs_stay_in_bounds(sk):
    """Canary regions before and after O, LSE and the workspace stay untouched."""
    w = wl.Workload("canary", 3, 8, 2, 128, 5, [300, 1, 2000], causal=True, seed=9)
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, True, -1)
    pad = 4096
    n_out = w.B * w.q_len * w.Hq * w.d
    n_lse = w.B * w.Hq * w.q_len
    out_buf = torch.full((n_out + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((n_lse + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    ws_bytes = int(info.workspace_bytes)
    ws_buf = torch.full((ws_bytes + 2 * 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    ws_buf[4096:4096 + ws_bytes] = 0
    out = out_buf[pad:pad + n_out]
    lse = lse_buf[pad:pad + n_lse]
    ws = ws_buf[4096:4096 + ws_bytes]
    sk.sk_attn_fwd(qg, kg, vg, out, lse, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.scale, 1, -1,
                   ws, ws_bytes)
    torch.cuda.synchronize()
    assert torch.all(out_buf[:pad] == 7.0) and torch.all(out_buf[pad + n_out:] == 7.0)
    assert torch.all(lse_buf[:pad] == 7.0) and torch.all(lse_buf[pad + n_lse:] == 7.0)
    assert torch.all(ws_buf[:4096] == 0xA5) and torch.all(ws_buf[4096 + ws_bytes:] == 0xA5)
    ref_o, ref_l = H.oracle_full(w, q, k, v)
    H.compare_full(out.view(w.B, w.q_len, w.Hq, w.d).float().cpu().numpy().astype(np.float64),
                   lse.view(w.B, w.Hq, w.q_len).cpu().numpy().astype(np.float64), ref_o, ref_l,
                   "canary")


@pytest.mark.parametrize("path", [1, 2])
def test_injected_stall_times_out_and_recovers(sk, path):
    """A kernel wait on a barrier that nothing signals gives up after the
    bounded wait; the host reads SK_ERR_DEVICE_TIMEOUT; the next call works."""
    w = wl.gqa_decode(4096) if path == 1 else wl.Workload("p", 1, 4, 4, 128, 256, [512],
                                                           causal=True, seed=2)
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    opts = sk.Opts()
    opts.debug_inject_stall = 1
    opts.wait_timeout_us = 20000
    out, lse, ws = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left, opts=opts)
    st, where = sk.sk_attn_workspace_status(ws)
    assert st == 6, "expected SK_ERR_DEVICE_TIMEOUT, got %d" % st
    assert (where & 0xFF) == 8 and (where >> 8) == path
    # status is cleared and a normal call on the same workspace is correct
    assert sk.sk_attn_workspace_status(ws)[0] == 0
    out, lse, ws = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left, workspace=ws)
    torch.cuda.synchronize()
    assert sk.sk_attn_workspace_status(ws)[0] == 0
    ref_o, ref_l = H.oracle_full(w, q, k, v)
    H.compare_full(out.float().cpu().numpy().astype(np.float64),
                   lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "after_timeout")


def test_host_side_errors(sk):
    w = wl.tiny_decode()
    q, k, v = wl.make_inputs(w)
    qg, kg, vg = H.to_gpu(q, k, v)
    info = sk.sk_attn_plan(1, 4, 4, 1, [256], 64)
    out = torch.empty((1, 1, 4, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 4, 1), dtype=torch.float32, device="cuda")
    ws = torch.zeros(int(info.workspace_bytes), dtype=torch.uint8, device="cuda")
    with pytest.raises(sk.SKError) as ei:   # workspace too small
        sk.sk_attn_fwd(qg, kg, vg, out, lse, 1, 4, 4, 1, [256], 64, 0.125, 0, -1, ws, 16)
    assert ei.value.status == 3
    with pytest.raises(sk.SKError) as ei:   # misaligned q
        sk.sk_attn_fwd(qg.data_ptr() + 2, kg, vg, out, lse, 1, 4, 4, 1, [256], 64, 0.125, 0, -1,
                       ws, ws.numel())
    assert ei.value.status == 4
    with pytest.raises(sk.SKError) as ei:   # bad scale
        sk.sk_attn_fwd(qg, kg, vg, out, lse, 1, 4, 4, 1, [256], 64, -1.0, 0, -1, ws, ws.numel())
    assert ei.value.status == 1
    with pytest.raises(sk.SKError) as ei:   # unsupported head dim
        sk.sk_attn_fwd(qg, kg, vg, out, lse, 1, 4, 4, 1, [256], 96, 0.125, 0, -1, ws, ws.numel())
    assert ei.value.status == 2
