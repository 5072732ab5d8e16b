"""Shared helpers for the GPU tests: run the CUDA path through the C ABI and the
oracle on the same seeded bf16 inputs, and compare."""
import numpy as np
import torch

import oracle
import workloads as wl

# Tolerances fixed by the parity contract: max |O - O_ref| <= 8e-3 (bf16 output),
# max |LSE - LSE_ref| <= 1e-3 (fp32 output).
TOL_O = 8e-3
TOL_LSE = 1e-3


def sk_mod():
    from split_kv_flash_gb300 import build as b
    b.build()
    import split_kv_flash_gb300 as sk
    return sk


def to_gpu(q, k, v):
    return q.cuda(), k.cuda(), v.cuda()


def run_gpu(sk, w, q, k, v, opts=None, stream=None):
    qg, kg, vg = to_gpu(q, k, v)
    out, lse, ws = sk.attn_fwd(qg, kg, vg, w.kv_len, w.scale, w.causal, w.window_left,
                               opts=opts, stream=stream)
    torch.cuda.synchronize()
    st, where = sk.sk_attn_workspace_status(ws)
    assert st == 0, "device status %d at %d" % (st, where)
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_full(w, q, k, v):
    return oracle.attn_fwd(wl.bits(q), wl.bits(k), wl.bits(v), w.kv_len, w.scale, w.causal,
                           w.window_left)


def sample_rows(w, n, seed=0):
    """Rows (b, h, i) spread over every batch, head and query position, with
    the first and last query rows and tile edges always included."""
    rng = np.random.default_rng(seed)
    rows = set()
    edge_i = sorted({0, w.q_len - 1, min(127, w.q_len - 1), min(128, w.q_len - 1),
                     w.q_len // 2, max(w.q_len - 128, 0)})
    for b in range(w.B):
        for i in edge_i:
            rows.add((b, int(rng.integers(0, w.Hq)), i))
    while len(rows) < n:
        rows.add((int(rng.integers(0, w.B)), int(rng.integers(0, w.Hq)),
                  int(rng.integers(0, w.q_len))))
    return np.array(sorted(rows), dtype=np.int32)


def compare_full(out, lse, ref_o, ref_l, tag=""):
    assert np.all(np.isfinite(out)), tag + ": non-finite output"
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin), tag + ": -inf pattern of LSE differs"
    err_o = float(np.max(np.abs(out - ref_o))) if out.size else 0.0
    err_l = float(np.max(np.abs(lse[fin] - ref_l[fin]))) if fin.any() else 0.0
    assert err_o <= TOL_O, "%s: max|dO| = %.3e" % (tag, err_o)
    assert err_l <= TOL_LSE, "%s: max|dLSE| = %.3e" % (tag, err_l)
    return err_o, err_l


def compare_rows(out, lse, rows, ref_o, ref_l, tag=""):
    o = np.stack([out[b, i, h] for b, h, i in rows])
    l = np.array([lse[b, h, i] for b, h, i in rows])
    return compare_full(o, l, ref_o, ref_l, tag)
