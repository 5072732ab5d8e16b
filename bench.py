"""Benchmark of the split-KV flash attention forward on GB300.

Headline (one JSON line on rank 0): small-grid long-context GQA decode,
B=1, Hq=32, Hkv=4, d=128, q_len=1, kv_len=131072 (Qwen3-30B-A3B-like, K scaled
by 0.5), as achieved HBM GB/s of algorithmic bytes (K + V + Q read, O + LSE
written).  One step = one sk_attn_fwd call through the C ABI: host plan,
partial (split) kernel, combine kernel.  The long causal prefill
(B=4, Hq=32, Hkv=8, d=128, 8192 x 8192) is reported beside it as TFLOP/s of
visible (query, key) pairs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (one process per GPU under torch.distributed.run) every rank runs
its own independent decode problem (no collective on the data path); value is
the bytes of all ranks divided by the slowest rank's time (weak scaling).
--impl reference times the fp64 CPU oracle on the host cores instead (rank 0
only), on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "decode attn HBM GB/s (% of peak) and prefill TFLOP/s (% of peak), 1 GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
# The partial kernel is bracketed by CUDA events on every 4th timed step only:
# an event between the partial and the combine kernel keeps the combine from
# being launched early (programmatic dependent launch), so most steps run without.
EVENT_EVERY = 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kv", type=int, default=131072)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="prefill only (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-config sweep")
    ap.add_argument("--workload", default=None,
                    help="profiling helper: run --steps calls of one named workload and exit "
                         "(names: see --list-workloads)")
    ap.add_argument("--list-workloads", action="store_true")
    return ap.parse_args()


def named_workloads():
    """Every workload by its short name (the sweep's, the headline and prefill)."""
    ws = {short_name(w.name): w for w in sweep_workloads()}
    ws["gqa_kv131072"] = wl.gqa_decode(131072)
    ws["prefill_causal"] = wl.prefill(False)
    ws["prefill_local1024"] = wl.prefill(True)
    for w in latent_workloads():
        ws[w.name.replace("latent_verify_", "latent_")] = w
    for w in linear_workloads():
        ws[w.name] = w
    return ws


def run_named(sk, name, calls, device):
    """Profiling helper: `calls` back-to-back calls of one workload on inputs
    drawn on the device; checks the device status word at the end."""
    w = named_workloads()[name]
    g = torch.Generator(device=device).manual_seed(w.seed)
    if isinstance(w, wl.LinearWorkload):
        shape = (w.B, w.T, w.H, w.d)
        q = torch.randn(shape, device=device, generator=g).to(torch.bfloat16)
        k = torch.nn.functional.normalize(torch.randn(shape, device=device, generator=g), dim=-1).to(torch.bfloat16)
        v = torch.randn(shape, device=device, generator=g).to(torch.bfloat16)
        gd = -w.gmax * torch.rand(shape, device=device, generator=g)
        out, ws = sk.linear_attn_fwd(q, k, v, gd, w.scale)
        for _ in range(calls):
            sk.linear_attn_fwd(q, k, v, gd, w.scale, out=out, workspace=ws)
        torch.cuda.synchronize(device)
        print(json.dumps({"workload": w.name, "calls": calls + 1, "status": "ok"}), flush=True)
        return
    if isinstance(w, wl.LatentWorkload):
        q = torch.randn((w.B, w.q_len, w.Hq, w.d), device=device, generator=g).to(torch.bfloat16)
        kv = (torch.randn((w.total_kv, w.d), device=device, generator=g) * w.kv_scale).to(torch.bfloat16)
        out, lse, ws = sk.attn_fwd_latent(q, kv, w.kv_len, w.scale, w.causal, w.window_left)
        for _ in range(calls):
            sk.attn_fwd_latent(q, kv, w.kv_len, w.scale, w.causal, w.window_left, out=out, lse=lse, workspace=ws)
        torch.cuda.synchronize(device)
        st, where = sk.sk_attn_workspace_status(ws)
        if st != 0:
            raise RuntimeError("device status %d at %d" % (st, where))
        print(json.dumps({"workload": w.name, "calls": calls + 1, "status": "ok"}), flush=True)
        return
    q = torch.randn((w.B, w.q_len, w.Hq, w.d), device=device, generator=g).to(torch.bfloat16)
    k = (torch.randn((w.total_kv, w.Hkv, w.d), device=device, generator=g) * w.k_scale).to(torch.bfloat16)
    v = torch.randn((w.total_kv, w.Hkv, w.d), device=device, generator=g).to(torch.bfloat16)
    out, lse, ws = sk.attn_fwd(q, k, v, w.kv_len, w.scale, w.causal, w.window_left)
    for _ in range(calls):
        sk.attn_fwd(q, k, v, w.kv_len, w.scale, w.causal, w.window_left, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize(device)
    st, where = sk.sk_attn_workspace_status(ws)
    if st != 0:
        raise RuntimeError("device status %d at %d" % (st, where))
    print(json.dumps({"workload": w.name, "calls": calls + 1, "status": "ok"}), flush=True)


# --------------------------------------------------------------------- env
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, bf16_sus, src = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"
    if os.path.exists(path):
        try:
            d = json.load(open(path))

            def find(keys):
                for k in keys:
                    if k in d and isinstance(d[k], (int, float)):
                        return float(d[k])
                return None
            h = find(["hbm_gbs", "hbm_GBps", "hbm_copy_gbs"])
            b = find(["bf16_tflops", "bf16_dense_tflops"])
            bs = find(["bf16_tflops_sustained"])
            if h:
                hbm, src = h, "measured"
            if b:
                bf16 = b
            if bs:
                bf16_sus = bs
        except Exception:  # noqa: BLE001
            pass
    return hbm, bf16, bf16_sus, src


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _code_only(text):
    """Source text without comments and blank lines (edits to comments leave the
    kernels, and so their counters, unchanged)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def file_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


DECODE_SOURCES = ["split_kv_flash_gb300/csrc/fwd_decode.cu", "split_kv_flash_gb300/csrc/sm103_ptx.cuh",
                  "split_kv_flash_gb300/csrc/fwd_common.cuh", "split_kv_flash_gb300/csrc/block_range.h",
                  "split_kv_flash_gb300/csrc/kv_producer.cuh"]
PREFILL_SOURCES = ["split_kv_flash_gb300/csrc/fwd_prefill.cu", "split_kv_flash_gb300/csrc/sm103_ptx.cuh",
                   "split_kv_flash_gb300/csrc/fwd_common.cuh", "split_kv_flash_gb300/csrc/block_range.h",
                   "split_kv_flash_gb300/csrc/kv_producer.cuh"]


def ncu_traffic(kernel_key, sources):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(kernel_key)
        if d and d.get("source_sha") == file_sha(sources):
            return float(d["dram_bytes_per_launch"])
    except Exception:  # noqa: BLE001
        pass
    return None


# --------------------------------------------------------------- workloads
def decode_bytes(w):
    kv = 2 * w.total_kv * w.Hkv * w.d * 2
    q = w.B * w.q_len * w.Hq * w.d * 2
    o = q
    lse = w.B * w.Hq * w.q_len * 4
    return kv + q + o + lse


def visible_pairs(w):
    n = 0
    for sk_b in w.kv_len:
        sq = w.q_len
        for i in range(sq):
            diag = i + sk_b - sq
            hi = min(sk_b - 1, diag) if w.causal else sk_b - 1
            lo = max(0, diag - w.window_left) if w.window_left >= 0 else 0
            n += max(0, hi - lo + 1)
    return n * w.Hq


def prefill_flops(w):
    # QK^T and PV: 2 * d flops each per visible (query, key, head)
    return 4.0 * w.d * visible_pairs(w)


# --------------------------------------------------------------- GPU arm
def gpu_decode(sk, w, steps, warmup, device, rotate=3):
    q, k, v = wl.make_inputs(w)
    qs = [q.to(device) for _ in range(rotate)]
    kv_dev = k.to(device), v.to(device)
    ks = [kv_dev[0]] + [kv_dev[0].clone() for _ in range(rotate - 1)]
    vs = [kv_dev[1]] + [kv_dev[1].clone() for _ in range(rotate - 1)]
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left)
    outs = [torch.empty((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device=device)
            for _ in range(rotate)]
    lses = [torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=device)
            for _ in range(rotate)]
    ws = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    ptrs = [(qs[i].data_ptr(), ks[i].data_ptr(), vs[i].data_ptr(), outs[i].data_ptr(),
             lses[i].data_ptr()) for i in range(rotate)]
    opts = sk.Opts()
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in ev_b + ev_e:
        e.record(stream)
    L = sk.lib()
    arr, _ = sk._kv_array(w.kv_len)
    ws_ptr, ws_n = ws.data_ptr(), ws.numel()

    def call(i, with_events=None):
        p = ptrs[i % rotate]
        if with_events is not None and with_events % EVENT_EVERY != 0:
            with_events = None
        if with_events is not None:
            opts.event_begin = ev_b[with_events].cuda_event
            opts.event_end = ev_e[with_events].cuda_event
        else:
            opts.event_begin = None
            opts.event_end = None
        st = L.sk_attn_fwd(p[0], p[1], p[2], p[3], p[4], w.B, w.Hq, w.Hkv, w.q_len, arr, w.d,
                           w.scale, int(w.causal), w.window_left, ws_ptr, ws_n, sh,
                           __import__("ctypes").byref(opts))
        if st != 0:
            raise RuntimeError("sk_attn_fwd: " + sk.sk_attn_last_error())

    for i in range(warmup):
        call(i)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(device)
    t0.record(stream)
    for i in range(steps):
        call(i, with_events=i)
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    total_ms = t0.elapsed_time(t1)
    kern_ms = [ev_b[i].elapsed_time(ev_e[i]) for i in range(0, steps, EVENT_EVERY)]
    st, where = sk.sk_attn_workspace_status(ws)
    if st != 0:
        raise RuntimeError("device status %d at %d" % (st, where))
    return total_ms, kern_ms, info


def gpu_e2e(sk, w, steps, device):
    """Host buffers in, host buffers out: H2D of Q, K, V from pinned memory,
    sk_attn_fwd, D2H of O and LSE, every step, inside the timed region."""
    q, k, v = wl.make_inputs(w)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    qd, kd, vd = (torch.empty_like(t, device=device) for t in (q, k, v))
    out_h = torch.empty((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32).pin_memory()
    out_d = torch.empty(out_h.shape, dtype=torch.bfloat16, device=device)
    lse_d = torch.empty(lse_h.shape, dtype=torch.float32, device=device)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left)
    ws = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        sk.sk_attn_fwd(qd, kd, vd, out_d, lse_d, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.scale,
                       w.causal, w.window_left, ws, ws.numel(), stream)
        out_h.copy_(out_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    return ms, h2d, d2h


def gpu_prefill(sk, w, steps, warmup, device):
    q, k, v = wl.make_inputs(w)
    qd, kd, vd = q.to(device), k.to(device), v.to(device)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left)
    out = torch.empty((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=device)
    ws = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    opts = sk.Opts()
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eve = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in evb + eve:
        e.record(stream)
    for _ in range(warmup):
        sk.sk_attn_fwd(qd, kd, vd, out, lse, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.scale,
                       w.causal, w.window_left, ws, ws.numel(), stream, opts)
    torch.cuda.synchronize(device)
    for i in range(steps):
        flush.fill_(float(i))  # L2 flush between timed launches (outside the events)
        opts.event_begin = evb[i].cuda_event
        opts.event_end = eve[i].cuda_event
        sk.sk_attn_fwd(qd, kd, vd, out, lse, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.scale,
                       w.causal, w.window_left, ws, ws.numel(), stream, opts)
    torch.cuda.synchronize(device)
    ms = [evb[i].elapsed_time(eve[i]) for i in range(steps)]
    return statistics.median(ms), info


def sweep_workloads():
    """Every other configuration: tiny decode, the other GQA decode lengths,
    speculative verify (q_len 9 / 17 / 33 x prefix 128 / 512 / 2048 / 8192) and
    varlen decode (B = 1 ... 32)."""
    ws = [wl.tiny_decode()]
    ws += [wl.gqa_decode(kv) for kv in (4096, 16384, 32768)]
    ws += [wl.spec_verify(q, p) for q in (9, 17, 33) for p in (128, 512, 2048, 8192)]
    ws += [wl.varlen_decode(b) for b in (1, 2, 4, 8, 16, 32)]
    return ws


def short_name(n):
    """Short key for a workload name (flat keys of the bench line)."""
    n = n.replace("gqa_decode_b1_hq32_hkv4_d128_", "gqa_").replace("verify_b2_h16_d128_", "verify_")
    n = n.replace("varlen_decode_", "varlen_").replace("_hq32_hkv8_d128", "")
    return n.replace("tiny_decode_b1_h4_d64_kv256", "tiny")


def gpu_sweep(sk, device, hbm_peak, reps=20, warmup=3, loop_reps=10):
    """Per configuration, two timings of whole calls (partial + combine):
      - "us": one call at a time, CUDA events on the stream around it, L2
        flushed before each call (includes the launch latency of a lone call);
      - "loop_us": calls back to back as a decode loop issues them, replayed
        from a CUDA graph over rotating copies of the inputs that together
        exceed twice the L2 size (so every call reads HBM), time per call.
    Inputs are drawn on the device (throughput does not depend on the values;
    parity is tested on the seeded CPU draws)."""
    rows = []
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for w in sweep_workloads():
        nbytes = decode_bytes(w)
        kv_bytes = 2 * w.total_kv * w.Hkv * w.d * 2
        R = max(1, min(4096, -(-2 * L2_BYTES // max(kv_bytes, 1))))
        g = torch.Generator(device=device).manual_seed(w.seed)
        q = torch.randn((R, w.B, w.q_len, w.Hq, w.d), device=device, generator=g).to(torch.bfloat16)
        k = (torch.randn((R, w.total_kv, w.Hkv, w.d), device=device, generator=g) * w.k_scale).to(torch.bfloat16)
        v = torch.randn((R, w.total_kv, w.Hkv, w.d), device=device, generator=g).to(torch.bfloat16)
        out = torch.empty((R, w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device=device)
        lse = torch.empty((R, w.B, w.Hq, w.q_len), dtype=torch.float32, device=device)
        info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.causal, w.window_left)
        wsb = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)

        def call(r, st):
            sk.sk_attn_fwd(q[r], k[r], v[r], out[r], lse[r], w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d,
                           w.scale, w.causal, w.window_left, wsb, wsb.numel(), st)

        for i in range(warmup):
            call(i % R, stream)
        evb = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        eve = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        for i in range(reps):
            flush.fill_(float(i))
            evb[i].record(stream)
            call(i % R, stream)
            eve[i].record(stream)
        torch.cuda.synchronize(device)
        st, where = sk.sk_attn_workspace_status(wsb)
        if st != 0:
            raise RuntimeError("device status %d at %d (%s)" % (st, where, w.name))
        ms = statistics.median(evb[i].elapsed_time(eve[i]) for i in range(reps))
        row = {"workload": w.name, "us": ms * 1e3, "bytes": nbytes,
               "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
               "path": "decode" if info.path == 1 else "prefill", "splits": info.num_splits,
               "ctas": info.num_ctas, "rotating_copies": R}
        loop_ms = None
        try:
            graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                call(0, side)  # warm the side stream outside the capture
            torch.cuda.synchronize(device)
            with torch.cuda.graph(graph, stream=side):
                for r in range(R):
                    call(r, side)
            graph.replay()
            torch.cuda.synchronize(device)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(loop_reps):
                graph.replay()
            t1.record(stream)
            torch.cuda.synchronize(device)
            loop_ms = t0.elapsed_time(t1) / (loop_reps * R)
            del graph
        except Exception as e:  # noqa: BLE001 - report, keep the isolated numbers
            row["loop_error"] = str(e)[:200]
        st, where = sk.sk_attn_workspace_status(wsb)
        if st != 0:
            raise RuntimeError("device status %d at %d (%s, loop)" % (st, where, w.name))
        if loop_ms is not None:
            row["loop_us"] = loop_ms * 1e3
            row["loop_frac_of_hbm_peak"] = nbytes / (loop_ms * 1e-3) / 1e9 / hbm_peak
        if w.q_len > 1:
            row["tflops"] = prefill_flops(w) / (ms * 1e-3) / 1e12
        rows.append(row)
        del q, k, v, out, lse, wsb
        torch.cuda.empty_cache()
    return rows


def latent_workloads():
    """Latent attention (absorbed MLA, one 576-column latent head): the verify
    shapes of "The Occupancy Awakening" and two longer prefixes at 64 heads."""
    return [wl.latent_verify(2, 16, 17, 2065), wl.latent_verify(1, 64, 33, 161),
            wl.latent_verify(2, 64, 9, 521), wl.latent_verify(1, 64, 9, 16384),
            wl.latent_verify(1, 64, 1, 65536)]


def latent_bytes(w):
    """Latent rows read once (the values are their first 512 columns), Q, O, LSE."""
    return w.total_kv * w.d * 2 + w.B * w.q_len * w.Hq * (w.d + w.dv) * 2 + w.B * w.Hq * w.q_len * 4


def latent_flops(w):
    """QK^T over 576 columns and PV over 512 per visible (query, key) pair per head."""
    return 2.0 * (w.d + w.dv) * visible_pairs(w)


def gpu_latent_sweep(sk, device, hbm_peak, bf16_peak, reps=20, warmup=3, loop_reps=10):
    """Lone-call and graph-loop timings of the latent path (same method as the
    decode sweep), with the tensor and HBM fractions of each."""
    rows = []
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for w in latent_workloads():
        nbytes = latent_bytes(w)
        R = max(1, min(4096, -(-2 * L2_BYTES // max(w.total_kv * w.d * 2, 1))))
        g = torch.Generator(device=device).manual_seed(w.seed)
        q = torch.randn((R, w.B, w.q_len, w.Hq, w.d), device=device, generator=g).to(torch.bfloat16)
        kv = (torch.randn((R, w.total_kv, w.d), device=device, generator=g) * w.kv_scale).to(torch.bfloat16)
        out = torch.empty((R, w.B, w.q_len, w.Hq, w.dv), dtype=torch.bfloat16, device=device)
        lse = torch.empty((R, w.B, w.Hq, w.q_len), dtype=torch.float32, device=device)
        info = sk.sk_attn_plan_latent(w.B, w.Hq, w.q_len, w.kv_len, w.d, w.dv, w.causal, w.window_left)
        wsb = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)

        def call(r, st):
            sk.sk_attn_fwd_latent(q[r], kv[r], out[r], lse[r], w.B, w.Hq, w.q_len, w.kv_len, w.d, w.dv,
                                  w.scale, w.causal, w.window_left, wsb, wsb.numel(), st)

        for i in range(warmup):
            call(i % R, stream)
        evb = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        eve = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        for i in range(reps):
            flush.fill_(float(i))
            evb[i].record(stream)
            call(i % R, stream)
            eve[i].record(stream)
        torch.cuda.synchronize(device)
        ms = statistics.median(evb[i].elapsed_time(eve[i]) for i in range(reps))
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call(0, side)
        torch.cuda.synchronize(device)
        with torch.cuda.graph(graph, stream=side):
            for r in range(R):
                call(r, side)
        graph.replay()
        torch.cuda.synchronize(device)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(loop_reps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize(device)
        loop_ms = t0.elapsed_time(t1) / (loop_reps * R)
        del graph
        st, where = sk.sk_attn_workspace_status(wsb)
        if st != 0:
            raise RuntimeError("device status %d at %d (%s)" % (st, where, w.name))
        fl = latent_flops(w)
        rows.append({"workload": w.name, "us": ms * 1e3, "loop_us": loop_ms * 1e3, "bytes": nbytes,
                     "flops": fl, "splits": info.num_splits, "ctas": info.num_ctas, "kBlockM": info.kBlockM,
                     "rotating_copies": R,
                     "loop_tflops": fl / (loop_ms * 1e-3) / 1e12,
                     "loop_frac_of_bf16_peak": fl / (loop_ms * 1e-3) / 1e12 / bf16_peak,
                     "loop_frac_of_hbm_peak": nbytes / (loop_ms * 1e-3) / 1e9 / hbm_peak})
        del q, kv, out, lse, wsb
        torch.cuda.empty_cache()
    return rows


def latent_summary(rows):
    flat = {}
    for r in rows:
        n = r["workload"].replace("latent_verify_", "")
        flat[n + "_us"] = round(r["us"], 2)
        flat[n + "_loop_us"] = round(r["loop_us"], 2)
        flat[n + "_loop_tflops"] = round(r["loop_tflops"], 1)
        flat[n + "_loop_frac_bf16"] = round(r["loop_frac_of_bf16_peak"], 4)
        flat[n + "_loop_frac_hbm"] = round(r["loop_frac_of_hbm_peak"], 4)
    return flat


def linear_workloads():
    """Chunk-parallel gated linear attention: the cuLA issue's worst case (B=1,
    H=4, T=8192), a longer sequence and two larger grids."""
    return [wl.linear_attn(1, 8192, 4), wl.linear_attn(1, 16384, 4), wl.linear_attn(2, 4096, 8),
            wl.linear_attn(8, 4096, 16)]


def linear_flops(w):
    """Per token and head: the state update (3 flops per state element: a S + k v)
    and the output (2 per element), dk = dv = 128."""
    return 5.0 * w.d * w.d * w.B * w.T * w.H


ALU_FP32_TFLOPS_PER_SM_GHZ = 128 * 2 / 1e3  # FP32 FMA lanes per SM x 2 flops, TFLOP/s per GHz


def linear_tensor_flops(w, N, L):
    """MMA work of the chunk path: per window of at most 128 tokens, four
    128 x 128 x 128 products in the output pass and one in the segment pass
    (segments 0 .. N-2); full windows when the decays do not cut them short."""
    per = 2.0 * 128 ** 3
    wins = [-(-min(L, w.T - s * L) // 128) for s in range(N)]
    return w.B * w.H * per * (4 * sum(wins) + sum(wins[:-1]))


def gpu_linear(sk, device, clock_mhz, bf16_peak, reps=10):
    """Lone calls (L2 flushed before each) of the default (tensor-core window)
    path at the planned segment count and, for the speedup the issue reports,
    with one segment per (sequence, head); and of the token-by-token path at the
    planned segment count."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    alu_peak = ALU_FP32_TFLOPS_PER_SM_GHZ * sms * clock_mhz / 1e3
    rows = []
    for w in linear_workloads():
        g_ = torch.Generator(device=device).manual_seed(w.seed)
        shape = (w.B, w.T, w.H, w.d)
        q = torch.randn(shape, device=device, generator=g_).to(torch.bfloat16)
        k = torch.nn.functional.normalize(torch.randn(shape, device=device, generator=g_), dim=-1).to(torch.bfloat16)
        v = torch.randn(shape, device=device, generator=g_).to(torch.bfloat16)
        g = -w.gmax * torch.rand(shape, device=device, generator=g_)
        row = {"workload": w.name}
        for tag, n, path in (("", 0, sk.SK_PATH_LINEAR_CHUNK), ("one_segment_", 1, sk.SK_PATH_LINEAR_CHUNK),
                             ("recurrent_", 0, sk.SK_PATH_LINEAR_RECURRENT)):
            o = sk.Opts()
            o.force_path = path
            info = sk.sk_linear_attn_plan(w.B, w.T, w.H, num_segments=n, opts=o)
            out, ws = sk.linear_attn_fwd(q, k, v, g, w.scale, n, opts=o)
            ms = []
            for i in range(reps):
                flush.fill_(float(i))
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                sk.linear_attn_fwd(q, k, v, g, w.scale, n, out=out, workspace=ws, stream=stream, opts=o)
                e1.record(stream)
                torch.cuda.synchronize(device)
                ms.append(e0.elapsed_time(e1))
            st, where = sk.sk_attn_workspace_status(ws)
            if st != 0:
                raise RuntimeError("linear attention: device status %d at %d (%s)" % (st, where, w.name))
            m = statistics.median(ms)
            row[tag + "us"] = m * 1e3
            row[tag + "segments"] = info.num_segments
            if not tag:
                row["tokens_per_s"] = w.B * w.T * w.H / (m * 1e-3)
                row["tflops"] = linear_flops(w) / (m * 1e-3) / 1e12
                row["frac_of_alu_peak"] = row["tflops"] / alu_peak
                row["tensor_tflops"] = linear_tensor_flops(w, info.num_segments, info.segment_len) / (m * 1e-3) / 1e12
                row["frac_of_bf16_peak"] = row["tensor_tflops"] / bf16_peak
        row["speedup_vs_one_segment"] = row["one_segment_us"] / row["us"]
        row["speedup_vs_recurrent"] = row["recurrent_us"] / row["us"]
        rows.append(row)
        del q, k, v, g, out, ws
    return rows, alu_peak


def sweep_summary(rows):
    """Flat scalars (per workload: isolated and loop microseconds and fractions
    of the HBM peak), plus the worst row of each kind."""
    flat = {}
    for r in rows:
        n = short_name(r["workload"])
        flat[n + "_us"] = round(r["us"], 2)
        flat[n + "_frac"] = round(r["frac_of_hbm_peak"], 4)
        if "loop_us" in r:
            flat[n + "_loop_us"] = round(r["loop_us"], 2)
            flat[n + "_loop_frac"] = round(r["loop_frac_of_hbm_peak"], 4)
    worst = min(rows, key=lambda r: r["frac_of_hbm_peak"])
    flat["worst_workload"] = worst["workload"]
    flat["worst_frac"] = round(worst["frac_of_hbm_peak"], 4)
    loops = [r for r in rows if "loop_frac_of_hbm_peak" in r]
    if loops:
        wl_ = min(loops, key=lambda r: r["loop_frac_of_hbm_peak"])
        flat["worst_loop_workload"] = wl_["workload"]
        flat["worst_loop_frac"] = round(wl_["loop_frac_of_hbm_peak"], 4)
    return flat


def host_cost_us(sk, device, calls=2000):
    """Host time of one sk_attn_fwd call through the C ABI (median over calls;
    plan, tensor maps and launches; GPU work is asynchronous).  GQA decode at
    16384 keys, one set of inputs."""
    import ctypes
    w = wl.gqa_decode(16384)
    q = torch.zeros((w.B, w.q_len, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    k = torch.zeros((w.total_kv, w.Hkv, w.d), dtype=torch.bfloat16, device=device)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=device)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d)
    wsb = torch.zeros(max(int(info.workspace_bytes), 256), dtype=torch.uint8, device=device)
    L = sk.lib()
    arr, _ = sk._kv_array(w.kv_len, w.B)
    sh = torch.cuda.current_stream(device).cuda_stream
    args = (q.data_ptr(), k.data_ptr(), k.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B, w.Hq, w.Hkv,
            w.q_len, arr, w.d, ctypes.c_float(w.scale), 0, -1, wsb.data_ptr(), wsb.numel(), sh, None)
    ts = []
    for i in range(calls):
        t0 = time.perf_counter()
        L.sk_attn_fwd(*args)
        ts.append(time.perf_counter() - t0)
        if i % 64 == 63:
            torch.cuda.synchronize(device)  # keep the launch queue short
    torch.cuda.synchronize(device)
    return statistics.median(ts) * 1e6


_pg = None


def barrier():
    if _pg is not None:
        torch.distributed.barrier()


def max_over_ranks(x):
    if _pg is None:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank, steps, world, local_ms):
    """Weak scaling: every rank processes its own problem; the job's time is
    the slowest rank's (max over ranks), the job's bytes are all ranks'."""
    job_ms = max_over_ranks(local_ms)
    return bytes_per_step_per_rank * steps * world / (job_ms * 1e-3) / 1e9, job_ms


# ----------------------------------------------------------------- CPU arm
def cpu_oracle(w, seconds, rows_per_call=None, threads=None):
    """Time the fp64 oracle on the host cores (all of them unless `threads`) on
    whole query rows of w: each call computes `rows_per_call` (b, h, i) rows;
    value in GB/s of the algorithmic bytes those rows stand for."""
    import oracle
    q, k, v = wl.make_inputs(w)
    qb, kb, vb = wl.bits(q), wl.bits(k), wl.bits(v)
    all_rows = np.array([(b, h, i) for b in range(w.B) for h in range(w.Hq) for i in range(w.q_len)],
                        dtype=np.int32)
    n = rows_per_call or len(all_rows)
    rows = all_rows[:n]
    threads = threads or os.cpu_count() or 1
    oracle.attn_rows(qb, kb, vb, w.kv_len, w.scale, rows[:1], w.causal, w.window_left, threads)
    t0 = time.perf_counter()
    calls = 0
    while True:
        oracle.attn_rows(qb, kb, vb, w.kv_len, w.scale, rows, w.causal, w.window_left, threads)
        calls += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / calls
    frac = n / len(all_rows)
    gbs = decode_bytes(w) * frac / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d query rows of %s per call, %d calls, %.1f s" % (
                n, len(all_rows), w.name, calls, dt * calls),
            "seconds_per_call": dt}


def reference_arm(args, world, rank):
    if rank != 0:
        return
    w = wl.gqa_decode(args.kv)
    steps, warmup = args.steps, args.warmup
    # each step: the oracle on every query row of the decode step (32 rows x
    # 131072 keys); at most 20 steps keep the run within minutes.
    budget_steps = max(1, min(steps, 20))
    import oracle
    q, k, v = wl.make_inputs(w)
    qb, kb, vb = wl.bits(q), wl.bits(k), wl.bits(v)
    rows = np.array([(b, h, i) for b in range(w.B) for h in range(w.Hq) for i in range(w.q_len)],
                    dtype=np.int32)
    threads = os.cpu_count() or 1
    for _ in range(min(warmup, 3)):
        oracle.attn_rows(qb, kb, vb, w.kv_len, w.scale, rows, w.causal, w.window_left, threads)
    t0 = time.perf_counter()
    for _ in range(budget_steps):
        oracle.attn_rows(qb, kb, vb, w.kv_len, w.scale, rows, w.causal, w.window_left, threads)
    dt = (time.perf_counter() - t0) / budget_steps
    frac = len(rows) / (w.B * w.Hq * w.q_len)
    value = decode_bytes(w) * frac / dt / 1e9
    sample = "all %d query rows of %s per step, %d steps" % (len(rows), w.name, budget_steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": budget_steps, "warmup": min(warmup, 3), "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "q_len": w.q_len, "kv_len": w.kv_len[0], "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- main
def main():
    global _pg
    args = parse()
    world, rank, local = dist_env()
    if args.list_workloads:
        print("\n".join(sorted(named_workloads())))
        return
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
        _pg = torch.distributed.group.WORLD
    import split_kv_flash_gb300 as sk
    from split_kv_flash_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    barrier()
    sk.lib()

    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()
    if args.workload:
        if rank == 0:
            run_named(sk, args.workload, args.steps, device)
        return
    if args.no_decode:  # profiling helper: the prefill kernels alone
        pre = {}
        for local_w in (False, True):
            pw = wl.prefill(local_w)
            ms, _ = gpu_prefill(sk, pw, max(1, min(args.steps, 10)), max(1, args.warmup), device)
            pre["local1024" if local_w else "causal"] = prefill_flops(pw) / (ms * 1e-3) / 1e12
        if rank == 0:
            print(json.dumps({"prefill_tflops": pre}), flush=True)
        return
    w = wl.gqa_decode(args.kv)
    with ClockSampler(local) as clk:
        total_ms, kern_ms, info = gpu_decode(sk, w, args.steps, args.warmup, device)
    bytes_step = decode_bytes(w)
    value, total_ms = whole_job_gbs(bytes_step, args.steps, world, total_ms)
    kern_avg = float(np.mean(kern_ms))
    achieved = bytes_step / (kern_avg * 1e-3) / 1e9
    clocks = clk.summary()

    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "q_len": w.q_len, "kv_len": w.kv_len[0], "k_scale": 0.5,
                   "num_splits": info.num_splits, "ctas": info.num_ctas,
                   "l2": "inputs larger than L2: 3 rotating copies of Q/K/V (%.0f MB each)" % (
                       bytes_step / 1e6),
                   "parallelism": "independent problem per GPU" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": ncu_traffic("decode_gqa_kv131072", DECODE_SOURCES),
                     "kernel": "fwd_decode_kernel<128,16,UniformSeqs>",
                     "kernel_ms": kern_avg, "peak_source": peak_src + " hbm_gbs"},
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
    }
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 30))
        ms, h2d, d2h = gpu_e2e(sk, w, e2e_steps, device)
        ms = max_over_ranks(ms)
        result["e2e"] = {"value": bytes_step * world / (ms * 1e-3) / 1e9, "unit": "GB/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": ms, "steps": e2e_steps}
    if not args.no_prefill:
        # Flat scalars only, so that every number survives in a parsed record.
        pre = {"unit": "TFLOP/s", "peak": bf16_peak, "peak_source": peak_src + " bf16_tflops (burst)",
               "flop_count": "4 * d per visible (query, key) pair per head"}
        for local_w in (False, True):
            pw = wl.prefill(local_w)
            ms, pinfo = gpu_prefill(sk, pw, 10, 3, device)
            fl = prefill_flops(pw)
            tf = fl / (ms * 1e-3) / 1e12
            key = "local1024" if local_w else "causal"
            pre[key + "_workload"] = pw.name
            pre[key + "_tflops"] = tf
            pre[key + "_ms"] = ms
            pre[key + "_flops"] = fl
            pre[key + "_frac_of_bf16_peak"] = tf / bf16_peak
        pre["traffic"] = ncu_traffic("prefill_causal_8192", PREFILL_SOURCES)
        result["prefill"] = pre
        # The same figures as top-level scalars, for readers that keep only those.
        for key in ("causal", "local1024"):
            result["prefill_%s_tflops" % key] = pre[key + "_tflops"]
            result["prefill_%s_ms" % key] = pre[key + "_ms"]
            result["prefill_%s_frac" % key] = pre[key + "_frac_of_bf16_peak"]
    if rank == 0 and not args.no_sweep:
        rows = gpu_sweep(sk, device, hbm_peak)
        result["sweep"] = {
            "unit": "us and fraction of the HBM peak", "peak": hbm_peak, "bound": "hbm",
            "method": "us: median of 20 lone calls (partial + combine), CUDA events around each, L2 "
                      "flushed before each; loop_us: calls back to back from a CUDA graph over rotating "
                      "inputs larger than 2x L2. bytes = K + V of every sequence + Q + O + LSE",
            **sweep_summary(rows)}
        result["sweep_rows"] = rows
        lrows = gpu_latent_sweep(sk, device, hbm_peak, bf16_peak)
        result["latent"] = {
            "unit": "us, TFLOP/s and fractions of the bf16 and HBM peaks",
            "method": "as the sweep; flops = 2 * (576 + 512) per visible (query, key) pair per head; "
                      "bytes = latent rows once + Q + O + LSE",
            **latent_summary(lrows)}
        result["latent_rows"] = lrows
        lin, alu_peak = gpu_linear(sk, device, clocks.get("sm_mhz") or 2070.0, bf16_peak)
        result["linear"] = {
            "unit": "us per call (L2 flushed), tokens x heads per s, TFLOP/s and fractions of the FP32 FMA and "
                    "bf16 tensor peaks",
            "path": "tensor-core windows (the default); recurrent_us: the token-by-token FMA path",
            "bound": "tensor", "peak_tflops": bf16_peak, "alu_peak_tflops": alu_peak,
            "peak_source": "measured bf16 burst; ALU: 152 SMs x 128 FP32 lanes x 2 flops x the SM clock "
                           "sampled during the run",
            "flop_count": "tflops: 5 dk dv per token and head (the recurrence's work); tensor_tflops: the "
                          "window products, 4 x 2 x 128^3 per window of the output pass and 2 x 128^3 per "
                          "window of the segment pass",
            **{r["workload"].replace("gla_", "") + "_" + k: (round(v, 4) if isinstance(v, float) else v)
               for r in lin for k, v in r.items() if k != "workload"}}
        result["host_us_per_call"] = host_cost_us(sk, device)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_oracle(w, args.cpu_seconds)
        one = cpu_oracle(w, max(2.0, args.cpu_seconds / 4), rows_per_call=4, threads=1)
        result["cpu_baseline"]["single_core_value"] = one["value"]
        result["cpu_baseline"]["single_core_sample"] = one["sample"]
    if rank == 0:
        print(json.dumps(result), flush=True)
    if _pg is not None:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
