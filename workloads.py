"""Seeded synthetic inputs and the workload table.

This module is shared by the tests, the benchmark and the oracle callers.  It
holds no attention arithmetic: only shapes, seeds and random draws.

Recipe (every workload): a CPU torch.Generator seeded with the workload's seed
draws, in this order, the per-sequence KV lengths (varlen workloads only,
uniform integers in [512, 65536]), then Q, K and V as float32 standard normals,
which are rounded to bfloat16 (round-to-nearest-even).  Where a workload says
"K scaled by 0.5" the bf16 K is multiplied by 0.5, which is exact.  The same
bf16 bits go to the GPU and, as uint16 bit patterns, to the oracle.

Layouts: Q [B, sq, Hq, d]; K, V [sum_b kv_len[b], Hkv, d] packed by sequence
(sequence b starts at the sum of the lengths before it); O [B, sq, Hq, d];
LSE [B, Hq, sq].

Latent workloads (one latent KV head of 576 columns shared by all query heads):
the generator draws Q [B, sq, Hq, 576] then KV [sum_b kv_len[b], 576] as float32
standard normals rounded to bf16, and multiplies the bf16 KV by kv_scale (0.5 by
default, exact); the values are the first 512 columns of KV.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    q_len: int
    kv_len: List[int]
    causal: bool = False
    window_left: int = -1
    k_scale: float = 1.0
    seed: int = 0
    varlen: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def total_kv(self) -> int:
        return int(sum(self.kv_len))


def varlen_lengths(B: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(512, 65537, (B,), generator=g)]


def make_inputs(w: Workload):
    """Return (q, k, v) as CPU bf16 tensors for workload w."""
    g = torch.Generator().manual_seed(w.seed)
    if w.varlen:
        torch.randint(512, 65537, (w.B,), generator=g)  # lengths come first in the stream
    T = w.total_kv
    q = torch.randn((w.B, w.q_len, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((T, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((T, w.Hkv, w.d), generator=g, dtype=torch.float32)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    if w.k_scale != 1.0:
        k = k * w.k_scale
    return q, k, v


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy array of its bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def tiny_decode() -> Workload:
    """Tiny decode: B=1, Hq=Hkv=4, d=64, q_len=1, kv_len=256, no mask."""
    return Workload("tiny_decode_b1_h4_d64_kv256", 1, 4, 4, 64, 1, [256], seed=1000)


def gqa_decode(kv: int) -> Workload:
    """Small-grid long-context GQA decode (Qwen3-30B-A3B-like): B=1, Hq=32,
    Hkv=4, d=128, q_len=1, K scaled by 0.5."""
    sub = {4096: 0, 16384: 1, 32768: 2, 131072: 3}.get(kv, 9)
    return Workload("gqa_decode_b1_hq32_hkv4_d128_kv%d" % kv, 1, 32, 4, 128, 1, [kv],
                    k_scale=0.5, seed=1100 + sub)


def spec_verify(q_len: int, prefix: int) -> Workload:
    """Speculative verify: B=2, Hq=Hkv=16, d=128, kv_len = prefix + q_len, causal
    with offset (query i sees keys <= kv_len - q_len + i)."""
    sub = {9: 0, 17: 10, 33: 20}.get(q_len, 90) + {128: 0, 512: 1, 2048: 2, 8192: 3}.get(prefix, 9)
    return Workload("verify_b2_h16_d128_q%d_prefix%d" % (q_len, prefix), 2, 16, 16, 128, q_len,
                    [prefix + q_len] * 2, causal=True, seed=1200 + sub)


def varlen_decode(B: int) -> Workload:
    """Batched varlen GQA decode: Hq=32, Hkv=8, d=128, q_len=1, kv_len ~ U[512, 65536]."""
    sub = {1: 0, 2: 1, 4: 2, 8: 3, 16: 4, 32: 5}.get(B, 9)
    seed = 1300 + sub
    return Workload("varlen_decode_b%d_hq32_hkv8_d128" % B, B, 32, 8, 128, 1,
                    varlen_lengths(B, seed), seed=seed, varlen=True)


def prefill(local: bool, seqlen: int = 8192, B: int = 4) -> Workload:
    """Long causal prefill (optionally with a 1024-token left window): B=4, Hq=32,
    Hkv=8, d=128, seqlen_q = seqlen_k = 8192."""
    return Workload("prefill_b%d_hq32_hkv8_d128_s%d_%s" % (B, seqlen, "local1024" if local else "causal"),
                    B, 32, 8, 128, seqlen, [seqlen] * B, causal=True,
                    window_left=1024 if local else -1, seed=1400 + (1 if local else 0))


@dataclass
class LatentWorkload:
    """Absorbed-MLA verify: one latent head (512 latent + 64 rotary columns)."""
    name: str
    B: int
    Hq: int
    q_len: int
    kv_len: List[int]
    causal: bool = True
    window_left: int = -1
    seed: int = 0
    kv_scale: float = 0.5
    d: int = 576
    dv: int = 512

    @property
    def scale(self) -> float:
        # The model's query-key width before absorption: 128 non-rotary + 64
        # rotary columns per head.
        return 1.0 / float(np.sqrt(192.0))

    @property
    def total_kv(self) -> int:
        return int(sum(self.kv_len))


def make_latent_inputs(w: LatentWorkload):
    """Return (q, kv) as CPU bf16 tensors for latent workload w."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.q_len, w.Hq, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.randn((w.total_kv, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if w.kv_scale != 1.0:
        kv = kv * w.kv_scale
    return q, kv


def latent_verify(B: int, Hq: int, q_len: int, kv_len, causal: bool = True, seed: int = 1500) -> LatentWorkload:
    """Latent-attention speculative verify (Kimi K2.6 shapes of "The Occupancy
    Awakening"): q_len = drafts + 1 query rows at the end of the sequence."""
    kv = [int(x) for x in (kv_len if isinstance(kv_len, (list, tuple)) else [kv_len] * B)]
    return LatentWorkload("latent_verify_b%d_h%d_q%d_kv%s%s" % (B, Hq, q_len, "-".join(map(str, sorted(set(kv)))),
                                                             "" if causal else "_nomask"),
                          B, Hq, q_len, kv, causal=causal, seed=seed)


@dataclass
class LinearWorkload:
    """Chunk-parallel gated linear attention (cuLA issue #11 shapes)."""
    name: str
    B: int
    T: int
    H: int
    seed: int = 0
    d: int = 128
    gmax: float = 0.1

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))


def make_linear_inputs(w: LinearWorkload):
    """(q, k, v, g) on the CPU: q, v standard normal, k standard normal scaled to
    unit L2 norm per token and head, all rounded to bf16; g float32 log decays
    drawn uniform in [-gmax, 0]."""
    gen = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.T, w.H, w.d)
    q = torch.randn(shape, generator=gen, dtype=torch.float32)
    k = torch.randn(shape, generator=gen, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, dtype=torch.float32)
    g = -w.gmax * torch.rand(shape, generator=gen, dtype=torch.float32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), g


def linear_attn(B: int, T: int, H: int, seed: int = 1700) -> LinearWorkload:
    return LinearWorkload("gla_b%d_t%d_h%d_d128" % (B, T, H), B, T, H, seed=seed)
