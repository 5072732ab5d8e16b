"""Scheduling oracle: the pages' tile-range, split and packing rules, restated.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  It shares no code with the
product scheduler in split_kv_flash_gb300/csrc; the tests compare the two
bit for bit.  Sources, all from the FlashAttention tiling strategy and
scheduling chapter (分块策略与调度) unless noted:

* section 3.1 / 3.2 (block.h, BlockMN::get_n_block_min_max): causal upper bound
  on n blocks, local lower bound, PackGQA conversion of packed rows back to
  query positions;
* section 5.3 (split in block.h): a split takes ceil(range / splits) blocks
  starting at split_idx * that, clipped to the range; the split word packs the
  split index in the low 16 bits and the sequence's split count in the high 16;
* section 5.2 (heuristics.h, num_splits_heuristic): the 0.8 * SMs gate, the
  50 MB L2 branch, the <= 4 n-block shortcut and the wave-efficiency scan with
  the 0.85 * best-efficiency threshold;
* section 6.2 (heuristics.h, should_pack_gqa): pack when the unpacked
  efficiency is below 0.9 times the packed one;
* "The Occupancy Awakening": NSPLIT = clamp(ceil(kv_len / 2048), 1, 32);
* llama.cpp PR #21086 review: at least two blocks per SM, more only while
  each block keeps a minimum KV chunk (256 suggested).

Integer division follows C semantics (truncation toward zero) because the
printed code is C++; efficiencies are binary32 as in the printed code and are
compared against double constants the way C++ promotes them.
"""
import math

import numpy as np

L2_SPLIT_BYTES = 50 * 1024 * 1024  # "KV head > L2 (50MB)" in the section 5.2 flowchart


def c_div(a: int, b: int) -> int:
    """C/C++ integer division (truncates toward zero)."""
    q = abs(a) // abs(b)
    return q if (a >= 0) == (b > 0) else -q


def ceil_div(a: int, b: int) -> int:
    """cute::ceil_div as printed: (a + b - 1) / b with C division."""
    return c_div(a + b - 1, b)


def should_pack_gqa(varlen_q: bool, seqlen_q: int, qhead_per_khead: int, block_m: int) -> bool:
    """Section 6.2: efficiency = useful rows / rows rounded up to block_m."""
    if varlen_q:
        return True

    def round_up(a, b):
        return c_div(a + b - 1, b) * b

    nopack = np.float32(seqlen_q) / np.float32(round_up(seqlen_q, block_m))
    packed = seqlen_q * qhead_per_khead
    pack = np.float32(packed) / np.float32(round_up(packed, block_m))
    return float(nopack) < 0.9 * float(pack)


def num_splits_heuristic(total_mblocks: int, num_sms: int, num_n_blocks: int,
                         num_m_blocks: int, size_one_kv_head: int,
                         is_causal_or_local: bool, max_splits: int) -> int:
    """Section 5.2 decision flow, with max_splits as the scan limit."""
    if total_mblocks >= 0.8 * num_sms:
        if size_one_kv_head > L2_SPLIT_BYTES:
            if num_m_blocks >= 2 * num_sms and not is_causal_or_local:
                return min(ceil_div(size_one_kv_head, L2_SPLIT_BYTES), max_splits)
        return 1
    if num_n_blocks <= 4:
        return 1
    effs = []
    for s in range(1, max_splits + 1):
        n_waves = np.float32(total_mblocks * s) / np.float32(num_sms)
        effs.append(np.float32(n_waves / np.float32(math.ceil(float(n_waves)))))
    best = max(effs) if effs else np.float32(1.0)
    for s in range(1, max_splits + 1):
        if float(effs[s - 1]) >= 0.85 * float(best):
            return s
    return 1


def nsplit_fixed_chunk(kv_len: int) -> int:
    """'The Occupancy Awakening': NSPLIT = ceil(kv_len / 2048) clamped to [1, 32]."""
    return max(1, min(32, ceil_div(kv_len, 2048)))


def nsplit_min_chunk(num_sms: int, tiles: int, kv_len: int, min_chunk: int = 256,
                     blocks_per_sm: int = 2) -> int:
    """llama.cpp PR #21086 review: aim for blocks_per_sm blocks per SM, but never
    give a block less than min_chunk keys."""
    fill = ceil_div(blocks_per_sm * num_sms, tiles)
    by_chunk = c_div(kv_len, min_chunk)
    return max(1, min(fill, by_chunk))


def n_block_min_max(seqlen_q: int, seqlen_k: int, m_block: int, block_m: int, block_n: int,
                    causal: bool, local: bool, window_left: int, window_right: int,
                    pack_gqa: bool, qhead_per_khead: int, split_word: int = None):
    """Sections 3.2 and 5.3.  split_word: low 16 bits split index, high 16 bits
    the number of splits of this sequence; None means no split."""
    n_block_max = ceil_div(seqlen_k, block_n)
    if causal or local:
        m_idx_max = (m_block + 1) * block_m
        if pack_gqa:
            m_idx_max = c_div(m_idx_max - 1, qhead_per_khead) + 1
        n_idx = m_idx_max + seqlen_k - seqlen_q
        n_idx_right = n_idx if not local else n_idx + window_right
        n_block_max = min(n_block_max, ceil_div(n_idx_right, block_n))
    n_block_min = 0
    if local:
        m_idx_min = m_block * block_m
        if pack_gqa:
            m_idx_min = c_div(m_idx_min, qhead_per_khead)
        n_idx = m_idx_min + seqlen_k - seqlen_q
        n_idx_left = n_idx - window_left
        n_block_min = max(0, c_div(n_idx_left, block_n))
    if split_word is not None:
        split_idx = split_word & 0xFFFF
        n_split = (split_word >> 16) & 0xFFFF
        per = ceil_div(n_block_max - n_block_min, n_split)
        n_block_min = n_block_min + split_idx * per
        n_block_max = min(n_block_min + per, n_block_max)
    return n_block_min, n_block_max


def split_counts(kv_lens, block_n: int, num_splits: int):
    """Per-sequence split counts when sequences differ in length: one chunk size
    ceil(n_blocks_max / S) for the whole batch, and each sequence takes as many
    chunks as it needs (reading of the high-16-bit count in section 5.3)."""
    nblk = [ceil_div(s, block_n) for s in kv_lens]
    nmax = max(nblk) if nblk else 0
    if num_splits <= 1 or nmax == 0:
        return [1] * len(kv_lens)
    chunk = ceil_div(nmax, num_splits)
    return [max(1, ceil_div(n, chunk)) for n in nblk]


# ----------------------------------------------------------------------------
# Composition of the rules above into a per-CTA schedule, with the readings
# that the pages leave open:
#  * causal with a window is the local case with right window 0; a window
#    without causal leaves the right side open (tiling chapter 3.2 code, where
#    the right bound is n_idx + window_size_right for local);
#  * total_mblocks = batch x (KV heads if packed else query heads) x m blocks
#    (section 5.2 says batch x heads x m blocks; packing makes KV heads the heads);
#  * max_splits = min(128, n blocks); the scan of section 5.2 runs 1..max_splits;
#  * one grid (m blocks, head tiles x splits, batch), launch order x fastest,
#    m block reversed for causal / local work (section 4.2 grid, section 4.4 LPT).

WINDOW_RIGHT_OPEN = 1 << 30
MAX_SPLITS = 128


def mask_flags(causal: bool, window_left: int):
    local = window_left >= 0
    return (bool(causal) and not local, local, max(window_left, 0),
            0 if causal else WINDOW_RIGHT_OPEN)


def choose_splits(policy: str, B: int, head_tiles: int, num_m_blocks: int, kv_lens, d: int,
                  block_n: int, num_sms: int, causal_or_local: bool, max_splits_opt: int = 128):
    max_kv = max(kv_lens) if kv_lens else 0
    nblk_max = ceil_div(max_kv, block_n)
    max_splits = max(1, min(min(max_splits_opt, MAX_SPLITS), max(nblk_max, 1)))
    tiles = B * head_tiles * num_m_blocks
    if policy == "fa":
        s = num_splits_heuristic(tiles, num_sms, nblk_max, num_m_blocks, max_kv * 2 * d * 2,
                                 causal_or_local, max_splits)
    elif policy == "fixed_chunk":
        s = nsplit_fixed_chunk(max_kv)
    elif policy == "min_chunk":
        s = nsplit_min_chunk(num_sms, max(tiles, 1), max_kv)
    else:
        raise ValueError(policy)
    return max(1, min(s, max_splits))


def cta_table(sq: int, kv_lens, G: int, pack_gqa: bool, head_tiles: int, block_m: int,
              block_n: int, num_m_blocks: int, num_splits_grid: int, splits_b, causal: bool,
              window_left: int, packed: bool = False):
    """Per-CTA (n_block_min, n_block_max, split word, has_work) in launch order.

    packed: the varlen scheduler's launch order (tiling chapter section 4.5, a
    warp prefix sum over the sequences' tile counts maps each launched CTA to a
    tile): only the CTAs whose split index is below their sequence's split
    count are launched, in the same relative order."""
    is_causal, local, wl, wr = mask_flags(causal, window_left)
    reverse = bool(causal) or window_left >= 0
    out = []
    for b in range(len(kv_lens)):
        for by in range(head_tiles * num_splits_grid):
            split = by % num_splits_grid
            for bx in range(num_m_blocks):
                m_block = num_m_blocks - 1 - bx if reverse else bx
                sb = splits_b[b]
                word = (sb << 16) | split
                if split >= sb:
                    if not packed:
                        out.append((0, 0, word, 0))
                    continue
                lo, hi = n_block_min_max(sq, kv_lens[b], m_block, block_m, block_n, is_causal,
                                         local, wl, wr, pack_gqa, G, split_word=word)
                out.append((lo, hi, word, 1))
    return out
