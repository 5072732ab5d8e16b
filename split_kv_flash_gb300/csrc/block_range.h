// block_range.h -- KV block ranges and the CTA -> tile map, shared by the host
// scheduler (plan.cpp) and the sm_103a kernels so that the device's ranges are
// bit-identical to the host plan.
//
// FlashAttention tiling strategy and scheduling chapter (分块策略与调度):
//   section 3.1/3.2 (block.h): causal upper bound on n blocks with the
//   seqlen_k - seqlen_q offset, local lower bound at window_size_left, PackGQA
//   rows converted back to query positions before the causal arithmetic;
//   section 5.3: a split owns ceil(range / count) consecutive blocks, clipped to
//   the range; the split word holds the split index (low 16 bits) and that
//   sequence's split count (high 16 bits);
//   section 4.2/4.4: grid (m blocks, heads x splits, batch) with the m block
//   index reversed for causal/local work (longest tile first).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SK_HD __host__ __device__ __forceinline__
#else
#define SK_HD inline
#endif

namespace sk {

constexpr int kWindowRightOpen = 1 << 30;  // "no right bound" for a window without causal
constexpr int kMaxSeqLen = 1 << 29;        // keeps every index below in int32 range

// Division truncating toward zero, as in the printed C++.
SK_HD int ceil_div_c(int a, int b) { return (a + b - 1) / b; }
SK_HD int imin(int a, int b) { return a < b ? a : b; }
SK_HD int imax(int a, int b) { return a > b ? a : b; }

struct MaskFlags {
    bool causal;       // Is_causal of block.h (a causal problem without a window)
    bool local;        // Is_local of block.h (any problem with a left window)
    int window_left;
    int window_right;
};

// User arguments (causal, window_left) -> block.h flags.  causal with a window
// is local with right window 0; a window without causal leaves the right open.
SK_HD MaskFlags mask_flags(int causal, int window_left) {
    MaskFlags f;
    f.local = window_left >= 0;
    f.causal = causal != 0 && !f.local;
    f.window_left = window_left >= 0 ? window_left : 0;
    f.window_right = causal ? 0 : kWindowRightOpen;
    return f;
}

struct BlockRange {
    int lo, hi;
};

SK_HD uint32_t split_word(int split_idx, int split_count) {
    return (uint32_t(split_count) << 16) | uint32_t(split_idx & 0xFFFF);
}

// [n_block_min, n_block_max) of one (m block, split) of a sequence.
SK_HD BlockRange n_block_range(int seqlen_q, int seqlen_k, int m_block, int kBlockM, int kBlockN,
                               const MaskFlags& f, bool pack_gqa, int G, uint32_t word) {
    int n_block_max = ceil_div_c(seqlen_k, kBlockN);
    if (f.causal || f.local) {
        int m_idx_max = (m_block + 1) * kBlockM;
        if (pack_gqa) m_idx_max = (m_idx_max - 1) / G + 1;
        const int n_idx = m_idx_max + seqlen_k - seqlen_q;
        const int n_idx_right = !f.local ? n_idx : n_idx + f.window_right;
        n_block_max = imin(n_block_max, ceil_div_c(n_idx_right, kBlockN));
    }
    int n_block_min = 0;
    if (f.local) {
        int m_idx_min = m_block * kBlockM;
        if (pack_gqa) m_idx_min = m_idx_min / G;
        const int n_idx = m_idx_min + seqlen_k - seqlen_q;
        const int n_idx_left = n_idx - f.window_left;
        n_block_min = imax(0, n_idx_left / kBlockN);
    }
    const int split_idx = int(word & 0xFFFF);
    const int split_cnt = int(word >> 16);
    const int per = ceil_div_c(n_block_max - n_block_min, split_cnt);
    n_block_min = n_block_min + split_idx * per;
    n_block_max = imin(n_block_min + per, n_block_max);
    return {n_block_min, n_block_max};
}

// Which tile one CTA of the partial kernel owns.
struct TileCoord {
    int m_block, head_tile, split, batch;
};

SK_HD TileCoord tile_of_cta(int bx, int by, int bz, int num_m_blocks, int num_splits,
                            bool reverse_m) {
    TileCoord t;
    t.m_block = reverse_m ? (num_m_blocks - 1 - bx) : bx;
    t.head_tile = by / num_splits;
    t.split = by % num_splits;
    t.batch = bz;
    return t;
}

}  // namespace sk
