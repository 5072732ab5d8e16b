// block_range.h -- which KV blocks a query tile needs, and which tile a CTA of
// the partial kernel owns.  Shared by the host scheduler (plan.cpp) and the
// sm_103a kernels, so that the ranges the kernels use are bit-identical to the
// host plan.
//
// The rule (FlashAttention tiling strategy and scheduling chapter, section 3:
// block-level skipping of fully masked blocks; section 5.3: a split's share of
// the range; section 6.3: packed rows are converted back to query positions
// before the mask is applied) is derived here from the key interval a tile can
// see:
//   * query i sees key j when j <= i + (kv_len - q_len) (causal, bottom-right
//     aligned) and j >= i + (kv_len - q_len) - window_left (a left window);
//   * the rows of a tile are ordered by query position, so the union of the
//     rows' visible keys is [first row's left edge, last row's right edge];
//   * the tile needs exactly the KV blocks that hold a key of that interval.
// A split t of S takes ceil(range / S) consecutive blocks starting at
// t * ceil(range / S), clipped to the range.  Every empty range is reported as
// [0, 0).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SK_HD __host__ __device__ __forceinline__
#else
#define SK_HD inline
#endif

namespace sk {

constexpr int kMaxSeqLen = 1 << 29;  // keeps every index below in int32 range

// Non-negative a, positive b.
SK_HD int div_up(int a, int b) { return (a + b - 1) / b; }
SK_HD int imin(int a, int b) { return a < b ? a : b; }
SK_HD int imax(int a, int b) { return a > b ? a : b; }

// Which keys a query row sees, relative to its diagonal key i + kv_len - q_len.
struct KeyWindow {
    int causal;       // 1: no key after the diagonal
    int has_left;     // 1: no key more than `left` before the diagonal
    int left;         // window_left when has_left
};

SK_HD KeyWindow key_window(int causal, int window_left) {
    KeyWindow w;
    w.causal = causal ? 1 : 0;
    w.has_left = window_left >= 0 ? 1 : 0;
    w.left = window_left >= 0 ? window_left : 0;
    return w;
}

struct BlockRange {
    int lo, hi;  // KV blocks [lo, hi); empty ranges are [0, 0)
};

// Split word of the partial kernel: split index in the low 16 bits, the
// sequence's split count in the high 16 bits (tiling chapter section 5.3).
SK_HD uint32_t split_word(int split_idx, int split_count) {
    return (uint32_t(split_count) << 16) | uint32_t(split_idx & 0xFFFF);
}

// KV blocks of `block_keys` keys that rows [tile * tile_rows, (tile + 1) *
// tile_rows) of a sequence need, cut to the share of split `word`.  With
// `group` > 1 the rows are packed: row r is query position r / group.
SK_HD BlockRange tile_key_blocks(int q_len, int kv_len, int tile, int tile_rows, int block_keys,
                                 const KeyWindow& w, int group, uint32_t word) {
    // (group 1 and one split are the common case: no integer division there)
    const int first_q = group == 1 ? tile * tile_rows : (tile * tile_rows) / group;
    const int last_q =
        imin(group == 1 ? tile * tile_rows + tile_rows - 1 : (tile * tile_rows + tile_rows - 1) / group, q_len - 1);
    const int shift = kv_len - q_len;  // query i's diagonal key is i + shift
    int begin = 0;
    int end = div_up(kv_len, block_keys);
    if (w.causal) {
        const int last_key = last_q + shift;
        end = last_key < 0 ? 0 : imin(end, last_key / block_keys + 1);
    }
    if (w.has_left) {
        const int first_key = first_q + shift - w.left;
        if (first_key > 0) begin = first_key / block_keys;
    }
    if (end <= begin) return {0, 0};
    const int count = int(word >> 16);
    const int idx = int(word & 0xFFFF);
    const int share = count == 1 ? end - begin : div_up(end - begin, count);
    const int lo = begin + idx * share;
    const int hi = imin(lo + share, end);
    if (hi <= lo) return {0, 0};
    return {lo, hi};
}

// Which tile one CTA of the partial kernel owns.  Grid (m blocks, head tiles x
// splits, sequences), x fastest (tiling chapter section 4.2).  With causal or
// windowed masks the m block index runs backwards, so the CTAs launched first
// own the tiles with the most KV blocks (longest processing time first,
// section 4.4).
struct TileCoord {
    int m_block, head_tile, split, batch;
};

SK_HD TileCoord tile_of_cta(int bx, int by, int bz, int num_m_blocks, int num_splits,
                            bool reverse_m) {
    TileCoord t;
    t.m_block = reverse_m ? (num_m_blocks - 1 - bx) : bx;
    t.head_tile = num_splits == 1 ? by : by / num_splits;
    t.split = num_splits == 1 ? 0 : by % num_splits;
    t.batch = bz;
    return t;
}

}  // namespace sk
