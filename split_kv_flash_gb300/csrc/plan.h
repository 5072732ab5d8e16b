// plan.h -- host scheduler for the split-KV attention forward (no CUDA needed).
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/sk_attn.h"
#include "block_range.h"

namespace sk {

constexpr int kMaxVarlenBatch = 1024;   // per-sequence tables travel as kernel parameters
constexpr int kDecodeMaxRows = 64;      // decode path: <= 64 packed rows per tile
constexpr int kDefaultMaxSplits = 128;
constexpr int kMaxSplits = 128;         // the combine kernel merges at most 128 partials
// Decode path: a split must save at least this many 128-key blocks of one CTA's
// time to pay for the combine kernel (about 2.2 us against 0.75-0.8 us a block).
constexpr int kDecodeCombineBlocks = 3;
// Split choice by list schedule (sequences of different lengths): a CTA's fixed
// cost in 128-key blocks (set-up, first copies, epilogue: ~3 us against 0.75 us
// a block), the cost of a CTA past its sequence's splits, and the largest grid
// that is simulated.
constexpr double kCtaOverheadBlocks = 4.0;
constexpr double kCtaEmptyBlocks = 0.3;
constexpr long long kScheduleMaxCtas = 16384;

// Shared-memory rings of the decode kernel (K and V slots of 128 rows), also
// needed by the scheduler: the in-kernel merge stages a tile's partials there.
constexpr int decode_stages_k(int hd, int np) { return hd == 128 ? 3 : 4; }
constexpr int decode_stages_v(int hd, int np) { return hd == 128 ? (np <= 32 ? 3 : 2) : (np <= 32 ? 4 : 3); }
constexpr int decode_p_bufs(int hd, int np) { return 2; }  // P^T buffers of NP x 128 bf16
constexpr int decode_ring_bytes(int hd, int np) {
    return decode_stages_k(hd, np) * 128 * hd * 2 + decode_stages_v(hd, np) * 128 * 128 * 2;
}

struct Plan {
    // problem
    int B = 0, Hq = 0, Hkv = 0, G = 1, sq = 0, d = 0;
    int dv = 0;           // value / output width (= d except for latent attention)
    bool latent = false;  // one latent KV head: keys are its rows, values their first dv columns
    int causal = 0, window_left = -1;
    KeyWindow win{};
    bool varlen = false;       // kv lengths differ between sequences
    std::vector<int> kv_len;   // [B]
    std::vector<long long> kv_off;  // [B + 1]
    int max_kv = 0;
    // decisions
    int path = SK_PATH_AUTO;
    int kBlockM = 0, kBlockN = 128;
    bool pack_gqa = false;
    int head_tiles = 0, rows = 0, num_m_blocks = 0;
    int nblk_max = 0;
    int num_splits_policy = 1, num_splits = 1;
    std::vector<int> splits_b;  // [B] per-sequence split counts
    bool needs_combine = false;
    bool fused_combine = false;  // the partial kernel merges the splits (no combine kernel)
    bool persistent = false;     // prefill: one CTA per SM walking the tile list
    int persistent_ctas = 0;
    int l2_section = 1;          // head tiles per L2 section of the persistent tile order
    bool reverse_m = false;
    bool packed_grid = false;    // decode, varlen: 1-D grid over the CTAs with work (tiling chapter 4.5)
    int grid_x = 0, grid_y = 0, grid_z = 0;
    long long num_ctas = 0;
    int num_sms = 0;
    // workspace
    size_t ws_bytes = 0, echo_off = 0, cnt_off = 0, lse_off = 0, o_off = 0;
};

// Builds the plan; on error returns the status and sets *why.
sk_status make_plan(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int causal,
                    int window_left, const sk_attn_opts* opts, int device_num_sms, Plan* plan,
                    std::string* why);
// Latent attention (one KV head whose rows are the keys and whose first dv
// columns are the values; "The Occupancy Awakening", absorbed-MLA verify).
sk_status make_plan_latent(int B, int Hq, int q_len, const int* kv_len_host, int d, int dv, int causal,
                           int window_left, const sk_attn_opts* opts, int device_num_sms, Plan* plan,
                           std::string* why);
constexpr int kLatentDqk = 576;  // 512 latent + 64 rotary columns
constexpr int kLatentDv = 512;
constexpr int kLatentKChunksPerCopy = 3;  // 64-column K chunks per TMA copy (9 per 128-key block)

// Host-side range table (see sk_attn_plan_ranges).
void plan_ranges(const Plan& p, int32_t* out);

// The policies, exposed for tests through the plan.
int num_splits_fa_heuristic(int total_mblocks, int num_sms, int num_n_blocks, int num_m_blocks,
                            long long size_one_kv_head, bool is_causal_or_local, int max_splits);
bool should_pack_gqa(bool varlen_q, int seqlen_q, int qhead_per_khead, int block_m);
std::vector<int> per_sequence_splits(const std::vector<int>& kv_len, int block_n, int num_splits);

void plan_to_info(const Plan& p, sk_attn_plan_info* info);

}  // namespace sk
