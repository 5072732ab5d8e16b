// plan.cpp -- host scheduler: path and tile choice, GQA packing, split count,
// per-sequence split counts, grid and workspace layout.  Pure C++; a plan for an
// explicit SM count needs no GPU.
#include "plan.h"

#include <math.h>
#include <string.h>

#include <algorithm>
#include <functional>

namespace sk {

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// FlashAttention tiling chapter, section 5.2: "KV head > L2 (50MB)" branch.
constexpr long long kL2SplitBytes = 50LL * 1024 * 1024;

}  // namespace

// PackGQA decision (tiling chapter section 6.2).  A tile's "fill" is the share
// of its rows that hold real queries once the rows are padded to whole tiles,
// in binary32 as the chapter defines it.  Packing G heads into the rows pays
// when the unpacked fill falls below 0.9 of the packed one.  Sequences of
// different query lengths always pack.
namespace {
float tile_fill(int rows, int tile_rows) {
    const int padded = div_up(rows, tile_rows) * tile_rows;
    return float(rows) / float(padded);
}
}  // namespace

bool should_pack_gqa(bool varlen_q, int seqlen_q, int qhead_per_khead, int block_m) {
    if (varlen_q) return true;
    const double packed_fill = tile_fill(seqlen_q * qhead_per_khead, block_m);
    return tile_fill(seqlen_q, block_m) < 0.9 * packed_fill;
}

// Tiling chapter section 5.2 (num_splits_heuristic): fill gate at 0.8 * SMs,
// L2 branch, short-K shortcut, then the smallest split count whose wave
// efficiency reaches 0.85 of the best one.
int num_splits_fa_heuristic(int total_mblocks, int num_sms, int num_n_blocks, int num_m_blocks,
                            long long size_one_kv_head, bool is_causal_or_local, int max_splits) {
    if (total_mblocks >= 0.8 * num_sms) {
        if (size_one_kv_head > kL2SplitBytes && num_m_blocks >= 2 * num_sms && !is_causal_or_local)
            return int(std::min<long long>((size_one_kv_head + kL2SplitBytes - 1) / kL2SplitBytes,
                                           (long long)max_splits));
        return 1;
    }
    if (num_n_blocks <= 4) return 1;
    std::vector<float> eff(size_t(std::max(max_splits, 0)));
    float best = 0.f;
    for (int s = 1; s <= max_splits; ++s) {
        const float waves = float(total_mblocks * s) / float(num_sms);
        const float e = waves / ceilf(waves);
        eff[size_t(s - 1)] = e;
        if (e > best) best = e;
    }
    for (int s = 1; s <= max_splits; ++s)
        if (eff[size_t(s - 1)] >= 0.85 * best) return s;
    return 1;
}

// Per-sequence split counts: one chunk ceil(n_blocks_max / S) for the batch,
// each sequence takes the chunks it needs (high 16 bits of the split word).
std::vector<int> per_sequence_splits(const std::vector<int>& kv_len, int block_n, int num_splits) {
    std::vector<int> out(kv_len.size(), 1);
    int nmax = 0;
    for (int s : kv_len) nmax = std::max(nmax, div_up(s, block_n));
    if (num_splits <= 1 || nmax == 0) return out;
    const int chunk = div_up(nmax, num_splits);
    for (size_t b = 0; b < kv_len.size(); ++b)
        out[b] = std::max(1, div_up(div_up(kv_len[b], block_n), chunk));
    return out;
}

namespace {

// SK_POLICY_FILL: the smallest per-CTA chunk (in KV blocks) for which every CTA
// of the partial kernel fits in one wave of `capacity` CTAs.  Returns S.
int fill_policy(const Plan& p, int capacity, int max_splits) {
    const long long tiles = (long long)p.B * p.head_tiles * p.num_m_blocks;
    if (tiles >= capacity || p.nblk_max <= 1) return 1;
    int best = 1;
    // S candidates from large to small; the first whose per-sequence counts
    // fit in one wave wins (larger S = smaller chunk per CTA).
    const int smax = std::min(max_splits, p.nblk_max);
    for (int S = smax; S >= 1; --S) {
        const std::vector<int> sb = per_sequence_splits(p.kv_len, p.kBlockN, S);
        long long ctas = 0;
        for (int c : sb) ctas += (long long)c * p.head_tiles * p.num_m_blocks;
        if (ctas <= capacity) { best = S; break; }
    }
    // drop splits that would only repeat the same chunk size
    const int chunk = div_up(p.nblk_max, best);
    return div_up(p.nblk_max, chunk);
}

// Finishing time, in KV blocks, of the partial kernel's CTAs when the SMs take
// them in launch order (x = m block fastest, then head tile x split, then
// sequence), each as soon as one frees up; a CTA costs its blocks plus
// kCtaOverheadBlocks, one past its sequence's splits kCtaEmptyBlocks.
double list_schedule_blocks(const Plan& p, int S, int sms) {
    const std::vector<int> sb = per_sequence_splits(p.kv_len, p.kBlockN, S);
    int grid_splits = 1;  // the grid's split dimension
    for (int c : sb) grid_splits = std::max(grid_splits, c);
    std::vector<double> free_at(size_t(std::max(sms, 1)), 0.0);
    std::make_heap(free_at.begin(), free_at.end(), std::greater<double>());
    double makespan = 0.0;
    for (int b = 0; b < p.B; ++b) {
        for (int y = 0; y < p.head_tiles * grid_splits; ++y) {
            const int split = y % grid_splits;
            for (int x = 0; x < p.num_m_blocks; ++x) {
                double cost = kCtaEmptyBlocks;
                if (split < sb[size_t(b)]) {
                    const int m = p.reverse_m ? p.num_m_blocks - 1 - x : x;
                    const BlockRange r = tile_key_blocks(p.sq, p.kv_len[size_t(b)], m, p.kBlockM, p.kBlockN, p.win,
                                                         p.pack_gqa ? p.G : 1, split_word(split, sb[size_t(b)]));
                    cost = double(r.hi - r.lo) + kCtaOverheadBlocks;
                }
                std::pop_heap(free_at.begin(), free_at.end(), std::greater<double>());
                free_at.back() += cost;
                makespan = std::max(makespan, free_at.back());
                std::push_heap(free_at.begin(), free_at.end(), std::greater<double>());
            }
        }
    }
    return makespan;
}

// Sequences of different lengths: one wave (the fill policy) can leave the
// longest sequences' CTAs streaming alone at the end.  Among the fill choice and
// 2, 4, 8, 16 splits, take the one whose list schedule finishes first; a
// candidate must win by more than 3 % (fewer splits: less to merge).
int refine_by_schedule(const Plan& p, int S_fill, int max_splits) {
    bool varied = false;
    for (int L : p.kv_len) varied = varied || L != p.kv_len[0];
    if (!varied) return S_fill;
    int best = S_fill;
    double best_t = list_schedule_blocks(p, S_fill, p.num_sms);
    const int cands[] = {1, 2, 4, 8, 16};
    for (int S : cands) {
        if (S == S_fill || S > max_splits || S > std::max(p.nblk_max, 1)) continue;
        const long long ctas = (long long)p.B * p.head_tiles * S * p.num_m_blocks;
        if (ctas > kScheduleMaxCtas) continue;
        const double t = list_schedule_blocks(p, S, p.num_sms);
        if (t < 0.97 * best_t) {
            best = S;
            best_t = t;
        }
    }
    return best;
}

}  // namespace

namespace {
sk_status make_plan_ex(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int dv, bool latent,
                       int causal, int window_left, const sk_attn_opts* opts_in, int device_num_sms, Plan* out,
                       std::string* why);
}  // namespace

sk_status make_plan(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int causal,
                    int window_left, const sk_attn_opts* opts, int device_num_sms, Plan* out,
                    std::string* why) {
    return make_plan_ex(B, Hq, Hkv, q_len, kv_len_host, d, d, false, causal, window_left, opts, device_num_sms,
                        out, why);
}

sk_status make_plan_latent(int B, int Hq, int q_len, const int* kv_len_host, int d, int dv, int causal,
                           int window_left, const sk_attn_opts* opts, int device_num_sms, Plan* out,
                           std::string* why) {
    return make_plan_ex(B, Hq, 1, q_len, kv_len_host, d, dv, true, causal, window_left, opts, device_num_sms,
                        out, why);
}

namespace {
sk_status make_plan_ex(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int dv, bool latent,
                       int causal, int window_left, const sk_attn_opts* opts_in, int device_num_sms, Plan* out,
                       std::string* why) {
    sk_attn_opts opts;
    memset(&opts, 0, sizeof opts);
    if (opts_in) opts = *opts_in;
    Plan p;
    auto fail = [&](sk_status s, const char* msg) {
        if (why) *why = msg;
        return s;
    };
    if (B <= 0 || B > 65535) return fail(SK_ERR_INVALID_ARG, "B must be in [1, 65535]");
    if (Hq <= 0 || Hkv <= 0) return fail(SK_ERR_INVALID_ARG, "head counts must be positive");
    if (Hq % Hkv != 0) return fail(SK_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
    if (q_len < 0 || q_len > kMaxSeqLen) return fail(SK_ERR_INVALID_ARG, "q_len out of range");
    if (!kv_len_host) return fail(SK_ERR_INVALID_ARG, "kv_len_host is NULL");
    if (latent) {
        if (d != kLatentDqk || dv != kLatentDv)
            return fail(SK_ERR_UNSUPPORTED, "latent attention: key width 576 and value width 512 only");
    } else if (d != 64 && d != 128) {
        return fail(SK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    }
    if (opts.policy < 0 || opts.policy > SK_POLICY_MIN_CHUNK)
        return fail(SK_ERR_INVALID_ARG, "unknown split policy");
    if (opts.force_path < 0 || opts.force_path > SK_PATH_PREFILL)
        return fail(SK_ERR_INVALID_ARG, "unknown path");
    if (opts.force_pack_gqa < -1 || opts.force_pack_gqa > 1)
        return fail(SK_ERR_INVALID_ARG, "force_pack_gqa must be -1, 0 or 1");
    if (opts.max_splits < 0 || opts.force_num_splits < 0 || opts.num_sms < 0 ||
        opts.wait_timeout_us < 0)
        return fail(SK_ERR_INVALID_ARG, "negative option");
    if (opts.combine_mode < SK_COMBINE_AUTO || opts.combine_mode > SK_COMBINE_IN_KERNEL)
        return fail(SK_ERR_INVALID_ARG, "unknown combine mode");
    if (opts.prefill_schedule < SK_SCHEDULE_AUTO || opts.prefill_schedule > SK_SCHEDULE_PERSISTENT)
        return fail(SK_ERR_INVALID_ARG, "unknown prefill schedule");
    if (opts.tile_map < SK_TILE_MAP_AUTO || opts.tile_map > SK_TILE_MAP_PACKED)
        return fail(SK_ERR_INVALID_ARG, "unknown tile map");

    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.sq = q_len; p.d = d;
    p.dv = dv;
    p.latent = latent;
    p.causal = causal ? 1 : 0;
    p.window_left = window_left < 0 ? -1 : window_left;
    p.win = key_window(p.causal, p.window_left);
    p.kv_len.assign(kv_len_host, kv_len_host + B);
    p.kv_off.assign(size_t(B) + 1, 0);
    long long total = 0;
    for (int b = 0; b < B; ++b) {
        if (p.kv_len[b] < 0 || p.kv_len[b] > kMaxSeqLen)
            return fail(SK_ERR_INVALID_ARG, "kv_len entries must be in [0, 2^29]");
        p.kv_off[size_t(b)] = total;
        total += p.kv_len[b];
        p.max_kv = std::max(p.max_kv, p.kv_len[b]);
        if (p.kv_len[b] != p.kv_len[0]) p.varlen = true;
    }
    p.kv_off[size_t(B)] = total;
    if (total >= (1LL << 31)) return fail(SK_ERR_UNSUPPORTED, "at most 2^31 - 1 KV rows in total");
    if (p.varlen && B > kMaxVarlenBatch)
        return fail(SK_ERR_UNSUPPORTED, "sequences of different lengths: at most 1024 per call");

    p.num_sms = opts.num_sms > 0 ? opts.num_sms : device_num_sms;
    if (p.num_sms <= 0) return fail(SK_ERR_INVALID_ARG, "unknown SM count");

    // GQA packing (tiling chapter section 6.2), judged against the 128-row tile.
    bool pack = should_pack_gqa(false, q_len, p.G, 128);
    if (opts.force_pack_gqa == 1) pack = true;
    if (opts.force_pack_gqa == -1) pack = false;
    if (latent) pack = true;  // every query head reads the one latent head
    if (p.G == 1) pack = false;
    p.pack_gqa = pack;
    p.head_tiles = pack ? Hkv : Hq;
    const long long rows = (long long)q_len * (pack ? p.G : 1);
    if (rows > kMaxSeqLen) return fail(SK_ERR_UNSUPPORTED, "q_len * G too large");
    p.rows = int(rows);

    // Kernel choice: at most 64 packed rows -> decode kernel (KV rows on MMA M).
    int path = latent ? int(SK_PATH_LATENT) : opts.force_path;
    if (path == SK_PATH_AUTO) path = (p.rows <= kDecodeMaxRows) ? SK_PATH_DECODE : SK_PATH_PREFILL;
    if (path == SK_PATH_DECODE && p.rows > kDecodeMaxRows)
        return fail(SK_ERR_UNSUPPORTED, "decode path holds at most 64 packed rows per tile");
    p.path = path;
    p.kBlockN = 128;
    if (path == SK_PATH_LATENT) {
        // Packed rows per tile (keys on the MMA M axis): 32 is the most that
        // leaves room for the K and V rings next to Q^T, and streams each latent
        // block for twice the rows.  Short ranges (at most 8 blocks of 128 keys)
        // take 16: twice the tiles fill the SMs with fewer splits (often none,
        // and then no combine), which measured faster there (verify H=64 q=33
        // 161 keys: 11.9 vs 19.6 us; q=9 521 keys: 15.9 vs 19.2 us).
        p.kBlockM = (p.rows <= 16 || div_up(p.max_kv, 128) <= 8) ? 16 : 32;
    } else if (path == SK_PATH_DECODE) {
        p.kBlockM = std::max(16, (p.rows + 15) / 16 * 16);
    } else {
        // Prefill kernel: 256-row tiles, two 128-row halves that share each K/V block.
        p.kBlockM = 256;
    }
    p.num_m_blocks = p.rows == 0 ? 0 : div_up(p.rows, p.kBlockM);
    p.nblk_max = div_up(p.max_kv, p.kBlockN);
    p.reverse_m = p.causal || p.window_left >= 0;

    // Split count.
    const int max_splits = std::max(
        1, std::min(std::min(opts.max_splits > 0 ? opts.max_splits : kDefaultMaxSplits, kMaxSplits),
                    std::max(p.nblk_max, 1)));
    int S = 1;
    const long long tiles = (long long)B * p.head_tiles * p.num_m_blocks;
    if (opts.force_num_splits > 0) {
        S = std::min(std::min(opts.force_num_splits, kMaxSplits), std::max(p.nblk_max, 1));
    } else {
        switch (opts.policy) {
            case SK_POLICY_FA_HEURISTIC: {
                const long long kv_head_bytes = (long long)p.max_kv * (d + dv) * 2;
                S = num_splits_fa_heuristic(int(std::min<long long>(tiles, 1LL << 30)), p.num_sms,
                                            p.nblk_max, p.num_m_blocks, kv_head_bytes,
                                            p.causal || p.window_left >= 0, max_splits);
                break;
            }
            case SK_POLICY_FIXED_CHUNK:
                S = std::max(1, std::min(32, div_up(p.max_kv, 2048)));
                break;
            case SK_POLICY_MIN_CHUNK: {
                const int fill = int(std::min<long long>(
                    (2LL * p.num_sms + std::max(tiles, 1LL) - 1) / std::max(tiles, 1LL), 1 << 20));
                S = std::max(1, std::min(fill, p.max_kv / 256));
                break;
            }
            default:
                S = fill_policy(p, p.num_sms, max_splits);
                // Several sequences of different lengths (decode path): the split
                // count whose schedule finishes first, several waves allowed
                // (varlen decode B=16: 369 -> 245 us; B=32: 619 -> 541 us).
                if (p.path == SK_PATH_DECODE && B > 1) S = refine_by_schedule(p, S, max_splits);
                // Splitting shortens the longest CTA by nblk_max - chunk blocks
                // and adds the combine kernel; on the decode path that pays
                // only from kDecodeCombineBlocks blocks on (verify q=9 over 137
                // keys: one split 4.9 us, two 6.3 us).  Latent blocks take
                // about 2.5 us each, so that path splits as the fill says.
                if (S > 1 && p.path == SK_PATH_DECODE &&
                    p.nblk_max - div_up(p.nblk_max, S) < kDecodeCombineBlocks)
                    S = 1;
                break;
        }
        S = std::max(1, std::min(S, max_splits));
    }
    p.num_splits_policy = S;
    p.splits_b = per_sequence_splits(p.kv_len, p.kBlockN, S);
    p.num_splits = 1;
    for (int c : p.splits_b) p.num_splits = std::max(p.num_splits, c);
    p.needs_combine = p.num_splits > 1;
    // In-kernel merge (decode path, on request): the last split CTA of a tile
    // stages every split's partial rows of the tile in its K/V rings, so they
    // must fit there.  The default keeps the separate combine kernel, which
    // measured faster (it merges a tile's rows on many SMs at once).
    if (p.needs_combine && p.path == SK_PATH_DECODE && opts.combine_mode == SK_COMBINE_IN_KERNEL) {
        const long long staged = (long long)p.num_splits * p.rows * d * 4;
        // The merge stages the partials in the K/V rings and its weights
        // (rows x splits floats) in the P^T buffers.
        const long long weights = (long long)p.num_splits * p.rows * 4;
        p.fused_combine = staged <= decode_ring_bytes(d, p.kBlockM) &&
                          weights <= (long long)decode_p_bufs(d, p.kBlockM) * p.kBlockM * 128 * 2;
    }

    // Persistent prefill (tiling chapter sections 4.3-4.4): one CTA per SM over
    // the tile list, when Q halves can come by TMA (whole 128-row boxes).
    {
        const int gp = p.pack_gqa ? p.G : 1;
        const long long tiles = (long long)p.num_m_blocks * p.head_tiles * p.num_splits * B;
        p.persistent = !latent && p.path == SK_PATH_PREFILL && opts.prefill_schedule == SK_SCHEDULE_PERSISTENT &&
                       128 % gp == 0 && (long long)B * q_len < (1LL << 31) && tiles > 0 && tiles < (1LL << 30);
        if (p.persistent) {
            p.persistent_ctas = int(std::min<long long>(tiles, p.num_sms));
            // Section 4.4: nearest_power_of_2(32 MB / size of one KV head) heads,
            // times the query heads per KV head when those are separate tiles
            // (power of two taken downwards, so that a section fits the budget).
            const long long kv_head_bytes = std::max<long long>(1, (long long)p.max_kv * (d + dv) * 2);
            long long per = (32LL << 20) / kv_head_bytes;
            long long pow2 = 1;
            while (pow2 * 2 <= per) pow2 *= 2;
            const long long sec = pow2 * (p.pack_gqa ? 1 : p.G);
            p.l2_section = int(std::max<long long>(1, std::min<long long>(sec, (long long)B * p.head_tiles)));
        }
    }

    p.grid_x = p.num_m_blocks;
    p.grid_y = p.head_tiles * p.num_splits;
    p.grid_z = B;
    if (p.grid_y > 65535) return fail(SK_ERR_UNSUPPORTED, "heads x splits exceeds 65535");
    p.num_ctas = (long long)p.grid_x * p.grid_y * p.grid_z;
    // Packed tile map (tiling chapter section 4.5, the varlen scheduler): only
    // the CTAs that have work, in the grid's order; sequence b owns head_tiles x
    // splits_b x num_m_blocks consecutive CTAs.
    if (opts.tile_map == SK_TILE_MAP_PACKED && p.path == SK_PATH_DECODE && !latent && B > 1) {
        long long work = 0;
        for (int b = 0; b < B; ++b) work += p.splits_b[size_t(b)];
        work *= (long long)p.head_tiles * p.num_m_blocks;
        if (work < p.num_ctas && work < (1LL << 31)) {
            p.packed_grid = true;
            p.grid_x = int(work);
            p.grid_y = 1;
            p.grid_z = 1;
            p.num_ctas = work;
        }
    }

    // Workspace: [status header 256 B][plan echo][LSE partials][O partials].
    size_t off = 256;
    p.echo_off = off;
    off = align_up(off + size_t(p.num_ctas) * 16, 256);
    p.cnt_off = off;
    if (p.fused_combine) off = align_up(off + size_t(B) * p.head_tiles * p.num_m_blocks * 4, 256);
    if (p.persistent) off = align_up(off + 2 * 4, 256);
    p.lse_off = off;
    if (p.needs_combine) {
        const size_t rows_all = size_t(p.num_splits) * B * Hq * size_t(q_len);
        off = align_up(off + rows_all * 4, 256);
        p.o_off = off;
        off = align_up(off + rows_all * size_t(dv) * 4, 256);
    } else {
        p.o_off = off;
    }
    p.ws_bytes = off;
    *out = std::move(p);
    return SK_OK;
}

}  // namespace

void plan_ranges(const Plan& p, int32_t* out) {
    long long idx = 0;
    const int gy = p.packed_grid ? p.head_tiles * p.num_splits : p.grid_y;
    const int gz = p.packed_grid ? p.B : p.grid_z;
    const int gx = p.packed_grid ? p.num_m_blocks : p.grid_x;
    for (int bz = 0; bz < gz; ++bz)
        for (int by = 0; by < gy; ++by)
            for (int bx = 0; bx < gx; ++bx) {
                const TileCoord t = tile_of_cta(bx, by, bz, p.num_m_blocks, p.num_splits, p.reverse_m);
                const int sb = p.splits_b[size_t(t.batch)];
                if (p.packed_grid && t.split >= sb) continue;  // the packed grid has no such CTA
                const uint32_t word = split_word(t.split, sb);
                int32_t* e = out + (idx++) * 4;
                if (t.split >= sb) {
                    e[0] = 0; e[1] = 0; e[2] = int32_t(word); e[3] = 0;
                    continue;
                }
                const BlockRange r = tile_key_blocks(p.sq, p.kv_len[size_t(t.batch)], t.m_block,
                                                     p.kBlockM, p.kBlockN, p.win, p.pack_gqa ? p.G : 1,
                                                     word);
                e[0] = r.lo; e[1] = r.hi; e[2] = int32_t(word); e[3] = 1;
            }
}

void plan_to_info(const Plan& p, sk_attn_plan_info* info) {
    memset(info, 0, sizeof *info);
    info->path = p.path;
    info->kBlockM = p.kBlockM;
    info->kBlockN = p.kBlockN;
    info->pack_gqa = p.pack_gqa ? 1 : 0;
    info->head_tiles = p.head_tiles;
    info->rows_per_head_tile = p.rows;
    info->num_m_blocks = p.num_m_blocks;
    info->num_splits = p.num_splits;
    info->num_splits_policy = p.num_splits_policy;
    info->num_n_blocks_max = p.nblk_max;
    info->grid_x = p.grid_x;
    info->grid_y = p.grid_y;
    info->grid_z = p.grid_z;
    info->num_ctas = p.num_ctas;
    info->needs_combine = p.needs_combine ? 1 : 0;
    info->workspace_bytes = p.ws_bytes;
    info->echo_offset = p.echo_off;
    info->lse_part_offset = p.lse_off;
    info->o_part_offset = p.o_off;
    info->combine_in_kernel = p.fused_combine ? 1 : 0;
    info->counter_offset = p.cnt_off;
    info->persistent = p.persistent ? 1 : 0;
    info->persistent_ctas = p.persistent_ctas;
    info->l2_section_heads = p.l2_section;
    info->tile_map = p.packed_grid ? SK_TILE_MAP_PACKED : SK_TILE_MAP_GRID;
}

}  // namespace sk
