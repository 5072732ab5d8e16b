// fwd_prefill_persistent.cu -- persistent form of the 256-row prefill kernel
// (prefill, large packed GQA groups), sm_103a.
//
// One CTA per SM walks a list of tiles (m block, head tile, split, sequence)
// instead of owning one (FlashAttention tiling strategy and scheduling chapter,
// section 4.3 persistent tile schedulers, section 4.4 dynamic persistent
// scheduler):
//   * tile order: longest processing time first (the m block index runs
//     backwards under a causal or windowed mask, so the tiles with the most KV
//     blocks start first), within L2 sections of head tiles whose K/V fit a
//     32 MB budget (section 4.4: sections of nearest_power_of_2(32 MB / size
//     of one KV head) heads, times the query heads per KV head when they are
//     not packed);
//   * each CTA starts on tile blockIdx.x and then takes tiles from an atomic
//     counter in the workspace; the producer warp fetches the next index while
//     the current tile is still running and hands the tile to the other warps
//     through a two-slot ring in shared memory;
//   * across tiles the K/V rings keep streaming, the next tile's Q halves load
//     as soon as the last QK^T of the previous tile has read them, and the next
//     tile's first QK^T runs while the softmax warps write the previous tile's
//     outputs, so a tile pays no launch, barrier set-up or TMEM allocation and
//     its first loads overlap the previous tile's epilogue.  The next tile's
//     first PV (which overwrites O_t) waits for P_t of that tile, which the
//     same softmax warps produce only after reading O_t out: no extra barrier.
// Per tile the work is that of the single-tile kernel (fwd_prefill.cu): two
// 128-row halves that share each K/V block, S_t = Q_t K^T and O_t += P_t V by
// tcgen05 into TMEM, online softmax with one thread per query row, blocks
// visited from the last one down.  Outputs leave with direct 16-byte stores
// from registers (the Q buffers are already refilled for the next tile).
//
// Warp roles (320 threads): warp 0 producer (tile fetch, Q halves, K/V rings),
// warp 1 TMEM owner and MMA issuer, warps 2-5 softmax + epilogue of half 0,
// warps 6-9 of half 1.  Per-tile barrier phases are counted in each role over
// the tiles that have work (a split beyond a sequence's split count has none).
#include <math.h>

#include "fwd_common.cuh"
#include "kv_producer.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kHalves = 2;
constexpr int kThreads = 64 + 128 * kHalves;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
struct PersistCfg {
    static constexpr int kStagesK = HD == 128 ? 3 : 4;
    static constexpr int kStagesV = HD == 128 ? 2 : 4;
    static constexpr int kKBytes = 128 * HD * 2;
    static constexpr int kVBytes = 128 * HD * 2;
    static constexpr int kQBytes = 128 * HD * 2;  // one half
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kHalves * kQBytes;
    static constexpr int kOffV = kOffK + kStagesK * kKBytes;
    static constexpr int kOffBars = kOffV + kStagesV * kVBytes;
    // kfull[K] kempty[K] vfull[V] vempty[V], then per half qfull qfree sfull pfull
    // ofinal, then tile_full[2] tile_empty[2], never, drain
    static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 5 * kHalves + 4 + 2;
    static constexpr int kOffTile = kOffBars + kNumBars * 8;  // int4 tile[2]
    static constexpr int kOffMisc = kOffTile + 32;            // tmem base, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr int kSlack = (kSmemBytes + 1024 <= 232448) ? 1024 : 0;
    static constexpr int kSmemAlloc = kSmemBytes + kSlack;
    static constexpr int kTmemCols = 512;  // S_0, S_1, O_0, O_1
    static constexpr int kPCol = 64;
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// Tile list: L2 sections of `sec` (sequence, head tile) pairs, pairs ordered by
// sequence then head tile; inside a section, m blocks (descending when masked),
// then pairs, then splits.  Returns {m_block, head_tile, split, sequence}.
struct TileList {
    int ntiles, nm, S, head_tiles, B, sec, masked;
};

__device__ __forceinline__ int4 tile_at(const TileList& L, int t) {
    const int pairs = L.B * L.head_tiles;
    const int per_sec = L.sec * L.nm * L.S;
    const int si = t / per_sec;
    const int off = t - si * per_sec;
    const int cs = min(L.sec, pairs - si * L.sec);
    const int mr = off / (cs * L.S);
    const int rem = off - mr * (cs * L.S);
    const int pair = si * L.sec + rem / L.S;
    const int split = rem % L.S;
    const int m_block = L.masked ? L.nm - 1 - mr : mr;
    return make_int4(m_block, pair % L.head_tiles, split, pair / L.head_tiles);
}

// Per-tile quantities every role derives the same way.
struct TileWork {
    int m_block, ht, split, b, sb, sk, kv_off;
    bool work;  // split < the sequence's split count
    BlockRange br;
    int nblocks;
    int first[kHalves], count[kHalves], rows_h[kHalves];
};

template <class Seqs>
__device__ __forceinline__ TileWork tile_work(const FwdParams& p, const Seqs& seqs, int4 ti) {
    TileWork w;
    w.m_block = ti.x;
    w.ht = ti.y;
    w.split = ti.z;
    w.b = ti.w;
    w.sb = seqs.splits_of(w.b);
    w.work = w.split < w.sb;
    w.sk = seqs.seq_len(w.b);
    w.kv_off = seqs.seq_off(w.b);
    w.br = w.work ? tile_key_blocks(p.sq, w.sk, w.m_block, p.kBlockM, p.kBlockN, p.win, p.pack_gqa ? p.G : 1,
                                    split_word(w.split, w.sb))
                  : BlockRange{0, 0};
    w.nblocks = w.br.hi > w.br.lo ? w.br.hi - w.br.lo : 0;
    const int m0 = w.m_block * (128 * kHalves);
#pragma unroll
    for (int t = 0; t < kHalves; ++t) {
        w.rows_h[t] = max(0, min(128, p.rows - (m0 + 128 * t)));
        const BlockRange hr = tile_key_blocks(p.sq, w.sk, w.m_block * kHalves + t, 128, p.kBlockN, p.win,
                                              p.pack_gqa ? p.G : 1, split_word(0, 1));
        const int lo = max(hr.lo, w.br.lo), hi = min(hr.hi, w.br.hi);
        w.count[t] = (w.work && w.rows_h[t] > 0 && hi > lo) ? hi - lo : 0;
        w.first[t] = w.count[t] > 0 ? w.br.hi - hi : 0;
    }
    return w;
}

template <int HD, class Seqs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_prefill_persistent_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                                  const __grid_constant__ Seqs seqs, const TileList tl) {
    using C = PersistCfg<HD>;
    constexpr int KST = C::kStagesK;
    constexpr int VST = C::kStagesV;
    constexpr int NB0 = 2 * KST + 2 * VST;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (C::kSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0u, (kKernPrefill << 8) | kSiteSmemAlign);
        return;
    }
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t bars = sbase + C::kOffBars;
    auto bar_kfull = [&](int s) { return bars + 8u * s; };
    auto bar_kempty = [&](int s) { return bars + 8u * (KST + s); };
    auto bar_vfull = [&](int s) { return bars + 8u * (2 * KST + s); };
    auto bar_vempty = [&](int s) { return bars + 8u * (2 * KST + VST + s); };
    auto bar_qfull = [&](int t) { return bars + 8u * (NB0 + t); };
    auto bar_qfree = [&](int t) { return bars + 8u * (NB0 + 2 + t); };
    auto bar_sfull = [&](int t) { return bars + 8u * (NB0 + 4 + t); };
    auto bar_pfull = [&](int t) { return bars + 8u * (NB0 + 6 + t); };
    auto bar_ofinal = [&](int t) { return bars + 8u * (NB0 + 8 + t); };
    auto bar_tfull = [&](int s) { return bars + 8u * (NB0 + 10 + s); };
    auto bar_tempty = [&](int s) { return bars + 8u * (NB0 + 12 + s); };
    const uint32_t bar_never = bars + 8u * (NB0 + 14);
    const uint32_t bar_drain = bars + 8u * (NB0 + 15);
    // Tile ring: plain shared stores / loads ordered by the mbarriers (release
    // on arrive, acquire on wait; both are compiler memory barriers).
    int* tile_slot = reinterpret_cast<int*>(smem + C::kOffTile);
    auto put_tile = [&](int slot, int4 v) {
        tile_slot[4 * slot] = v.x;
        tile_slot[4 * slot + 1] = v.y;
        tile_slot[4 * slot + 2] = v.z;
        tile_slot[4 * slot + 3] = v.w;
    };
    auto get_tile = [&](int slot) {
        return make_int4(tile_slot[4 * slot], tile_slot[4 * slot + 1], tile_slot[4 * slot + 2], tile_slot[4 * slot + 3]);
    };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    auto stage_k = [&](int s) { return sbase + C::kOffK + uint32_t(s) * C::kKBytes; };
    auto stage_v = [&](int s) { return sbase + C::kOffV + uint32_t(s) * C::kVBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(bar_vfull(s), 1);
            mbar_init(bar_vempty(s), 1);
        }
        for (int t = 0; t < kHalves; ++t) {
            mbar_init(bar_qfull(t), 1);   // TMA transaction
            mbar_init(bar_qfree(t), 1);   // MMA commit after the tile's last QK^T of the half
            mbar_init(bar_sfull(t), 1);
            mbar_init(bar_pfull(t), 4);   // one arrival per softmax warp
            mbar_init(bar_ofinal(t), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_tfull(s), 1);
            mbar_init(bar_tempty(s), 1 + 4 * kHalves);  // the MMA warp and every softmax warp
        }
        mbar_init(bar_never, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmQ);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    const uint32_t tmem = *tmem_holder;
    auto tS = [&](int t) { return tmem + uint32_t(t) * 128u; };
    auto tO = [&](int t) { return tmem + 256u + uint32_t(t) * 128u; };
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int grid_y = p.head_tiles * p.num_splits;

    if (warp == 0) {
        // ===================== producer: tiles, Q halves, K/V rings
        const bool leader = elect_one();
        const KvRing kr{stage_k(0), uint32_t(C::kKBytes), bar_kfull(0), bar_kempty(0), KST};
        const KvRing vr{stage_v(0), uint32_t(C::kVBytes), bar_vfull(0), bar_vempty(0), VST};
        int t = blockIdx.x;
        int kpos = 0, vpos = 0;  // ring positions (blocks loaded so far)
        int kw = 0;              // tiles with work so far
        bool ok = true;
        for (int k = 0;; ++k) {
            const int slot = k & 1;
            if (k >= 2) ok = mbar_wait(bar_tempty(slot), ((k - 2) >> 1) & 1, wc, (kKernPrefill << 8) | kSiteProducerEmpty) && ok;
            const bool end = t >= tl.ntiles || !ok;
            const int4 ti = end ? make_int4(0, 0, 0, -1) : tile_at(tl, t);
            int next = 0;
            if (leader) {
                if (!end) next = int(atomicAdd(p.counters, 1u)) + int(gridDim.x);
                put_tile(slot, ti);
                mbar_arrive(bar_tfull(slot));
            }
            next = __shfl_sync(0xffffffffu, next, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
            if (end) break;
            const TileWork w = tile_work(p, seqs, ti);
            if (p.echo_plan && leader) {
                const int bx = tl.masked ? tl.nm - 1 - w.m_block : w.m_block;
                const long long lin = bx + (long long)tl.nm * (w.ht * p.num_splits + w.split + (long long)grid_y * w.b);
                *reinterpret_cast<int4*>(p.echo + lin * 4) =
                    make_int4(w.work ? w.br.lo : 0, w.work ? w.br.hi : 0, int(split_word(w.split, w.sb)), w.work ? 1 : 0);
            }
            if (w.work) {
                const int m0 = w.m_block * (128 * kHalves);
#pragma unroll
                for (int h = 0; h < kHalves; ++h) {
                    // Q_h of the previous tile has had its last QK^T.
                    if (kw >= 1) ok = mbar_wait(bar_qfree(h), (kw - 1) & 1, wc, (kKernPrefill << 8) | kSiteProducerEmpty) && ok;
                    if (leader && ok) {
                        mbar_arrive_expect_tx(bar_qfull(h), C::kQBytes);
                        const int qrow = w.b * p.sq + (m0 + 128 * h) / p.q_gp;
#pragma unroll
                        for (int c = 0; c < HD / 64; ++c)
                            tma_load_4d(sQ + uint32_t(h * C::kQBytes + c * 16384), &tmQ, bar_qfull(h), c * 64, 0, w.ht,
                                        qrow, l2_policy_evict_first());
                    }
                }
                __syncwarp();
                const int kvh = p.pack_gqa ? w.ht : w.ht / p.G;
                ok = produce_kv_tile<HD>(&tmK, &tmV, kr, vr, kpos, w.nblocks, kvh * HD, w.kv_off + w.br.lo * 128, true,
                                         l2_policy_evict_last(), wc, (kKernPrefill << 8) | kSiteProducerEmpty, leader,
                                         kpos, vpos) && ok;
                ++kw;
            }
            t = next;
        }
        // Every CTA reaches the end of the list once; the last one re-arms the
        // counters for the next call on this workspace.
        griddep_launch_dependents();
        if (leader) {
            const uint32_t done = atomicAdd(p.counters + 1, 1u);
            if (done + 1u == gridDim.x) {
                p.counters[0] = 0u;
                p.counters[1] = 0u;
            }
        }
        drain_ring(kr, kpos, wc.limit_ns);
        drain_ring(vr, vpos, wc.limit_ns);
        if (kw >= 1)
            for (int h = 0; h < kHalves; ++h) mbar_drain(bar_qfull(h), (kw - 1) & 1, wc.limit_ns);
    } else if (warp == 1) {
        // ===================== MMA issuer (whole warp, one elected lane issues)
        const bool leader = elect_one();
        constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_pv = make_idesc_bf16(128, HD, false, true);
        const uint64_t qdesc0 = make_sdesc_sw128(sQ, 16, 1024);
        const uint64_t kdesc0 = make_sdesc_sw128(stage_k(0), 16, 1024);
        const uint64_t vdesc0 = make_sdesc_sw128(stage_v(0), 16384, 1024);
        bool ok = true;
        if (p.inject_stall) {
            const WaitCtl wc_half{wc.abort_flag, wc.status, wc.limit_ns / 2};
            ok = mbar_wait(bar_never, 0, wc_half, (kKernPrefill << 8) | kSiteInjected);
        }
        int g = 0;                   // ring position of the tile's first block
        int kw = 0;                  // tiles with work so far
        int sq_cnt[kHalves] = {0, 0};  // pfull phases consumed per half
        for (int k = 0;; ++k) {
            const int slot = k & 1;
            mbar_wait(bar_tfull(slot), (k >> 1) & 1, wc, (kKernPrefill << 8) | kSiteMmaQ);
            const int4 ti = get_tile(slot);
            __syncwarp();
            if (leader) mbar_arrive(bar_tempty(slot));
            if (ti.w < 0) break;
            const TileWork w = tile_work(p, seqs, ti);
            if (!w.work) continue;
            auto active = [&](int t, int j) { return j >= w.first[t] && j < w.first[t] + w.count[t]; };
            // A half with no block this tile still takes its Q phase and hands
            // the buffer back.
#pragma unroll
            for (int t = 0; t < kHalves; ++t) {
                if (w.count[t] == 0) {
                    ok = mbar_wait(bar_qfull(t), kw & 1, wc, (kKernPrefill << 8) | kSiteMmaQ) && ok;
                    __syncwarp();
                    if (leader) umma_commit(bar_qfree(t));
                }
            }
            int zeroed_step = -1;
            auto issue_pv = [&](int t, int j) {
                const int i = j - w.first[t];
                const int pos = g + j;
                const int s = pos % VST;
                // P_t of this block is in TMEM.  For the tile's first PV this also
                // orders it after the epilogue that read O_t of the previous tile
                // (the same softmax warps, earlier in program order).
                bool good = mbar_wait(bar_pfull(t), sq_cnt[t] & 1, wc, (kKernPrefill << 8) | kSiteMmaPFull);
                ++sq_cnt[t];
                good = mbar_wait(bar_vfull(s), (pos / VST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull) && good;
                const int tail_row = w.sk - (w.br.hi - 1 - j) * 128;
                if (good && tail_row < 128 && zeroed_step != j) zero_rows<HD>(stage_v(s), tail_row, lane);
                zeroed_step = j;
                tc_fence_after();
                __syncwarp();
                if (leader) {
                    if (good && ok) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t bd = vdesc0 + uint64_t((s * C::kVBytes + kk * 2048) >> 4);
                            umma_bf16_ts(tO(t), tS(t) + C::kPCol + kk * 8, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    if (i == w.count[t] - 1) umma_commit(bar_ofinal(t));
                }
            };
            int issued[kHalves] = {0, 0};
            for (int j = 0; j <= w.nblocks; ++j) {
                bool k_ready = false;
                const int pos = g + j;
#pragma unroll
                for (int t = 0; t < kHalves; ++t) {
                    if (j >= 1 && active(t, j - 1)) issue_pv(t, j - 1);
                    if (t == kHalves - 1 && j >= 1) {
                        const int vp = pos - 1;
                        if (!active(0, j - 1) && !active(1, j - 1))
                            mbar_wait(bar_vfull(vp % VST), (vp / VST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                        __syncwarp();
                        if (leader) umma_commit(bar_vempty(vp % VST));
                    }
                    if (j < w.nblocks && active(t, j)) {
                        const int s = pos % KST;
                        bool good = true;
                        if (!k_ready) {
                            good = mbar_wait(bar_kfull(s), (pos / KST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                            k_ready = true;
                        }
                        if (issued[t] == 0)
                            good = mbar_wait(bar_qfull(t), kw & 1, wc, (kKernPrefill << 8) | kSiteMmaQ) && good;
                        tc_fence_after();
                        __syncwarp();
                        if (leader) {
                            if (good && ok) {
                                const uint64_t qd = qdesc0 + uint64_t((t * C::kQBytes) >> 4);
#pragma unroll
                                for (int kk = 0; kk < HD / 16; ++kk) {
                                    const uint32_t off = uint32_t((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                                    const uint64_t bd = kdesc0 + uint64_t((s * C::kKBytes) >> 4) + off;
                                    umma_bf16(tS(t), qd + off, bd, idesc_qk, kk > 0 ? 1u : 0u);
                                }
                            }
                            umma_commit(bar_sfull(t));
                            if (issued[t] == w.count[t] - 1) umma_commit(bar_qfree(t));  // Q_t read for the last time
                        }
                        ++issued[t];
                    }
                }
                if (j < w.nblocks) {
                    if (!k_ready) mbar_wait(bar_kfull(pos % KST), (pos / KST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                    __syncwarp();
                    if (leader) umma_commit(bar_kempty(pos % KST));
                }
            }
            g += w.nblocks;
            ++kw;
        }
        __syncwarp();
        if (leader) umma_commit(bar_drain);
        mbar_drain(bar_drain, 0, p.timeout_ns);
    } else {
        // ===================== softmax warpgroup of half t
        const int t = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;  // row of the half = TMEM lane
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const bool has_causal = p.causal != 0;
        const bool has_window = p.window_left >= 0;
        const float sl2 = p.scale_log2;
        int kw = 0;
        int s_cnt = 0;    // sfull phases consumed
        int fin_cnt = 0;  // ofinal phases consumed
        for (int k = 0;; ++k) {
            const int slot = k & 1;
            mbar_wait(bar_tfull(slot), (k >> 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxSFull);
            const int4 ti = get_tile(slot);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty(slot));
            if (ti.w < 0) break;
            const TileWork w = tile_work(p, seqs, ti);
            if (!w.work) continue;
            const int b = w.b, ht = w.ht, sk = w.sk;
            const int mt = w.m_block * (128 * kHalves) + 128 * t;
            const int rows_valid = w.rows_h[t];
            const int cnt = w.count[t];
            const int hi_t = w.br.hi - w.first[t];
            const bool row_ok = r < rows_valid;
            const RowMap my = map_row(p, ht, mt + (row_ok ? r : 0));
            const int diag = my.i + sk - p.sq;
            int key_hi = min(sk - 1, has_causal ? diag : sk - 1);
            const int key_lo = has_window ? max(diag - p.window_left, 0) : 0;
            if (!row_ok) key_hi = -1;
            const int i_lo = map_row(p, ht, mt).i;
            const int i_hi = map_row(p, ht, mt + max(rows_valid, 1) - 1).i;
            const int diag_lo = i_lo + sk - p.sq;
            const int diag_hi = i_hi + sk - p.sq;

            float m_run = -INFINITY;
            float l_run = 0.f;
            for (int i = 0; i < cnt; ++i) {
                const int n = hi_t - 1 - i;
                mbar_wait(bar_sfull(t), s_cnt & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxSFull);
                ++s_cnt;
                tc_fence_after();
                const int blk_first = n * 128, blk_last = n * 128 + 127;
                const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                       (has_window && blk_first < diag_hi - p.window_left) || rows_valid < 128;
                const int c_lo = key_lo - blk_first, c_hi = key_hi - blk_first;
                // Two passes over the scores in TMEM, 32 columns at a time, so that
                // a row's 128 scores never sit in registers at once (this warp's
                // state lives across tiles).  Pass 1: the row max.
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[32];
                    tmem_ld16(tS(t) + lane_off + c * 32, x);
                    tmem_ld16(tS(t) + lane_off + c * 32 + 16, x + 16);
                    tmem_wait_ld();
                    if (need_mask) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c * 32 + e < c_lo || c * 32 + e > c_hi) x[e] = -INFINITY;
                    }
                    float ma = mx, mb = -INFINITY;  // two chains, two columns per three-input max
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        ma = fmax3(ma, x[e], x[e + 1]);
                        mb = fmax3(mb, x[e + 2], x[e + 3]);
                    }
                    mx = fmaxf(ma, mb);
                }
                const float cand = mx * sl2;
                bool rescale = false;
                float alpha = 1.f;
                if (cand > m_run + kRescaleThreshold) {
                    alpha = fast_exp2(m_run - cand);
                    rescale = (m_run != -INFINITY);
                    l_run *= alpha;
                    m_run = cand;
                }
                if (i >= 1 && __any_sync(0xffffffffu, rescale)) {
                    const float a = rescale ? alpha : 1.f;
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        float o[16];
                        const uint32_t ta = tO(t) + lane_off + c * 16;
                        tmem_ld16(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] *= a;
                        tmem_st16(ta, o);
                    }
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                // Pass 2: P = 2^(s * x - m) as packed bf16 pairs over the upper half
                // of S_t.  Chunks run from the last one down: chunk c's P lands on
                // the scores of chunks c + 1 .. 3 (already consumed), never on
                // scores still to be read.
#pragma unroll
                for (int c4 = 3; c4 >= 0; --c4) {
                    float x[32];
                    tmem_ld16(tS(t) + lane_off + c4 * 32, x);
                    tmem_ld16(tS(t) + lane_off + c4 * 32 + 16, x + 16);
                    tmem_wait_ld();
                    if (need_mask) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c4 * 32 + e < c_lo || c4 * 32 + e > c_hi) x[e] = -INFINITY;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {  // scale-and-shift and row sums on f32x2 pairs
                        float s0, s1;
                        fma_f32x2(s0, s1, x[2 * e], x[2 * e + 1], sl2, sl2, neg_m, neg_m);
                        const float p0 = fast_exp2(s0);
                        const float p1 = fast_exp2(s1);
                        add_f32x2(ls[2 * (e & 1)], ls[2 * (e & 1) + 1], p0, p1);
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16u(tS(t) + C::kPCol + lane_off + c4 * 16, pk);
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pfull(t));
            }

            // ---- epilogue: O / l straight from TMEM to global memory
            if (cnt >= 1) {
                mbar_wait(bar_ofinal(t), fin_cnt & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
                ++fin_cnt;
                tc_fence_after();
            }
            const float inv = (cnt >= 1 && l_run > 0.f) ? 1.f / l_run : 0.f;
            const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            const bool final_out = (w.sb == 1);
            const size_t orow = final_out ? ((size_t(b) * p.sq + my.i) * p.Hq + my.h)
                                          : (((size_t(w.split) * p.B + b) * p.Hq + my.h) * p.sq + my.i);
#pragma unroll
            for (int c = 0; c < HD / 16; ++c) {
                float o[16];
                if (cnt >= 1) {
                    tmem_ld16(tO(t) + lane_off + c * 16, o);  // warp-collective: every lane takes part
                    tmem_wait_ld();
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = cnt >= 1 ? o[e] * inv : 0.f;
                if (row_ok) {
                    if (final_out) {
                        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * HD + c * 16);
                        dst[0] = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                            pack_bf16x2(o[6], o[7]));
                        dst[1] = make_uint4(pack_bf16x2(o[8], o[9]), pack_bf16x2(o[10], o[11]),
                                            pack_bf16x2(o[12], o[13]), pack_bf16x2(o[14], o[15]));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.o_part + orow * HD + c * 16);
                        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
                        dst[2] = make_float4(o[8], o[9], o[10], o[11]);
                        dst[3] = make_float4(o[12], o[13], o[14], o[15]);
                    }
                }
            }
            if (row_ok) {
                if (final_out)
                    p.lse[(size_t(b) * p.Hq + my.h) * p.sq + my.i] = lse;
                else
                    p.lse_part[orow] = lse;
            }
            tc_fence_before();
            ++kw;
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int HD, class Seqs>
cudaError_t launch_one(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmQ, const Seqs& seqs, cudaStream_t stream) {
    using C = PersistCfg<HD>;
    auto kern = fwd_prefill_persistent_kernel<HD, Seqs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    TileList tl;
    tl.nm = plan.num_m_blocks;
    tl.S = plan.num_splits;
    tl.head_tiles = plan.head_tiles;
    tl.B = plan.B;
    tl.ntiles = int(plan.num_ctas);
    tl.sec = plan.l2_section;
    tl.masked = plan.reverse_m ? 1 : 0;
    dim3 grid(plan.persistent_ctas);
    return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), C::kSmemAlloc, stream, p, tmK, tmV,
                      tmQ, seqs, tl);
}

}  // namespace

cudaError_t launch_prefill_persistent(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, const CUtensorMap& tmQ, cudaStream_t stream) {
    if (plan.kBlockM != 128 * kHalves || plan.kBlockN != 128 || !p.q_tma) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        if (plan.d == 128) return launch_one<128, UniformSeqs>(plan, p, tmK, tmV, tmQ, u, stream);
        return launch_one<64, UniformSeqs>(plan, p, tmK, tmV, tmQ, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    if (plan.d == 128) return launch_one<128, VarlenSeqs>(plan, p, tmK, tmV, tmQ, v, stream);
    return launch_one<64, VarlenSeqs>(plan, p, tmK, tmV, tmQ, v, stream);
}

}  // namespace sk
