// fwd_prefill.cu -- split-KV partial kernel for 256-row query tiles (prefill,
// large packed GQA groups), sm_103a.
//
// One CTA owns (m block, head tile, split, sequence): 256 query rows (packed
// rows with PackGQA, tiling chapter section 6) against the KV blocks of its
// range (section 3.2 causal / local skipping, section 5.3 split share).  The
// tile is two 128-row halves t = 0, 1 that share every K/V block in shared
// memory:
//   S_t[128 x 128] = Q_t[128 x d] . K_blk^T       (tcgen05 SS, S_t in TMEM)
//   O_t[128 x d]  += P_t[128 x 128] . V_blk[128 x d] (tcgen05 TS, P_t in TMEM)
// The halves ping-pong: while one softmax warpgroup turns S_0 into P_0, the
// tensor pipe runs the other half's PV and QK^T, so neither the exp2 work nor
// the tensor pipe waits on the other.  Each softmax thread owns one query row
// (TMEM lane) of its half: running max and sum in registers, the fp32
// accumulator in TMEM, rescaled in place only when the row max grows by more
// than 2^8 (P stays <= 256 meanwhile).
//
// Blocks are visited from the last one of the range down, so causal and local
// tiles meet their masked diagonal blocks first; a half whose own range is
// shorter (under a causal mask half 0, the tile's first 128 query rows, sees
// one block fewer than half 1) skips the steps outside it.
//
// Q halves arrive by TMA (a 4-D map whose 128-row box is in packed-row order)
// unless a half is not whole row groups of that map; then the softmax warps
// load them.
//
// Warp roles (320 threads): warp 0 TMA producer (Q, K/V rings), warp 1 TMEM
// owner and MMA issuer (both run whole, warp-uniform; one elected lane issues
// the copies / MMAs), warps 2-5 softmax + correction + epilogue of half 0,
// warps 6-9 the same for half 1.
#include <math.h>

#include "fwd_common.cuh"
#include "kv_producer.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kHalves = 2;
constexpr int kThreads = 64 + 128 * kHalves;  // producer warp, MMA warp, softmax warpgroups
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
struct PrefillCfg {
    static constexpr int kStagesK = HD == 128 ? 3 : 4;
    static constexpr int kStagesV = HD == 128 ? 2 : 4;
    static constexpr int kKBytes = 128 * HD * 2;
    static constexpr int kVBytes = 128 * HD * 2;
    static constexpr int kQBytes = 128 * HD * 2;                  // one half
    static constexpr int kOffQ = 0;                               // Q_0, Q_1
    static constexpr int kOffK = kOffQ + kHalves * kQBytes;       // K ring: kStagesK slots
    static constexpr int kOffV = kOffK + kStagesK * kKBytes;      // V ring: kStagesV slots
    static constexpr int kOffBars = kOffV + kStagesV * kVBytes;
    static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 4 * kHalves + 2;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16;
    // 1024 bytes of slack let the kernel align the operand base itself; when the
    // budget has no room for it the kernel instead checks that the dynamic
    // shared-memory base is already 1024-byte aligned.
    static constexpr int kSlack = (kSmemBytes + 1024 <= 232448) ? 1024 : 0;
    static constexpr int kSmemAlloc = kSmemBytes + kSlack;
    // TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256, 256+HD), O_1 [384, 384+HD).
    // P_t (128 keys as 64 columns of packed bf16 pairs) overwrites the upper
    // half of S_t once the softmax has read it.
    static constexpr int kTmemCols = 512;
    static constexpr int kPCol = 64;
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

template <int HD, class Seqs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_prefill_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmO, const __grid_constant__ Seqs seqs) {
    using C = PrefillCfg<HD>;
    constexpr int KST = C::kStagesK;
    constexpr int VST = C::kStagesV;
    constexpr int NB0 = 2 * KST + 2 * VST;  // first barrier after the rings
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (C::kSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
        // No room to realign: report and leave before touching shared memory.
        if (threadIdx.x == 0) atomicCAS(p.status, 0u, (kKernPrefill << 8) | kSiteSmemAlign);
        return;
    }
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const TileCoord tc = tile_of_cta(blockIdx.x, blockIdx.y, blockIdx.z, p.num_m_blocks, p.num_splits,
                                     p.reverse_m != 0);
    const int b = tc.batch;
    const int ht = tc.head_tile;
    const int sb = seqs.splits_of(b);
    const uint32_t word = split_word(tc.split, sb);
    const long long cta_lin =
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    if (tc.split >= sb) {
        griddep_launch_dependents();
        griddep_wait();
        if (p.echo_plan && threadIdx.x == 0)
            *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(0, 0, int(word), 0);
        return;
    }
    const int m0 = tc.m_block * (128 * kHalves);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t bars = sbase + C::kOffBars;
    // barriers: kfull[KST] kempty[KST] vfull[VST] vempty[VST] qfull[2] sfull[2] pfull[2] ofinal[2] never drain
    auto bar_kfull = [&](int s) { return bars + 8u * s; };
    auto bar_kempty = [&](int s) { return bars + 8u * (KST + s); };
    auto bar_vfull = [&](int s) { return bars + 8u * (2 * KST + s); };
    auto bar_vempty = [&](int s) { return bars + 8u * (2 * KST + VST + s); };
    auto bar_qfull = [&](int t) { return bars + 8u * (NB0 + t); };
    auto bar_sfull = [&](int t) { return bars + 8u * (NB0 + kHalves + t); };
    auto bar_pfull = [&](int t) { return bars + 8u * (NB0 + 2 * kHalves + t); };
    auto bar_ofinal = [&](int t) { return bars + 8u * (NB0 + 3 * kHalves + t); };
    const uint32_t bar_never = bars + 8u * (NB0 + 4 * kHalves);
    const uint32_t bar_drain = bars + 8u * (NB0 + 4 * kHalves + 1);
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
            mbar_init(bar_qfull(t), p.q_tma ? 1 : 128);  // TMA transaction, or every thread of the half
            mbar_init(bar_sfull(t), 1);
            mbar_init(bar_pfull(t), 4);  // one arrival per softmax warp
            mbar_init(bar_ofinal(t), 1);
        }
        mbar_init(bar_never, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.q_tma) {
            // The tile's Q halves go out first, before the block ranges below are
            // worked out.  Q may be the previous kernel's output: wait for it.
            griddep_wait();
#pragma unroll
            for (int t = 0; t < kHalves; ++t) {
                mbar_arrive_expect_tx(bar_qfull(t), C::kQBytes);
                const int qrow = b * p.sq + (m0 + 128 * t) / p.q_gp;
#pragma unroll
                for (int c = 0; c < HD / 64; ++c)
                    tma_load_4d(sQ + uint32_t(t * C::kQBytes + c * 16384), &tmQ, bar_qfull(t), c * 64, 0, ht, qrow,
                                l2_policy_evict_first());
            }
        }
    }
    const int sk = seqs.seq_len(b);
    const int kv_off = seqs.seq_off(b);
    const BlockRange br =
        tile_key_blocks(p.sq, sk, tc.m_block, 128 * kHalves, 128, p.win, p.pack_gqa ? p.G : 1, word);
    const int nblocks = br.hi > br.lo ? br.hi - br.lo : 0;
    const int kvh = p.pack_gqa ? ht : ht / p.G;
    // The first K block (the last of the range: blocks are visited downwards)
    // follows the Q halves at once, into slot 0 of the K ring (free at start).
    const bool k0_early = p.q_tma && nblocks > 0;
    if (threadIdx.x == 0 && k0_early) {
        mbar_arrive_expect_tx(bar_kfull(0), C::kKBytes);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
            tma_load_2d(stage_k(0) + c * 16384, &tmK, bar_kfull(0), kvh * HD + c * 64, kv_off + (br.hi - 1) * 128,
                        l2_policy_evict_last());
    }

    // Each half's own block range (section 3.2 applied to its 128 rows), clipped
    // to the CTA's split share.  Visiting step j (block br.hi - 1 - j) belongs to
    // half t for j in [first[t], first[t] + count[t]).
    int first[kHalves], count[kHalves], rows_h[kHalves];
#pragma unroll
    for (int t = 0; t < kHalves; ++t) {
        rows_h[t] = max(0, min(128, p.rows - (m0 + 128 * t)));
        const BlockRange hr = tile_key_blocks(p.sq, sk, tc.m_block * kHalves + t, 128, 128, p.win,
                                              p.pack_gqa ? p.G : 1, split_word(0, 1));
        const int lo = max(hr.lo, br.lo), hi = min(hr.hi, br.hi);
        count[t] = (rows_h[t] > 0 && hi > lo) ? hi - lo : 0;
        first[t] = count[t] > 0 ? br.hi - hi : 0;
    }

    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (p.q_tma) tma_prefetch_desc(&tmQ);
        if (p.o_tma) tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Everything above touched only shared memory, TMEM and kernel parameters.
    // Under programmatic dependent launch this grid may start while the previous
    // kernel on the stream is still running: wait for it before any global access.
    griddep_wait();
    if (p.echo_plan && threadIdx.x == 0)
        *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(br.lo, br.hi, int(word), 1);
    const uint32_t tmem = *tmem_holder;
    auto tS = [&](int t) { return tmem + uint32_t(t) * 128u; };
    auto tO = [&](int t) { return tmem + 256u + uint32_t(t) * 128u; };
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ===================== producer: the K/V rings (thread 0 issued the Q halves)
        const bool leader = elect_one();
        // K/V of one head are re-read by the other m blocks: keep them in L2.
        const KvRing kr{stage_k(0), uint32_t(C::kKBytes), bar_kfull(0), bar_kempty(0), KST};
        const KvRing vr{stage_v(0), uint32_t(C::kVBytes), bar_vfull(0), bar_vempty(0), VST};
        int kpos = 0, vpos = 0;
        produce_kv_tile<HD>(&tmK, &tmV, kr, vr, 0, nblocks, kvh * HD, kv_off + br.lo * 128, true,
                            l2_policy_evict_last(), wc, (kKernPrefill << 8) | kSiteProducerEmpty, leader, kpos, vpos,
                            k0_early);
        drain_ring(kr, kpos, wc.limit_ns);
        drain_ring(vr, vpos, wc.limit_ns);
        // Q copies land before the CTA exits (the MMA waited for them unless it gave up).
        if (p.q_tma)
            for (int t = 0; t < kHalves; ++t) mbar_drain(bar_qfull(t), 0, wc.limit_ns);
    } else if (warp == 1) {
        // The whole warp runs the MMA schedule (warp-uniform control flow, so
        // descriptors and loop state stay warp-uniform); one elected lane issues
        // every tcgen05 op, and tcgen05.commit tracks that lane's MMAs.
        const bool leader = elect_one();
        constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_pv = make_idesc_bf16(128, HD, false, true);
        // Descriptors are built once; per MMA only a constant is added to the
        // start-address field (all operands lie below 256 KB, so the field
        // never carries).
        const uint64_t qdesc0 = make_sdesc_sw128(sQ, 16, 1024);
        const uint64_t kdesc0 = make_sdesc_sw128(stage_k(0), 16, 1024);
        const uint64_t vdesc0 = make_sdesc_sw128(stage_v(0), 16384, 1024);
        bool ok = true;
        if (p.inject_stall) {
            // The injected stall gives up first (half the limit), so the status
            // names it rather than a wait that starves behind it.
            const WaitCtl wc_half{wc.abort_flag, wc.status, wc.limit_ns / 2};
            ok = mbar_wait(bar_never, 0, wc_half, (kKernPrefill << 8) | kSiteInjected);
        }
        auto active = [&](int t, int j) { return j >= first[t] && j < first[t] + count[t]; };
        int zeroed_step = -1;  // visiting step whose V tail rows were zeroed
        // O_t += P_t . V(j), the i-th block of half t.  P_t sits in the upper
        // columns of S_t; the QK^T that next overwrites S_t is issued after
        // this MMA, and the tensor pipe runs a CTA's MMAs in issue order.
        auto issue_pv = [&](int t, int j) {
            const int i = j - first[t];
            const int s = j % VST;
            bool good = mbar_wait(bar_pfull(t), i & 1, wc, (kKernPrefill << 8) | kSiteMmaPFull);
            good = mbar_wait(bar_vfull(s), (j / VST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull) && good;
            // The block that holds the end of the sequence also holds rows of
            // the next sequence: their P is 0, but 0 * (Inf or NaN) is NaN, so
            // those V rows are zeroed before the first PV MMA reads the slot.
            const int tail_row = sk - (br.hi - 1 - j) * 128;
            if (good && tail_row < 128 && zeroed_step != j) zero_rows<HD>(stage_v(s), tail_row, lane);
            zeroed_step = j;
            tc_fence_after();
            __syncwarp();
            if (leader) {
                if (good && ok) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // A = P from TMEM: 16 keys = 8 packed columns per MMA.
                        const uint64_t bd = vdesc0 + uint64_t((s * C::kVBytes + kk * 2048) >> 4);
                        umma_bf16_ts(tO(t), tS(t) + C::kPCol + kk * 8, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                if (i == count[t] - 1) umma_commit(bar_ofinal(t));
            }
        };
        int issued[kHalves] = {0, 0};
        for (int j = 0; j <= nblocks; ++j) {
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < kHalves; ++t) {
                // PV of the previous block first: it frees P_t (= S_t) for the next QK^T.
                if (j >= 1 && active(t, j - 1)) issue_pv(t, j - 1);
                if (t == kHalves - 1 && j >= 1) {
                    // V(j-1) has no reader left.  A block that no half read is
                    // still waited for, so no load is outstanding on a freed slot.
                    if (!active(0, j - 1) && !active(1, j - 1))
                        mbar_wait(bar_vfull((j - 1) % VST), ((j - 1) / VST) & 1, wc,
                                  (kKernPrefill << 8) | kSiteMmaFull);
                    __syncwarp();
                    if (leader) umma_commit(bar_vempty((j - 1) % VST));
                }
                if (j < nblocks && active(t, j)) {
                    const int s = j % KST;
                    bool good = true;
                    if (!k_ready) {
                        good = mbar_wait(bar_kfull(s), (j / KST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                        k_ready = true;
                    }
                    if (issued[t] == 0)
                        good = mbar_wait(bar_qfull(t), 0, wc, (kKernPrefill << 8) | kSiteMmaQ) && good;
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
                    }
                    ++issued[t];
                }
            }
            if (j < nblocks) {
                if (!k_ready) mbar_wait(bar_kfull(j % KST), (j / KST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                __syncwarp();
                if (leader) umma_commit(bar_kempty(j % KST));
            }
        }
        __syncwarp();
        if (leader) umma_commit(bar_drain);
        mbar_drain(bar_drain, 0, p.timeout_ns);
    } else {
        // Softmax warpgroup of half t: warp w owns TMEM lanes 32 * (w % 4) ...
        const int t = (warp - 2) >> 2;
        const int sidx = threadIdx.x - 64 - 128 * t;        // 0 .. 127
        const int r = 32 * (warp & 3) + lane;               // row of the half = TMEM lane
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const int mt = m0 + 128 * t;                        // first packed row of the half
        const int rows_valid = rows_h[t];
        const int cnt = count[t];
        const int hi_t = br.hi - first[t];                  // half's blocks: hi_t - 1 down to hi_t - cnt
        const uint32_t sQt = sQ + uint32_t(t * C::kQBytes);

        // Q half -> smem when it does not come by TMA: K-major 128B swizzle
        // (granule g of row rr at sw128_offset); loads are issued before any store.
        if (!p.q_tma) {
            constexpr int kGran = HD / 8;
            uint4 val[kGran];
#pragma unroll
            for (int u = 0; u < kGran; ++u) {
                const int idx = sidx + u * 128;
                const int rr = idx / kGran;
                const int g16 = idx - rr * kGran;
                val[u] = make_uint4(0, 0, 0, 0);
                if (rr < rows_valid) {
                    const RowMap rm = map_row(p, ht, mt + rr);
                    val[u] = __ldg(reinterpret_cast<const uint4*>(
                        p.q + ((size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * HD + g16 * 8));
                }
            }
#pragma unroll
            for (int u = 0; u < kGran; ++u) {
                const int idx = sidx + u * 128;
                const int rr = idx / kGran;
                const int g16 = idx - rr * kGran;
                const uint32_t dst = sQt + (g16 >> 3) * 16384 + sw128_offset(rr, g16 & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(val[u].x), "r"(val[u].y),
                             "r"(val[u].z), "r"(val[u].w)
                             : "memory");
            }
        }
        if (!p.q_tma) {
            fence_proxy_async_smem();
            mbar_arrive(bar_qfull(t));
        }

        const bool row_ok = r < rows_valid;
        const RowMap my = map_row(p, ht, mt + (row_ok ? r : 0));
        const int diag = my.i + sk - p.sq;
        // Keys this row sees: [key_lo, key_hi] (empty for a padding row).
        int key_hi = min(sk - 1, p.causal ? diag : sk - 1);
        const int key_lo = p.window_left >= 0 ? max(diag - p.window_left, 0) : 0;
        if (!row_ok) key_hi = -1;
        // the half's diagonal range (rows are ordered by query position)
        const int i_lo = map_row(p, ht, mt).i;
        const int i_hi = map_row(p, ht, mt + max(rows_valid, 1) - 1).i;
        const int diag_lo = i_lo + sk - p.sq;
        const int diag_hi = i_hi + sk - p.sq;
        const bool has_causal = p.causal != 0;
        const bool has_window = p.window_left >= 0;
        const float sl2 = p.scale_log2;

        float m_run = -INFINITY;  // running row max, log2 units (scaled)
        float l_run = 0.f;        // running row sum
        for (int i = 0; i < cnt; ++i) {
            const int n = hi_t - 1 - i;
            float x[128];
            mbar_wait(bar_sfull(t), i & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxSFull);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_ld16(tS(t) + lane_off + c * 16, x + c * 16);
            tmem_wait_ld();

            const int blk_first = n * 128, blk_last = n * 128 + 127;
            const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                   (has_window && blk_first < diag_hi - p.window_left) || rows_valid < 128;
            if (need_mask) {
                // A diagonal block cuts its rows above (c_hi), a block at the
                // window's left edge below (c_lo); the warp takes the one-sided
                // test unless one of its rows needs both.
                const int c_lo = key_lo - blk_first, c_hi = key_hi - blk_first;
                const bool cut_hi = __any_sync(0xffffffffu, c_hi < 127);
                const bool cut_lo = __any_sync(0xffffffffu, c_lo > 0);
                if (cut_hi && cut_lo) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c < c_lo || c > c_hi) x[c] = -INFINITY;
                } else if (cut_hi) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > c_hi) x[c] = -INFINITY;
                } else if (cut_lo) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c < c_lo) x[c] = -INFINITY;
                }
            }
            // Row max: 8 chains of 16 columns, two columns per three-input max.
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float m = fmax3(x[k], x[k + 8], x[k + 16]);
#pragma unroll
                for (int c = 24; c < 120; c += 16) m = fmax3(m, x[k + c], x[k + c + 8]);
                mx8[k] = fmaxf(m, x[k + 120]);
            }
            const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                   fmaxf(mx8[6], mx8[7]));
            const float cand = mx * sl2;
            bool rescale = false;
            float alpha = 1.f;
            if (cand > m_run + kRescaleThreshold) {
                alpha = fast_exp2(m_run - cand);  // 0 when m_run = -inf
                rescale = (m_run != -INFINITY);
                l_run *= alpha;
                m_run = cand;
            }
            // O_t holds blocks 0 .. i-1: their PV completed before the QK^T whose
            // completion signalled sfull.  tcgen05.ld/st are warp-collective
            // (.sync.aligned): the whole warp enters; rows that keep their max x 1.
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
            // P row -> TMEM (upper half of S_t): 64 columns of packed bf16 pairs.
            // Scale-and-shift and the row sum run on column pairs (f32x2).
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float s0, s1;
                    fma_f32x2(s0, s1, x[c4 * 32 + 2 * e], x[c4 * 32 + 2 * e + 1], sl2, sl2, neg_m, neg_m);
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

        // Let the dependent grid (the combine, or the next call's partial kernel)
        // get scheduled; it waits for this grid's completion before reading.
        griddep_launch_dependents();
        // ---- epilogue: O / l for this row
        if (cnt >= 1) {
            mbar_wait(bar_ofinal(t), 0, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
            tc_fence_after();
        }
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        const bool final_out = (sb == 1);
        // Final rows go out through the O map: staged as bf16 in Q_t's buffer (the
        // half's last QK^T, complete once ofinal fired, was its last reader; a
        // half with no block waits for its Q copy first) and stored by one TMA
        // copy per 64 columns, coalesced, clipped at the end of the sequence.
        const bool stage = final_out && p.o_tma;
        if (stage && cnt == 0 && p.q_tma) {
            mbar_wait(bar_qfull(t), 0, wc, (kKernPrefill << 8) | kSiteMmaQ);
        }
        // O row read from TMEM 64 columns per wait, then scaled and written 16 at a time.
        float o64[64];
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
            float* o = o64 + 16 * (c & 3);
            if ((c & 3) == 0 && cnt >= 1) {
#pragma unroll
                for (int u = 0; u < 4; ++u) tmem_ld16(tO(t) + lane_off + (c + u) * 16, o64 + 16 * u);
                tmem_wait_ld();
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = (cnt >= 1 && l_run > 0.f) ? o[e] * inv : 0.f;
            const int dcol = c * 16;
            if (stage) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(o[2 * e], o[2 * e + 1]);
                const uint32_t dst = sQt + (c >> 2) * 16384;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + sw128_offset(r, (2 * c) & 7)),
                             "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + sw128_offset(r, (2 * c + 1) & 7)),
                             "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                             : "memory");
            } else if (row_ok) {
                if (final_out) {
                    __nv_bfloat16* dst = p.out + ((size_t(b) * p.sq + my.i) * p.Hq + my.h) * HD + dcol;
                    uint4 w0, w1;
                    w0.x = pack_bf16x2(o[0], o[1]); w0.y = pack_bf16x2(o[2], o[3]);
                    w0.z = pack_bf16x2(o[4], o[5]); w0.w = pack_bf16x2(o[6], o[7]);
                    w1.x = pack_bf16x2(o[8], o[9]); w1.y = pack_bf16x2(o[10], o[11]);
                    w1.z = pack_bf16x2(o[12], o[13]); w1.w = pack_bf16x2(o[14], o[15]);
                    reinterpret_cast<uint4*>(dst)[0] = w0;
                    reinterpret_cast<uint4*>(dst)[1] = w1;
                } else {
                    const size_t prow = ((size_t(tc.split) * p.B + b) * p.Hq + my.h) * p.sq + my.i;
                    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * HD + dcol);
                    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
                    dst[2] = make_float4(o[8], o[9], o[10], o[11]);
                    dst[3] = make_float4(o[12], o[13], o[14], o[15]);
                }
            }
            if (stage && (c & 3) == 3) {
                // 64 columns of the half's rows are staged: their TMA store goes
                // out while the next 64 are written.
                fence_proxy_async_smem();
                named_bar_sync(2 + t, 128);  // the half's 128 threads
                if (sidx == 0)
                    tma_store_5d(&tmO, sQt + uint32_t((c >> 2) * 16384), (c >> 2) * 64, 0, ht,
                                 (m0 + 128 * t) / p.q_gp, b);
            }
        }
        if (stage && sidx == 0) {
            bulk_commit_group();
            bulk_wait_group_read0();  // the source stays valid until the copies have read it
        }
        if (row_ok) {
            if (final_out)
                p.lse[(size_t(b) * p.Hq + my.h) * p.sq + my.i] = lse;
            else
                p.lse_part[((size_t(tc.split) * p.B + b) * p.Hq + my.h) * p.sq + my.i] = lse;
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
                       const CUtensorMap& tmQ, const CUtensorMap& tmO, const Seqs& seqs, cudaStream_t stream) {
    using C = PrefillCfg<HD>;
    auto kern = fwd_prefill_kernel<HD, Seqs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), C::kSmemAlloc, stream, p, tmK, tmV,
                      tmQ, tmO, seqs);
}

}  // namespace

cudaError_t launch_prefill(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmQ, const CUtensorMap& tmO, cudaStream_t stream) {
    if (plan.kBlockM != 128 * kHalves || plan.kBlockN != 128) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        if (plan.d == 128) return launch_one<128, UniformSeqs>(plan, p, tmK, tmV, tmQ, tmO, u, stream);
        return launch_one<64, UniformSeqs>(plan, p, tmK, tmV, tmQ, tmO, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    if (plan.d == 128) return launch_one<128, VarlenSeqs>(plan, p, tmK, tmV, tmQ, tmO, v, stream);
    return launch_one<64, VarlenSeqs>(plan, p, tmK, tmV, tmQ, tmO, v, stream);
}

}  // namespace sk
