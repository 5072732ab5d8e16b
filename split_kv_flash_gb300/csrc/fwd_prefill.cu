// fwd_prefill.cu -- split-KV partial kernel for 128-row query tiles (prefill,
// large packed GQA groups), sm_103a.
//
// One CTA owns (m block, head tile, split, sequence): 128 query rows (packed
// rows with PackGQA, tiling chapter section 6) against the KV blocks of its
// range (section 3.2 causal / local skipping, section 5.3 split share).
//   S[128 x 128] = Q_tile[128 x d] . K_blk^T        (tcgen05, S in TMEM, 2 buffers)
//   O[128 x d]  += P[128 x 128] . V_blk[128 x d]    (tcgen05, O in TMEM)
// Each softmax thread owns one query row (TMEM lane): its running max and sum
// live in registers, the fp32 accumulator lives in TMEM and is rescaled in place
// only when the row max grows by more than 2^8 (P stays <= 256 meanwhile).
//
// Warp roles (192 threads): warp 0 TMA producer (K/V ring), warp 1 TMEM owner
// and MMA issuer, warps 2-5 softmax + correction + epilogue.
#include <math.h>

#include "fwd_common.cuh"
#include "kv_producer.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

// The 128 key columns of every row are split over kGroups softmax warpgroups
// (warps w and w + 4 share TMEM lane quadrant w % 4): more warps per scheduler
// hide the latency of the TMEM loads, the exp2 and the barriers.
#ifndef SK_PREFILL_COLGROUPS
#define SK_PREFILL_COLGROUPS 2
#endif
constexpr int kGroups = SK_PREFILL_COLGROUPS;
constexpr int kSoftmaxThreads = 128 * kGroups;
constexpr int kThreads = 64 + kSoftmaxThreads;  // producer warp, MMA warp, softmax warps
constexpr int kCW = 128 / kGroups;              // S / P columns (keys) per thread
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
struct PrefillCfg {
    // P lives in TMEM (A operand of the PV MMA), which leaves room for a third K slot.
    static constexpr int kStagesK = HD == 128 ? 3 : 4;
    static constexpr int kStagesV = HD == 128 ? (kGroups > 2 ? 2 : 3) : 4;
    static constexpr int kKBytes = 128 * HD * 2;
    static constexpr int kVBytes = 128 * HD * 2;
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kQBytes = 128 * HD * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;              // K ring: kStagesK slots
    static constexpr int kOffV = kOffK + kStagesK * kKBytes;   // V ring: kStagesV slots
    static constexpr int kOffXchg = kOffV + kStagesV * kVBytes;  // float [2 slots][kGroups][128 rows]
    static constexpr int kOffBars = kOffXchg + 2 * kGroups * 128 * 4;
    static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 2 + 1 + 1 + 1;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16;
    // 1024 bytes of slack let the kernel align the operand base itself; when the
    // budget has no room for it the kernel instead checks that the dynamic
    // shared-memory base is already 1024-byte aligned.
    static constexpr int kSlack = (kSmemBytes + 1024 <= 232448) ? 1024 : 0;
    static constexpr int kSmemAlloc = kSmemBytes + kSlack;
    // TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+HD), P0 [384,448), P1 [448,512)
    // (P: 128 keys as 64 columns of packed bf16 pairs).
    static constexpr int kTmemCols = 512;
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// PAIR: the CTA is one of a 2-CTA cluster (two query heads of one KV head with
// identical block ranges) that share every K/V block through TMA multicast.
template <int HD, class Seqs, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_prefill_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Seqs seqs) {
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
    const int sk = seqs.seq_len(b);
    const int kv_off = seqs.seq_off(b);
    const BlockRange br =
        n_block_range(p.sq, sk, tc.m_block, p.kBlockM, p.kBlockN, p.flags, p.pack_gqa != 0, p.G, word);
    const int nblocks = br.hi > br.lo ? br.hi - br.lo : 0;
    const int kvh = p.pack_gqa ? ht : ht / p.G;
    // per-CTA starting block (spreads the CTAs of one KV head over its K/V; equal
    // within a cluster pair, which shares the loads)
    uint32_t hsh = uint32_t(tc.m_block) * 0x9E3779B1u + uint32_t(kvh) * 0x85EBCA77u + uint32_t(b) * 0xC2B2AE3Du;
    hsh ^= hsh >> 15;
    hsh *= 0x2C1B3C6Du;
    hsh ^= hsh >> 12;
    const int rot = nblocks > 0 ? int(hsh % uint32_t(nblocks)) : 0;
    const int m0 = tc.m_block * 128;
    const int rows_valid = min(128, p.rows - m0);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t bars = sbase + C::kOffBars;
    // barriers: kfull[KST] kempty[KST] vfull[VST] vempty[VST] sfull[2] sempty[2] pfull[2] odone[2] q never drain
    auto bar_kfull = [&](int s) { return bars + 8u * s; };
    auto bar_kempty = [&](int s) { return bars + 8u * (KST + s); };
    auto bar_vfull = [&](int s) { return bars + 8u * (2 * KST + s); };
    auto bar_vempty = [&](int s) { return bars + 8u * (2 * KST + VST + s); };
    auto bar_sfull = [&](int i) { return bars + 8u * (NB0 + i); };
    auto bar_sempty = [&](int i) { return bars + 8u * (NB0 + 2 + i); };
    auto bar_pfull = [&](int i) { return bars + 8u * (NB0 + 4 + i); };
    auto bar_odone = [&](int i) { return bars + 8u * (NB0 + 6 + i); };
    const uint32_t bar_qfull = bars + 8u * (NB0 + 8);
    const uint32_t bar_never = bars + 8u * (NB0 + 9);
    const uint32_t bar_drain = bars + 8u * (NB0 + 10);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    auto stage_k = [&](int s) { return sbase + C::kOffK + uint32_t(s) * C::kKBytes; };
    auto stage_v = [&](int s) { return sbase + C::kOffV + uint32_t(s) * C::kVBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), PAIR ? 2 : 1);  // a paired slot is released by both CTAs
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(bar_vfull(s), 1);
            mbar_init(bar_vempty(s), PAIR ? 2 : 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull(i), 1);
            mbar_init(bar_sempty(i), kSoftmaxThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_pfull(i), kSoftmaxThreads);
            mbar_init(bar_odone(i), 1);
        }
        mbar_init(bar_qfull, kSoftmaxThreads);
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
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the partner's barriers are initialised before any multicast
    tc_fence_after();
    // Everything above touched only shared memory, TMEM and kernel parameters.
    // Under programmatic dependent launch this grid may start while the previous
    // kernel on the stream is still running: wait for it before any global access.
    griddep_wait();
    if (p.echo_plan && threadIdx.x == 0)
        *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(br.lo, br.hi, int(word), 1);
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS0 = tmem;        // columns [0,128) and [128,256)
    const uint32_t tO = tmem + 256;   // columns [256, 256 + HD)
    const uint32_t tP0 = tmem + 384;  // P buffers: columns [384, 448) and [448, 512)
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // K/V of one head are re-read by the other m blocks: keep them in L2.
            const KvRing kr{stage_k(0), uint32_t(C::kKBytes), bar_kfull(0), bar_kempty(0), KST};
            const KvRing vr{stage_v(0), uint32_t(C::kVBytes), bar_vfull(0), bar_vempty(0), VST};
            if constexpr (PAIR)
                produce_kv_pair<HD>(&tmK, &tmV, kr, vr, nblocks, kvh * HD, kv_off + br.lo * 128, rot,
                                    cluster_ctarank(), l2_policy_evict_last(), wc,
                                    (kKernPrefill << 8) | kSiteProducerEmpty);
            else
                produce_kv<HD>(&tmK, &tmV, kr, vr, nblocks, kvh * HD, kv_off + br.lo * 128, rot,
                               l2_policy_evict_last(), wc, (kKernPrefill << 8) | kSiteProducerEmpty);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = make_idesc_bf16(128, HD, false, true);
            // Descriptors are built once; per MMA only a constant is added to the
            // start-address field (all operands lie below 256 KB, so the field
            // never carries).  This keeps the single issuing thread ahead of the
            // tensor pipe.
            const uint64_t qdesc0 = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t kdesc0 = make_sdesc_sw128(stage_k(0), 16, 1024);
            const uint64_t vdesc0 = make_sdesc_sw128(stage_v(0), 16384, 1024);
            bool ok = true;
            if (p.inject_stall) ok = mbar_wait(bar_never, 0, wc, (kKernPrefill << 8) | kSiteInjected);
            if (nblocks > 0) ok = mbar_wait(bar_qfull, 0, wc, (kKernPrefill << 8) | kSiteMmaQ) && ok;
            auto issue_pv = [&](int jj) {
                const int s = jj % VST;
                bool good = mbar_wait(bar_pfull(jj & 1), (jj >> 1) & 1, wc, (kKernPrefill << 8) | kSiteMmaPFull);
                good = mbar_wait(bar_vfull(s), (jj / VST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull) && good;
                tc_fence_after();
                if (good) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // A = P from TMEM: 16 keys = 8 packed columns per MMA.
                        const uint64_t bd = vdesc0 + uint64_t((s * C::kVBytes + kk * 2048) >> 4);
                        umma_bf16_ts(tO, tP0 + (jj & 1) * 64 + kk * 8, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar_odone(jj & 1));
                    if constexpr (PAIR)
                        umma_commit_mc(bar_vempty(s), uint16_t(0x3));
                    else
                        umma_commit(bar_vempty(s));
                }
            };
            for (int j = 0; j < nblocks; ++j) {
                const int s = j % KST;
                bool good = mbar_wait(bar_kfull(s), (j / KST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                if (j >= 2)
                    good = mbar_wait(bar_sempty(j & 1), ((j >> 1) - 1) & 1, wc,
                                     (kKernPrefill << 8) | kSiteMmaSEmpty) && good;
                tc_fence_after();
                if (good && ok) {
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = uint32_t((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        const uint64_t a = qdesc0 + off;
                        const uint64_t bd = kdesc0 + uint64_t((s * C::kKBytes) >> 4) + off;
                        umma_bf16(tS0 + (j & 1) * 128, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar_sfull(j & 1));
                    if constexpr (PAIR)
                        umma_commit_mc(bar_kempty(s), uint16_t(0x3));
                    else
                        umma_commit(bar_kempty(s));
                }
                if (j >= 1) issue_pv(j - 1);
            }
            if (nblocks >= 1) issue_pv(nblocks - 1);
            umma_commit(bar_drain);
            mbar_drain(bar_drain, 0, p.timeout_ns);
        }
    } else {
        // Softmax warps 2..(2 + 4 * kGroups): group g owns key columns
        // [g * kCW, (g + 1) * kCW) of every row and O columns [g * HD / kGroups, ...).
        const int sidx = threadIdx.x - 64;                 // 0 .. kSoftmaxThreads - 1
        const int grp = (warp - 2) >> 2;                   // column group
        const int r = 32 * (warp & 3) + lane;              // query row of the tile = TMEM lane
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        float* xchg = reinterpret_cast<float*>(smem + C::kOffXchg);  // [slot][group][row]
        constexpr int kOW = HD / kGroups;                  // O columns per thread

        // Q tile -> smem, K-major 128B swizzle (granule g of row rr at sw128_offset).
        // All of a thread's loads are issued before any store so that they overlap.
        {
            constexpr int kGran = HD / 8;
            constexpr int kPer = 128 * kGran / kSoftmaxThreads;
            uint4 val[kPer];
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int idx = sidx + t * kSoftmaxThreads;
                const int rr = idx / kGran;
                const int g16 = idx - rr * kGran;
                val[t] = make_uint4(0, 0, 0, 0);
                if (rr < rows_valid) {
                    const RowMap rm = map_row(p, ht, m0 + rr);
                    val[t] = __ldg(reinterpret_cast<const uint4*>(
                        p.q + ((size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * HD + g16 * 8));
                }
            }
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int idx = sidx + t * kSoftmaxThreads;
                const int rr = idx / kGran;
                const int g16 = idx - rr * kGran;
                const uint32_t dst = sQ + (g16 >> 3) * 16384 + sw128_offset(rr, g16 & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(val[t].x), "r"(val[t].y),
                             "r"(val[t].z), "r"(val[t].w)
                             : "memory");
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_qfull);

        const bool row_ok = r < rows_valid;
        const RowMap my = map_row(p, ht, m0 + (row_ok ? r : 0));
        const int diag = my.i + sk - p.sq;
        // tile-wide diagonal range (rows are ordered by query position)
        const int i_lo = map_row(p, ht, m0).i;
        const int i_hi = map_row(p, ht, m0 + max(rows_valid, 1) - 1).i;
        const int diag_lo = i_lo + sk - p.sq;
        const int diag_hi = i_hi + sk - p.sq;
        const bool has_causal = p.causal != 0;
        const bool has_window = p.window_left >= 0;
        const float sl2 = p.scale_log2;
        const int col0 = grp * kCW;

        float m_run = -INFINITY;  // running row max, log2 units (scaled); same in every group
        float l_run = 0.f;        // this group's share of the row sum
        for (int j = 0; j < nblocks; ++j) {
            const int n = br.lo + rotated_block(j, rot, nblocks);
            float x[kCW];
            mbar_wait(bar_sfull(j & 1), (j >> 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxSFull);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kCW / 16; ++c) tmem_ld16(tS0 + (j & 1) * 128 + col0 + lane_off + c * 16, x + c * 16);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar_sempty(j & 1));

            const int blk_first = n * 128, blk_last = n * 128 + 127;
            const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                   (has_window && blk_first < diag_hi - p.window_left) || rows_valid < 128;
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < kCW; ++c) {
                    const int key = blk_first + col0 + c;
                    const bool vis = row_ok && key < sk && !(has_causal && key > diag) &&
                                     !(has_window && key < diag - p.window_left);
                    if (!vis) x[c] = -INFINITY;
                }
            }
            float mx8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx8[c] = x[c];
#pragma unroll
            for (int c = 8; c < kCW; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], x[c]);
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            // row max over the groups (double-buffered exchange slot)
            xchg[((j & 1) * kGroups + grp) * 128 + r] = mx;
            named_bar_sync(1, kSoftmaxThreads);
#pragma unroll
            for (int g = 0; g < kGroups; ++g)
                if (g != grp) mx = fmaxf(mx, xchg[((j & 1) * kGroups + g) * 128 + r]);
            const float cand = mx * sl2;
            bool rescale = false;
            float alpha = 1.f;
            if (cand > m_run + kRescaleThreshold) {
                alpha = fast_exp2(m_run - cand);  // 0 when m_run = -inf
                rescale = (m_run != -INFINITY);
                l_run *= alpha;
                m_run = cand;
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kCW; ++c) {
                x[c] = fast_exp2(fmaf(x[c], sl2, neg_m));
                ls[c & 3] += x[c];
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);

            // Each row rescales its own TMEM lane (this group's HD/kGroups columns) once
            // the previous PV is done.  tcgen05.ld/st are warp-collective
            // (.sync.aligned): the whole warp enters; rows that keep their max x 1.
            if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
                mbar_wait(bar_odone((j - 1) & 1), ((j - 1) >> 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
                tc_fence_after();
                const float a = rescale ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < kOW / 16; ++c) {
                    float o[16];
                    const uint32_t ta = tO + grp * kOW + lane_off + c * 16;
                    tmem_ld16(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] *= a;
                    tmem_st16(ta, o);
                }
                tmem_wait_st();
            }
            // P buffer (j & 1) in TMEM was last read by the PV of block j - 2.
            if (j >= 2) {
                mbar_wait(bar_odone(j & 1), ((j >> 1) - 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
                tc_fence_after();
            }
            // This group's keys of the P row -> TMEM: kCW / 2 columns of packed bf16 pairs.
            {
                uint32_t pk[kCW / 2];
#pragma unroll
                for (int c = 0; c < kCW / 2; ++c) pk[c] = pack_bf16x2(x[2 * c], x[2 * c + 1]);
                const uint32_t ta = tP0 + (j & 1) * 64 + grp * (kCW / 2) + lane_off;
#pragma unroll
                for (int c = 0; c < kCW / 32; ++c) tmem_st16u(ta + c * 16, pk + c * 16);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar_pfull(j & 1));
        }

        // Let the dependent grid (the combine, or the next call's partial kernel)
        // get scheduled; it waits for this grid's completion before reading.
        griddep_launch_dependents();
        // ---- epilogue: row sum over the groups, O / l, this group's HD/kGroups columns
        xchg[grp * 128 + r] = l_run;
        named_bar_sync(1, kSoftmaxThreads);
        float l_tot = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) l_tot += xchg[g * 128 + r];
        if (nblocks >= 1) {
            mbar_wait(bar_odone((nblocks - 1) & 1), ((nblocks - 1) >> 1) & 1, wc,
                      (kKernPrefill << 8) | kSiteSoftmaxODone);
            tc_fence_after();
        }
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        const float lse = l_tot > 0.f ? (m_run + log2f(l_tot)) * kLn2 : -INFINITY;
        const bool final_out = (sb == 1);
#pragma unroll
        for (int c = 0; c < kOW / 16; ++c) {
            float o[16];
            if (nblocks >= 1) {
                tmem_ld16(tO + grp * kOW + lane_off + c * 16, o);
                tmem_wait_ld();
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = (nblocks >= 1 && l_tot > 0.f) ? o[e] * inv : 0.f;
            const int dcol = grp * kOW + c * 16;
            if (row_ok) {
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
        }
        if (row_ok && grp == 0) {
            if (final_out)
                p.lse[(size_t(b) * p.Hq + my.h) * p.sq + my.i] = lse;
            else
                p.lse_part[((size_t(tc.split) * p.B + b) * p.Hq + my.h) * p.sq + my.i] = lse;
        }
        tc_fence_before();
    }

    __syncthreads();
    // Neither CTA of a pair leaves while its partner may still multicast into it
    // or arrive on its barriers.
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int HD, class Seqs, bool PAIR>
cudaError_t launch_one(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const Seqs& seqs, cudaStream_t stream) {
    using C = PrefillCfg<HD>;
    auto kern = fwd_prefill_kernel<HD, Seqs, PAIR>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), C::kSmemAlloc, stream, p, tmK, tmV,
                      seqs, PAIR ? 2 : 1);
}

// Two query heads of one KV head with one split each see the same blocks:
// launch them as a 2-CTA cluster sharing the K/V loads.
inline bool use_pairs(const Plan& plan) {
    return plan.d == 128 && !plan.pack_gqa && plan.G % 2 == 0 && plan.num_splits == 1 && plan.grid_y % 2 == 0;
}

}  // namespace

cudaError_t launch_prefill(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t stream) {
    const bool pair = use_pairs(plan);
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        if (plan.d == 128)
            return pair ? launch_one<128, UniformSeqs, true>(plan, p, tmK, tmV, u, stream)
                        : launch_one<128, UniformSeqs, false>(plan, p, tmK, tmV, u, stream);
        return launch_one<64, UniformSeqs, false>(plan, p, tmK, tmV, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    if (plan.d == 128)
        return pair ? launch_one<128, VarlenSeqs, true>(plan, p, tmK, tmV, v, stream)
                    : launch_one<128, VarlenSeqs, false>(plan, p, tmK, tmV, v, stream);
    return launch_one<64, VarlenSeqs, false>(plan, p, tmK, tmV, v, stream);
}

}  // namespace sk
