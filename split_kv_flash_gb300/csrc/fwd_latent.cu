// fwd_latent.cu -- split-KV partial kernel for latent attention: one KV head
// whose rows serve as the keys (576 columns: 512 latent + 64 rotary) and whose
// first 512 columns serve as the values, shared by every query head.  This is
// the absorbed-MLA speculative-verify workload of "The Occupancy Awakening"
// (Kimi K2.6: 16-64 query heads over one latent head, q_len = draft + 1).
//
// One CTA owns (m block of NP packed rows, split, sequence); packed row r is
// query position r / Hq of query head r % Hq (tiling chapter section 6, PackGQA
// with all heads in one group).  As in the decode kernel the 128 keys of a block
// sit on the tcgen05 M axis ("swap AB"):
//   S^T[128 x NP]  = sum over 9 column chunks c of K_c[128 x 64] . Q_c^T[64 x NP]
//   O_g^T[128 x NP] += V_g^T[128 x 128] . P^T[128 x NP],  g = 0..3 (128 value columns each)
// K arrives as copies of three 64-column chunks (48 KB) through a 2-slot ring;
// V arrives as one 32 KB copy per 128-column group through a 2- or 3-slot ring,
// loaded from the same latent rows (the second read of a row hits L2).  Q^T
// arrives by TMA as well.  Online softmax, masks, split epilogue and bounded
// waits are those of the decode kernel (fwd_decode.cu).
//
// Warp roles (224 threads): warp 0 TMA producer of K chunks, warp 6 of V
// groups, warp 1 TMEM owner and MMA issuer, warps 2-5 softmax (thread t <->
// TMEM lane t = key t of S^T and value column t of each O_g^T) and epilogue.
#include <math.h>

#include "fwd_common.cuh"
#include "kv_producer.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kThreads = 224;  // K producer, MMA, 4 softmax warps, V producer
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kDq = kLatentDqk;        // 576
constexpr int kDv = kLatentDv;         // 512
constexpr int kQChunks = kDq / 64;     // 9
constexpr int kVGroups = kDv / 128;    // 4
constexpr int kLatentL2Warm = 2;       // latent blocks of a split range prefetched into L2 before the grid dependency
static_assert(kQChunks % kLatentKChunksPerCopy == 0, "K copies cover whole blocks");

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Ring depths per tile height (K slots of kLatentKChunksPerCopy chunks, V
// groups, P^T buffers): what the shared memory left after Q^T (9 x NP x 128
// bytes) holds.
template <int NP>
struct LatentRings;
template <>
struct LatentRings<16> {
    static constexpr int k = 2, v = 3, p = 2;
};
template <>
struct LatentRings<32> {
    static constexpr int k = 2, v = 2, p = 2;
};

template <int NP>
struct LatentCfg {
    static constexpr int kStagesK = LatentRings<NP>::k;  // K slots
    static constexpr int kStagesV = LatentRings<NP>::v;  // 128-column V groups
    static constexpr int kKChunks = kLatentKChunksPerCopy;  // 64-column chunks per K slot
    static constexpr int kKCopies = kQChunks / kKChunks;    // K copies per block
    static constexpr int kKBytes = kKChunks * 128 * 64 * 2;  // 48 KB
    static constexpr int kVBytes = 128 * 128 * 2;            // 32 KB (two 64-column chunks)
    static constexpr int kQChunkBytes = NP * 128;      // NP rows x 64 columns
    static constexpr int kPBuf = NP * 128 * 2;
    static constexpr int kPBufs = LatentRings<NP>::p;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kStagesK * kKBytes;
    static constexpr int kOffQ = kOffV + kStagesV * kVBytes;
    static constexpr int kOffP = kOffQ + kQChunks * kQChunkBytes;
    static constexpr int kOffRed = kOffP + kPBufs * kPBuf;  // float red[4][NP]
    static constexpr int kOffM = kOffRed + 4 * NP * 4;     // float m[NP]
    static constexpr int kOffAlpha = kOffM + NP * 4;       // float alpha[NP]
    static constexpr int kOffL = kOffAlpha + NP * 4;       // float l[NP]
    static constexpr int kOffDiag = kOffL + NP * 4;        // int diag[NP]
    static constexpr int kOffBars = (kOffDiag + NP * 4 + 7) / 8 * 8;
    static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 1 + 1 + 1;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    static constexpr int kTmemCols = (6 * NP <= 128) ? 128 : (6 * NP <= 256) ? 256 : 512;  // S^T x 2, O_g^T x 4
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
    static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kQChunkBytes % 1024 == 0 && kPBuf % 1024 == 0,
                  "UMMA operands need 1024-byte alignment");
};

template <int NP, class Seqs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_latent_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ Seqs seqs) {
    static_assert(NP <= 32, "the visible-row mask is one 32-bit word");
    using C = LatentCfg<NP>;
    constexpr int KST = C::kStagesK;
    constexpr int VST = C::kStagesV;
    constexpr int NB0 = 2 * KST + 2 * VST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const TileCoord tc = tile_of_cta(blockIdx.x, blockIdx.y, blockIdx.z, p.num_m_blocks, p.num_splits,
                                     p.reverse_m != 0);
    const int b = tc.batch;
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
    const BlockRange br = tile_key_blocks(p.sq, sk, tc.m_block, p.kBlockM, p.kBlockN, p.win, p.G, word);
    const int nblocks = br.hi > br.lo ? br.hi - br.lo : 0;
    const int m0 = tc.m_block * p.kBlockM;
    const int rows_valid = min(p.kBlockM, p.rows - m0);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t sP = sbase + C::kOffP;
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* sm_m = reinterpret_cast<float*>(smem + C::kOffM);
    float* sm_alpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
    int* sm_diag = reinterpret_cast<int*>(smem + C::kOffDiag);
    const uint32_t bars = sbase + C::kOffBars;
    auto bar_kfull = [&](int s) { return bars + 8u * s; };
    auto bar_kempty = [&](int s) { return bars + 8u * (KST + s); };
    auto bar_vfull = [&](int s) { return bars + 8u * (2 * KST + s); };
    auto bar_vempty = [&](int s) { return bars + 8u * (2 * KST + VST + s); };
    auto bar_sfull = [&](int i) { return bars + 8u * (NB0 + i); };
    auto bar_pfull = [&](int i) { return bars + 8u * (NB0 + 2 + i); };
    auto bar_odone = [&](int i) { return bars + 8u * (NB0 + 4 + i); };
    const uint32_t bar_qfull = bars + 8u * (NB0 + 6);
    const uint32_t bar_never = bars + 8u * (NB0 + 7);
    const uint32_t bar_drain = bars + 8u * (NB0 + 8);
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull(i), 1);
            mbar_init(bar_pfull(i), 128);
            mbar_init(bar_odone(i), 1);
        }
        mbar_init(bar_qfull, 1);
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
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        // A split CTA's first latent blocks into L2 while the previous kernel
        // on the stream (the previous call's combine) may still be running: a
        // hint only, global writes land in L2 (as in the decode kernel).  The
        // values are the same rows, so the K copies cover them.
        const int npre = sb > 1 ? min(nblocks, kLatentL2Warm) : 0;
        for (int j = 0; j < npre; ++j)
#pragma unroll
            for (int c = 0; c < C::kKCopies; ++c)
                tma_prefetch_l2_3d(&tmK, 0, kv_off + (br.lo + j) * 128, c * C::kKChunks);
    }
    if (warp == 6 && lane == 0) tma_prefetch_desc(&tmV);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    if (p.echo_plan && threadIdx.x == 0)
        *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(br.lo, br.hi, int(word), 1);
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS0 = tmem;            // S^T buffers: columns [0, NP), [NP, 2NP)
    const uint32_t tO = tmem + 2 * NP;    // O_g^T: columns [2NP + g NP, 2NP + (g+1) NP)
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};
    const int y0 = kv_off + br.lo * 128;  // first latent row of the range

    if (warp == 0 || warp == 6) {
        // ===================== producers: warp 0 streams the 9 K chunks of
        // every block, warp 6 the 4 V groups, each through its own ring, so a
        // K chunk never waits behind a V slot (and the reverse).
        const bool leader = elect_one();
        const uint64_t pol = l2_policy_evict_last();  // rows are read twice (as K, then as V)
        const int where = (kKernDecode << 8) | kSiteProducerEmpty;
        const bool is_k = warp == 0;
        const int slots = is_k ? KST : VST;
        const uint32_t full0 = is_k ? bar_kfull(0) : bar_vfull(0);
        const uint32_t empty0 = is_k ? bar_kempty(0) : bar_vempty(0);
        const uint32_t base = is_k ? stage_k(0) : stage_v(0);
        const uint32_t stride = is_k ? uint32_t(C::kKBytes) : uint32_t(C::kVBytes);
        const int per_block = is_k ? C::kKCopies : kVGroups;
        const CUtensorMap* tm = is_k ? &tmK : &tmV;
        // Q^T first (warp 0): the tile's packed rows are consecutive rows of the
        // [B * q_len * Hq][576] query tensor; rows past the tile's last valid
        // row are padding (their scores are discarded), rows past the tensor
        // arrive as zeros.
        const bool q_issued = is_k && nblocks > 0;
        if (q_issued && leader) {
            constexpr uint32_t kQBytes = uint32_t(kQChunks * C::kQChunkBytes);
            const int qrow = (b * p.sq) * p.Hq + m0;
            mbar_arrive_expect_tx(bar_qfull, kQBytes);
#pragma unroll
            for (int c3 = 0; c3 < 3; ++c3)
                tma_load_3d(sQ + uint32_t(3 * c3 * C::kQChunkBytes), &tmQ, bar_qfull, 0, qrow, 3 * c3,
                            l2_policy_evict_first());
        }
        // Ring positions count the copies issued; a wait that gives up ends the loop.
        int pos = 0;
        for (int j = 0; j < nblocks; ++j) {
            bool ok = true;
            for (int c = 0; c < per_block; ++c) {
                const int sl = pos % slots, u = pos / slots;
                ok = __all_sync(0xffffffffu, u < 1 || mbar_wait(empty0 + 8u * sl, (u - 1) & 1, wc, where));
                if (!ok) break;
                if (leader) {
                    const uint32_t dst = base + uint32_t(sl) * stride, bar = full0 + 8u * sl;
                    const int y = y0 + j * 128;
                    // K copy c: chunks kKChunks c .. kKChunks (c + 1) - 1; V copy c:
                    // chunks 2c, 2c + 1 (value columns 128c .. 128c + 127).
                    mbar_arrive_expect_tx(bar, stride);
                    tma_load_3d(dst, tm, bar, 0, y, is_k ? c * C::kKChunks : 2 * c, pol);
                }
                ++pos;
            }
            if (!ok) break;
        }
        drain_ring(KvRing{base, stride, full0, empty0, slots}, pos, wc.limit_ns);
        if (q_issued) mbar_drain(bar_qfull, 0, wc.limit_ns);
    } else if (warp == 1) {
        // ===================== MMA issuer (whole warp; one elected lane issues)
        const bool leader = elect_one();
        constexpr uint32_t idesc_qk = make_idesc_bf16(128, NP, false, false);
        constexpr uint32_t idesc_pv = make_idesc_bf16(128, NP, true, true);
        const uint64_t kdesc0 = make_sdesc_sw128(stage_k(0), 16, 1024);
        const uint64_t vdesc0 = make_sdesc_sw128(stage_v(0), 16384, 1024);
        const uint64_t qdesc0 = make_sdesc_sw128(sQ, 16, 1024);
        const uint64_t pdesc0 = make_sdesc_noswz(sP, (NP / 8) * 128, 128);
        bool ok = true;
        if (p.inject_stall) {
            const WaitCtl wc_half{wc.abort_flag, wc.status, wc.limit_ns / 2};
            ok = mbar_wait(bar_never, 0, wc_half, (kKernDecode << 8) | kSiteInjected);
        }
        if (nblocks > 0) ok = mbar_wait(bar_qfull, 0, wc, (kKernDecode << 8) | kSiteMmaQ) && ok;
        int kpos = 0, vpos = 0;
        for (int j = 0; j <= nblocks; ++j) {
            if (j < nblocks) {
                for (int c3 = 0; c3 < C::kKCopies; ++c3, ++kpos) {
                    const int s = kpos % KST;
                    const bool good =
                        mbar_wait(bar_kfull(s), (kpos / KST) & 1, wc, (kKernDecode << 8) | kSiteMmaFull);
                    tc_fence_after();
                    __syncwarp();
                    if (leader) {
                        if (good && ok) {
#pragma unroll
                            for (int cc = 0; cc < C::kKChunks; ++cc) {
                                const int c = c3 * C::kKChunks + cc;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t a =
                                        kdesc0 + uint64_t((s * C::kKBytes + cc * 16384 + kk * 32) >> 4);
                                    const uint64_t bd = qdesc0 + uint64_t((c * C::kQChunkBytes + kk * 32) >> 4);
                                    umma_bf16(tS0 + (j & 1) * NP, a, bd, idesc_qk, (c > 0 || kk > 0) ? 1u : 0u);
                                }
                            }
                        }
                        umma_commit(bar_kempty(s));
                    }
                }
                __syncwarp();
                if (leader) umma_commit(bar_sfull(j & 1));
            }
            if (j >= 1) {
                const int jj = j - 1;
                bool good = mbar_wait(bar_pfull(jj & 1), (jj >> 1) & 1, wc, (kKernDecode << 8) | kSiteMmaPFull);
                const int tail_row = sk - (br.lo + jj) * 128;
                for (int g = 0; g < kVGroups; ++g, ++vpos) {
                    const int s = vpos % VST;
                    const bool gv =
                        mbar_wait(bar_vfull(s), (vpos / VST) & 1, wc, (kKernDecode << 8) | kSiteMmaFull) && good;
                    // Rows of the next sequence in the last block: their P is 0,
                    // but 0 * (Inf or NaN) is NaN, so they are zeroed first.
                    if (gv && tail_row < 128) zero_rows<128>(stage_v(s), tail_row, lane);
                    tc_fence_after();
                    __syncwarp();
                    if (leader) {
                        if (gv && ok) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t a = vdesc0 + uint64_t((s * C::kVBytes + kk * 2048) >> 4);
                                const uint64_t bd =
                                    pdesc0 + uint64_t(((jj % C::kPBufs) * C::kPBuf + kk * 2 * (NP / 8) * 128) >> 4);
                                umma_bf16(tO + g * NP, a, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        umma_commit(bar_vempty(s));
                    }
                }
                __syncwarp();
                if (leader) umma_commit(bar_odone(jj & 1));
            }
        }
        __syncwarp();
        if (leader) umma_commit(bar_drain);
        mbar_drain(bar_drain, 0, p.timeout_ns);
    } else if (warp <= 5) {
        // ===================== softmax / correction / epilogue (128 threads)
        const int sidx = threadIdx.x - 64;
        const int kt = 32 * (warp & 3) + lane;  // TMEM lane: key kt of S^T, value column kt of O_g^T
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const int diag_shift = sk - p.sq;

        if (sidx < NP) {
            sm_m[sidx] = -INFINITY;
            sm_diag[sidx] = (sidx < rows_valid) ? map_row(p, 0, m0 + sidx).i + diag_shift : 0;
        }
        named_bar_sync(1, 128);

        const int diag_lo = (rows_valid > 0) ? sm_diag[0] : 0;
        const int diag_hi = (rows_valid > 0) ? sm_diag[rows_valid - 1] : 0;
        const bool has_causal = p.causal != 0;
        const bool has_window = p.window_left >= 0;
        // neg_m[q] = -(running max of row q) in log2 units: 0 until the row
        // sees a key, -1e30 for padding rows (their P is then 0).  Until every
        // valid row has a finite max, every block takes the rescale path.
        float l_t[NP];
        float neg_m[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            l_t[q] = 0.f;
            neg_m[q] = (q < rows_valid) ? 0.f : -1e30f;
        }
        bool unstarted = rows_valid > 0;
        const float sl2 = p.scale_log2;
        const uint32_t p_st = sP + uint32_t((kt >> 3) * (NP / 8) * 128 + (kt & 7) * 16);
        // Rows that see this thread's key, as bits, from a rolled loop (short
        // code: the masked blocks are often a CTA's first, run from a cold
        // instruction cache).
        auto visible_rows = [&](int key) -> unsigned {
            unsigned vis = 0u;
            if (key < sk) {
#pragma unroll 4
                for (int q = 0; q < rows_valid; ++q) {
                    const int dg = sm_diag[q];
                    const bool ok = (!has_causal || key <= dg) && (!has_window || key >= dg - p.window_left);
                    vis |= unsigned(ok) << q;
                }
            }
            return vis;
        };

        for (int j = 0; j < nblocks; ++j) {
            const int n = br.lo + j;
            const uint32_t tS = tS0 + (j & 1) * NP + lane_off;
            float t[NP];
            mbar_wait(bar_sfull(j & 1), (j >> 1) & 1, wc, (kKernDecode << 8) | kSiteSoftmaxSFull);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) tmem_ld16(tS + c * 16, t + c * 16);
            tmem_wait_ld();
            const int key = n * 128 + kt;
            const int blk_first = n * 128, blk_last = n * 128 + 127;
            const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                   (has_window && blk_first < diag_hi - p.window_left);
#pragma unroll
            for (int q = 0; q < NP; ++q) t[q] = fmaf(t[q], sl2, neg_m[q]);
            if (need_mask) {
                const unsigned vis = visible_rows(key);
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    if (!((vis >> q) & 1u)) t[q] = -INFINITY;
            }
            bool need = unstarted;
#pragma unroll
            for (int q = 0; q < NP; ++q) need |= t[q] > kRescaleThreshold;
            if (named_bar_or(1, 128, need)) {
                // Block max of each row from t - neg_m (the scaled score, -inf
                // where masked), new running maxima, scores shifted by the change.
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float v = warp_max_f32(t[q] - neg_m[q]);
                    if (lane == 0) red[(warp & 3) * NP + q] = v;
                }
                named_bar_sync(1, 128);
                bool still = false;
                if (sidx < NP) {
                    const int q = sidx;
                    float a = 1.f;
                    if (q < rows_valid) {
                        const float bm = fmaxf(fmaxf(red[q], red[NP + q]), fmaxf(red[2 * NP + q], red[3 * NP + q]));
                        const float mo = sm_m[q];
                        const float mn = fmaxf(mo, bm);
                        a = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
                        sm_m[q] = mn;
                        still = mn == -INFINITY;
                    }
                    sm_alpha[q] = a;
                }
                unstarted = named_bar_or(1, 128, still);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    if (q < rows_valid) {
                        const float mq = sm_m[q];
                        const float nm = (mq == -INFINITY) ? 0.f : -mq;
                        t[q] += nm - neg_m[q];
                        neg_m[q] = nm;
                    }
                    l_t[q] *= sm_alpha[q];
                }
                if (j >= 1) {
                    mbar_wait(bar_odone((j - 1) & 1), ((j - 1) >> 1) & 1, wc,
                              (kKernDecode << 8) | kSiteSoftmaxODone);
                    tc_fence_after();
                    for (int g = 0; g < kVGroups; ++g) {
#pragma unroll
                        for (int c = 0; c < NP / 16; ++c) {
                            float o[16];
                            const uint32_t ta = tO + g * NP + lane_off + c * 16;
                            tmem_ld16(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] *= sm_alpha[c * 16 + e];
                            tmem_st16(ta, o);
                        }
                    }
                    tmem_wait_st();
                }
            }
            uint32_t pk[NP / 2];
#pragma unroll
            for (int e = 0; e < NP / 2; ++e) {
                const float p0 = fast_exp2(t[2 * e]);
                const float p1 = fast_exp2(t[2 * e + 1]);
                l_t[2 * e] += p0;
                l_t[2 * e + 1] += p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            // P buffer j % kPBufs was last read by the PV of block j - kPBufs.
            if (j >= C::kPBufs) {
                const int jp = j - C::kPBufs;
                mbar_wait(bar_odone(jp & 1), (jp >> 1) & 1, wc, (kKernDecode << 8) | kSiteSoftmaxODone);
                tc_fence_after();
            }
            {
                const uint32_t dst = p_st + uint32_t((j % C::kPBufs) * C::kPBuf);
#pragma unroll
                for (int g = 0; g < NP / 8; ++g)
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + g * 128), "r"(pk[4 * g]),
                                 "r"(pk[4 * g + 1]), "r"(pk[4 * g + 2]), "r"(pk[4 * g + 3])
                                 : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_pfull(j & 1));
        }

        griddep_launch_dependents();
        // ---- epilogue: l across the 128 key lanes, then O_g^T / l
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const float v = warp_sum(l_t[q]);
            if (lane == 0) red[(warp & 3) * NP + q] = v;
        }
        named_bar_sync(1, 128);
        const bool final_out = (sb == 1);
        // Per row: 1 / l (into sm_alpha) and the element offset of its output
        // row (into red, free again once the sums are read), so the stores
        // below need no index arithmetic.
        long long* row_off = reinterpret_cast<long long*>(red);
        float l_row = 0.f;
        if (sidx < NP) l_row = red[sidx] + red[NP + sidx] + red[2 * NP + sidx] + red[3 * NP + sidx];
        named_bar_sync(1, 128);
        if (sidx < NP) {
            const int q = sidx;
            long long off = 0;
            if (q < rows_valid) {
                const RowMap rm = map_row(p, 0, m0 + q);
                off = final_out ? ((long long)(size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * kDv
                                : (((long long)(size_t(tc.split) * p.B + b) * p.Hq + rm.h) * p.sq + rm.i) * kDv;
                const float lse = l_row > 0.f ? (sm_m[q] + log2f(l_row)) * kLn2 : -INFINITY;
                if (final_out)
                    p.lse[(size_t(b) * p.Hq + rm.h) * p.sq + rm.i] = lse;
                else
                    p.lse_part[((size_t(tc.split) * p.B + b) * p.Hq + rm.h) * p.sq + rm.i] = lse;
            }
            row_off[q] = off;
            sm_alpha[q] = l_row > 0.f ? 1.f / l_row : 0.f;
        }
        named_bar_sync(1, 128);
        if (nblocks >= 1) {
            mbar_wait(bar_odone((nblocks - 1) & 1), ((nblocks - 1) >> 1) & 1, wc,
                      (kKernDecode << 8) | kSiteSoftmaxODone);
            tc_fence_after();
        }
#pragma unroll 1
        for (int g = 0; g < kVGroups; ++g) {
            float o[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) o[q] = 0.f;
            if (nblocks >= 1) {
#pragma unroll
                for (int c = 0; c < NP / 16; ++c) tmem_ld16(tO + g * NP + lane_off + c * 16, o + c * 16);
                tmem_wait_ld();
            }
            const int col = g * 128 + kt;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                if (q < rows_valid) {
                    const float val = o[q] * sm_alpha[q];
                    if (final_out)
                        p.out[row_off[q] + col] = __float2bfloat16_rn(val);
                    else
                        p.o_part[row_off[q] + col] = val;
                }
            }
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

template <int NP, class Seqs>
cudaError_t launch_one(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmQ, const Seqs& seqs, cudaStream_t stream) {
    using C = LatentCfg<NP>;
    auto kern = fwd_latent_kernel<NP, Seqs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), C::kSmemAlloc, stream, p, tmK,
                      tmV, tmQ, seqs);
}

template <class Seqs>
cudaError_t dispatch(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     const CUtensorMap& tmQ, const Seqs& seqs, cudaStream_t stream) {
    if (plan.kBlockM == 16) return launch_one<16>(plan, p, tmK, tmV, tmQ, seqs, stream);
    if (plan.kBlockM == 32) return launch_one<32>(plan, p, tmK, tmV, tmQ, seqs, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_latent(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmQ, cudaStream_t stream) {
    if (!plan.latent || plan.d != kDq || plan.dv != kDv || plan.kBlockN != 128) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return dispatch(plan, p, tmK, tmV, tmQ, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    return dispatch(plan, p, tmK, tmV, tmQ, v, stream);
}

}  // namespace sk
