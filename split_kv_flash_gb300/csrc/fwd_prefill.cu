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
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
struct PrefillCfg {
    static constexpr int kStages = HD == 128 ? 2 : 4;
    static constexpr int kKBytes = 128 * HD * 2;
    static constexpr int kVBytes = 128 * HD * 2;
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kQBytes = 128 * HD * 2;
    static constexpr int kPBytes = 128 * 128 * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffStages = kOffQ + kQBytes;
    static constexpr int kOffP = kOffStages + kStages * kStageBytes;
    static constexpr int kOffBars = kOffP + kPBytes;
    static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1 + 1 + 1 + 1;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    static constexpr int kTmemCols = 512;  // S0, S1 (128 columns each), O (HD columns)
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

template <int HD, class Seqs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_prefill_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Seqs seqs) {
    using C = PrefillCfg<HD>;
    constexpr int ST = C::kStages;
    extern __shared__ uint8_t smem_raw[];
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
        if (p.echo_plan && threadIdx.x == 0)
            *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(0, 0, int(word), 0);
        return;
    }
    const int sk = seqs.seq_len(b);
    const int kv_off = seqs.seq_off(b);
    const BlockRange br =
        n_block_range(p.sq, sk, tc.m_block, p.kBlockM, p.kBlockN, p.flags, p.pack_gqa != 0, p.G, word);
    const int nblocks = br.hi > br.lo ? br.hi - br.lo : 0;
    if (p.echo_plan && threadIdx.x == 0)
        *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(br.lo, br.hi, int(word), 1);
    const int m0 = tc.m_block * 128;
    const int rows_valid = min(128, p.rows - m0);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t sP = sbase + C::kOffP;
    const uint32_t bars = sbase + C::kOffBars;
    auto bar_full = [&](int s) { return bars + 8u * s; };
    auto bar_empty = [&](int s) { return bars + 8u * (ST + s); };
    auto bar_sfull = [&](int i) { return bars + 8u * (2 * ST + i); };
    auto bar_sempty = [&](int i) { return bars + 8u * (2 * ST + 2 + i); };
    const uint32_t bar_pfull = bars + 8u * (2 * ST + 4);
    const uint32_t bar_odone = bars + 8u * (2 * ST + 5);
    const uint32_t bar_qfull = bars + 8u * (2 * ST + 6);
    const uint32_t bar_never = bars + 8u * (2 * ST + 7);
    const uint32_t bar_drain = bars + 8u * (2 * ST + 8);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    auto stage_k = [&](int s) { return sbase + C::kOffStages + uint32_t(s) * C::kStageBytes; };
    auto stage_v = [&](int s) { return stage_k(s) + C::kKBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull(i), 1);
            mbar_init(bar_sempty(i), 128);
        }
        mbar_init(bar_pfull, 128);
        mbar_init(bar_odone, 1);
        mbar_init(bar_qfull, 128);
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
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS0 = tmem;        // columns [0,128) and [128,256)
    const uint32_t tO = tmem + 256;   // columns [256, 256 + HD)
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) {
            // K/V of one head are re-read by the other m blocks: keep them in L2.
            const uint64_t pol = l2_policy_evict_last();
            int issued = 0;
            for (int j = 0; j < nblocks; ++j) {
                const int s = j % ST;
                const int u = j / ST;
                if (u >= 1 && !mbar_wait(bar_empty(s), (u - 1) & 1, wc, (kKernPrefill << 8) | kSiteProducerEmpty))
                    break;
                mbar_arrive_expect_tx(bar_full(s), C::kKBytes + C::kVBytes);
                const int y = kv_off + (br.lo + j) * 128;
                const int kvh = p.pack_gqa ? ht : ht / p.G;
#pragma unroll
                for (int c = 0; c < HD / 64; ++c) {
                    tma_load_2d(stage_k(s) + c * 16384, &tmK, bar_full(s), kvh * HD + c * 64, y, pol);
                    tma_load_2d(stage_v(s) + c * 16384, &tmV, bar_full(s), kvh * HD + c * 64, y, pol);
                }
                issued = j + 1;
            }
            for (int j = issued - 1; j >= 0 && j >= issued - ST; --j)
                mbar_drain(bar_full(j % ST), (j / ST) & 1, p.timeout_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = make_idesc_bf16(128, HD, false, true);
            bool ok = true;
            if (p.inject_stall) ok = mbar_wait(bar_never, 0, wc, (kKernPrefill << 8) | kSiteInjected);
            if (nblocks > 0) ok = mbar_wait(bar_qfull, 0, wc, (kKernPrefill << 8) | kSiteMmaQ) && ok;
            auto issue_pv = [&](int jj) {
                const bool good = mbar_wait(bar_pfull, jj & 1, wc, (kKernPrefill << 8) | kSiteMmaPFull);
                tc_fence_after();
                if (good) {
                    const int s = jj % ST;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t a = make_sdesc_sw128(sP + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = make_sdesc_sw128(stage_v(s) + kk * 2048, 16384, 1024);
                        umma_bf16(tO, a, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar_odone);
                    umma_commit(bar_empty(s));
                }
            };
            for (int j = 0; j < nblocks; ++j) {
                const int s = j % ST;
                bool good = mbar_wait(bar_full(s), (j / ST) & 1, wc, (kKernPrefill << 8) | kSiteMmaFull);
                if (j >= 2)
                    good = mbar_wait(bar_sempty(j & 1), ((j >> 1) - 1) & 1, wc,
                                     (kKernPrefill << 8) | kSiteMmaSEmpty) && good;
                tc_fence_after();
                if (good && ok) {
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint64_t a = make_sdesc_sw128(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = make_sdesc_sw128(stage_k(s) + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        umma_bf16(tS0 + (j & 1) * 128, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar_sfull(j & 1));
                }
                if (j >= 1) issue_pv(j - 1);
            }
            if (nblocks >= 1) issue_pv(nblocks - 1);
            umma_commit(bar_drain);
            mbar_drain(bar_drain, 0, p.timeout_ns);
        }
    } else {
        const int sidx = threadIdx.x - 64;
        const int r = 32 * (warp & 3) + lane;  // query row of the tile = TMEM lane
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;

        // Q tile -> smem, K-major 128B swizzle (granule g of row r at sw128_offset).
        constexpr int kGran = HD / 8;
        for (int idx = sidx; idx < 128 * kGran; idx += 128) {
            const int rr = idx / kGran;
            const int g16 = idx - rr * kGran;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (rr < rows_valid) {
                const RowMap rm = map_row(p, ht, m0 + rr);
                val = __ldg(reinterpret_cast<const uint4*>(
                    p.q + ((size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * HD + g16 * 8));
            }
            const uint32_t dst = sQ + (g16 >> 3) * 16384 + sw128_offset(rr, g16 & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(val.x), "r"(val.y),
                         "r"(val.z), "r"(val.w)
                         : "memory");
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

        float m_run = -INFINITY;  // running max, log2 units (scaled)
        float l_run = 0.f;
        for (int j = 0; j < nblocks; ++j) {
            const int n = br.lo + j;
            float x[128];
            mbar_wait(bar_sfull(j & 1), (j >> 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxSFull);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_ld16(tS0 + (j & 1) * 128 + lane_off + c * 16, x + c * 16);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar_sempty(j & 1));

            const int blk_first = n * 128, blk_last = n * 128 + 127;
            const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                   (has_window && blk_first < diag_hi - p.window_left) || rows_valid < 128;
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int key = blk_first + c;
                    const bool vis = row_ok && key < sk && !(has_causal && key > diag) &&
                                     !(has_window && key < diag - p.window_left);
                    if (!vis) x[c] = -INFINITY;
                }
            }
            float mx = x[0];
#pragma unroll
            for (int c = 1; c < 128; ++c) mx = fmaxf(mx, x[c]);
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
            float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
                x[c + 0] = fast_exp2(fmaf(x[c + 0], sl2, neg_m));
                x[c + 1] = fast_exp2(fmaf(x[c + 1], sl2, neg_m));
                x[c + 2] = fast_exp2(fmaf(x[c + 2], sl2, neg_m));
                x[c + 3] = fast_exp2(fmaf(x[c + 3], sl2, neg_m));
                ls0 += x[c + 0];
                ls1 += x[c + 1];
                ls2 += x[c + 2];
                ls3 += x[c + 3];
            }
            l_run += (ls0 + ls1) + (ls2 + ls3);

            if (j >= 1) {
                mbar_wait(bar_odone, (j - 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
                tc_fence_after();
            }
            // Each row rescales its own TMEM lane.  tcgen05.ld/st are warp-collective
            // (.sync.aligned), so the whole warp enters together; rows that keep
            // their max multiply by 1.
            if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
                const float a = rescale ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < HD / 16; ++c) {
                    float o[16];
                    tmem_ld16(tO + lane_off + c * 16, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] *= a;
                    tmem_st16(tO + lane_off + c * 16, o);
                }
                tmem_wait_st();
            }
            // P row (bf16) -> smem, K-major over keys, 128B swizzle.
#pragma unroll
            for (int g16 = 0; g16 < 16; ++g16) {
                const uint32_t w0 = pack_bf16x2(x[g16 * 8 + 0], x[g16 * 8 + 1]);
                const uint32_t w1 = pack_bf16x2(x[g16 * 8 + 2], x[g16 * 8 + 3]);
                const uint32_t w2 = pack_bf16x2(x[g16 * 8 + 4], x[g16 * 8 + 5]);
                const uint32_t w3 = pack_bf16x2(x[g16 * 8 + 6], x[g16 * 8 + 7]);
                const uint32_t dst = sP + (g16 >> 3) * 16384 + sw128_offset(r, g16 & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w0), "r"(w1),
                             "r"(w2), "r"(w3)
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_pfull);
        }

        // ---- epilogue
        if (nblocks >= 1) {
            mbar_wait(bar_odone, (nblocks - 1) & 1, wc, (kKernPrefill << 8) | kSiteSoftmaxODone);
            tc_fence_after();
        }
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        const bool final_out = (sb == 1);
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
            float o[16];
            if (nblocks >= 1) {
                tmem_ld16(tO + lane_off + c * 16, o);
                tmem_wait_ld();
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = (nblocks >= 1 && l_run > 0.f) ? o[e] * inv : 0.f;
            if (row_ok) {
                if (final_out) {
                    __nv_bfloat16* dst = p.out + ((size_t(b) * p.sq + my.i) * p.Hq + my.h) * HD + c * 16;
                    uint4 w0, w1;
                    w0.x = pack_bf16x2(o[0], o[1]); w0.y = pack_bf16x2(o[2], o[3]);
                    w0.z = pack_bf16x2(o[4], o[5]); w0.w = pack_bf16x2(o[6], o[7]);
                    w1.x = pack_bf16x2(o[8], o[9]); w1.y = pack_bf16x2(o[10], o[11]);
                    w1.z = pack_bf16x2(o[12], o[13]); w1.w = pack_bf16x2(o[14], o[15]);
                    reinterpret_cast<uint4*>(dst)[0] = w0;
                    reinterpret_cast<uint4*>(dst)[1] = w1;
                } else {
                    const size_t prow = ((size_t(tc.split) * p.B + b) * p.Hq + my.h) * p.sq + my.i;
                    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * HD + c * 16);
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
cudaError_t launch_one(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const Seqs& seqs, cudaStream_t stream) {
    using C = PrefillCfg<HD>;
    auto kern = fwd_prefill_kernel<HD, Seqs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    kern<<<grid, kThreads, C::kSmemAlloc, stream>>>(p, tmK, tmV, seqs);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t stream) {
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return plan.d == 128 ? launch_one<128>(plan, p, tmK, tmV, u, stream)
                             : launch_one<64>(plan, p, tmK, tmV, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    return plan.d == 128 ? launch_one<128>(plan, p, tmK, tmV, v, stream)
                         : launch_one<64>(plan, p, tmK, tmV, v, stream);
}

}  // namespace sk
