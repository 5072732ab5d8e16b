// linear_attn_tc.cu -- the segment and output passes of the chunk-parallel gated
// linear attention (inclusionAI/cuLA issue #11) on the tensor cores.
//
// Same recurrence and segments as linear_attn.cu (per sequence b and head h,
// dk = dv = 128, fp32 state):
//   S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t.
// A segment's tokens are taken in windows of at most 128.  Inside a window that
// starts from the state P (the state before its first token) and with
// b_t = sum of g over the window's tokens up to t (per key channel i):
//   S_t = Diag(e^{b_t}) P + sum_{s <= t} Diag(e^{b_t - b_s}) k_s v_s^T
//   o_t = scale * [ (q_t e^{b_t})^T P + sum_{s <= t} <q_t e^{b_t - c}, k_s e^{c - b_s}> v_s ]
// for any per-channel constant c, so the window is four dense products of
// 128 x 128 x 128 (bf16 operands in shared memory, fp32 accumulators in TMEM):
//   A  = Qt Kt^T           Qt[t][i] = q_t[i] e^{b_t[i] - c},  Kt[s][i] = k_s[i] e^{c - b_s[i]}
//   O  = Qt St             St[i][j] = e^{c_i} P[i][j]
//   O += mask(A) V         mask keeps s <= t
//   S   = Diag(e^{b_end}) S + Kh^T V,   Kh[s][i] = k_s[i] e^{b_end[i] - b_s[i]}
// with c the middle of the window's range of b (so every exponent above stays
// within +-30 once the range is at most 60).  A window ends before the first
// token that would widen some channel's range beyond 60; a single token is
// always taken, its log decay clamped to [-100, 100] (exp(-100) is below the
// fp32 normal range, so the clamp changes no fp32 result).  The state itself
// stays fp32 in TMEM across windows; only its copy St for the window's first
// product is rounded to bf16.
//
// One CTA per (segment, head, sequence); 160 threads: warps 0-3 own TMEM lanes
// 0-127 (thread i: key channel i for the operands and the state, token row i
// of A and O); a window's q, k, v rows arrive by TMA in the operand
// tiles' layout and are turned into the decayed operands in place, its log
// decays by TMA as a row-major fp32 block; warp 4 issues the MMAs from one
// elected lane.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fwd_common.cuh"
#include "linear_attn.h"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kD = kLinearAttnDim;  // 128 = dk = dv = window rows
constexpr int kTcThreads = 160;
constexpr int kTile = kD * kD * 2;   // one 128 x 128 bf16 operand tile, two 64-column SW128 chunks
constexpr int kOffQ = 0;             // Qt [t][i]
constexpr int kOffK = kTile;         // Kt [s][i]
constexpr int kOffKh = 2 * kTile;    // Kh [s][i]
constexpr int kOffV = 3 * kTile;     // V  [s][j]
constexpr int kOffA = 4 * kTile;     // mask(A) [t][s]
constexpr int kOffS = 5 * kTile;     // St [i][j]
constexpr int kOffMisc = 6 * kTile;  // window ends, barriers, TMEM address, flags
constexpr int kSmemTc = kOffMisc + 1024 + 1024;  // + misc + alignment slack
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWindowRange = 60.f;  // largest range of b inside a window of more than one token
constexpr float kLogDecayClamp = 100.f;

enum : uint32_t {
    kKernLinear = 3,
    kSiteLinOperands = 11,  // MMA warp waits for a window's operands
    kSiteLinMasked = 12,    // MMA warp waits for mask(A) and the scaled state
    kSiteLinScores = 13,    // operand warps wait for A
    kSiteLinOut = 14,       // operand warps wait for O
    kSiteLinState = 15,     // operand warps wait for the state update
    kSiteLinLoad = 16,      // operand warps wait for a window's q, k, v copies
};

struct LaTcParams {
    __nv_bfloat16* out;
    float* hs;     // [N][B][H][dk][dv]: h_s, then (after the combine) S_in(s)
    float* logm;   // [N][B][H][dk]
    uint32_t* status;
    uint64_t timeout_ns;
    int B, T, H, N, L;
    float scale;
    int clear_status;  // 1 on the call's first launch: CTA (0, 0, 0) zeroes the status word
};

__device__ __forceinline__ unsigned short bf16_bits(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const unsigned short*>(&h);
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float clamp_g(float x) {
    return fminf(fmaxf(x, -kLogDecayClamp), kLogDecayClamp);
}

// Columns 32 q .. 32 q + 31 of row `row` of a tile from 32 fp32 values (times
// `mul`), as 4 16-byte stores.
__device__ __forceinline__ void store_row32_bf16(uint32_t tile, int row, int q, const float* x, float mul) {
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
        const int gg = 4 * q + g8;  // 16-byte granule of the row, 0 .. 15
        const uint32_t a = pack_bf16x2(x[8 * g8] * mul, x[8 * g8 + 1] * mul);
        const uint32_t b = pack_bf16x2(x[8 * g8 + 2] * mul, x[8 * g8 + 3] * mul);
        const uint32_t c = pack_bf16x2(x[8 * g8 + 4] * mul, x[8 * g8 + 5] * mul);
        const uint32_t d = pack_bf16x2(x[8 * g8 + 6] * mul, x[8 * g8 + 7] * mul);
        const uint32_t dst = tile + uint32_t(gg >> 3) * 16384u + sw128_offset(row, gg & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(a), "r"(b), "r"(c), "r"(d)
                     : "memory");
    }
}
// 32 columns of a TMEM row (lane of this warp's quarter, columns col .. col + 31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* x) {
    tmem_ld16(taddr, x);
    tmem_ld16(taddr + 16, x + 16);
    tmem_wait_ld();
}

// OUT = false: the segment pass (h_s and log M_s from a zero state, segments
// 0 .. N-2); OUT = true: the output pass (o_t from S_in(s), every segment).
template <bool OUT>
__global__ void __launch_bounds__(kTcThreads, 1)
    gla_tc_kernel(const __grid_constant__ LaTcParams p, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmG) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t0 = seg * p.L, t1 = min(p.T, (seg + 1) * p.L);

    const uint32_t base = smem_u32(smem);
    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sKh = base + kOffKh, sV = base + kOffV;
    const uint32_t sA = base + kOffA, sS = base + kOffS;
    int* wmin = reinterpret_cast<int*>(smem + kOffMisc);          // [4] per-warp window ends
    volatile int* win_n = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 20);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc + 24);
    const uint32_t bars = base + kOffMisc + 64;
    const uint32_t bar_op = bars, bar_at = bars + 8, bar_a = bars + 16, bar_o = bars + 24, bar_s = bars + 32,
                   bar_drain = bars + 40, bar_ld = bars + 48;

    if (threadIdx.x == 0) {
        if (p.clear_status && seg == 0 && h == 0 && b == 0) *p.status = 0u;
        mbar_init(bar_op, 128);
        mbar_init(bar_at, 128);
        mbar_init(bar_a, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_ld, 1);
        *abort_flag = 0;
        *win_n = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmG);
        if (OUT) tma_prefetch_desc(&tmQ);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tA = tmem, tO = tmem + 128, tS = tmem + 256;  // A, O, S: 128 columns each
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp < 4) {
        // ===================== operand warps: thread i = key channel / TMEM lane i
        const int i = threadIdx.x;
        const uint32_t lane_off = uint32_t(32 * warp) << 16;
        const size_t tok = size_t(p.H) * kD;                              // elements between tokens

        // The state in TMEM: S_in(s) (output pass, s > 0) or zero.
        {
            const float* src = (OUT && seg > 0) ? p.hs + ((size_t(seg) * p.B + b) * p.H + h) * kD * kD + size_t(i) * kD
                                                : nullptr;
#pragma unroll
            for (int c = 0; c < kD / 16; ++c) {
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float4 v4 = src ? *reinterpret_cast<const float4*>(src + c * 16 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[e] = v4.x; x[e + 1] = v4.y; x[e + 2] = v4.z; x[e + 3] = v4.w;
                }
                tmem_st16(tS + lane_off + c * 16, x);
            }
            tmem_wait_st();
        }

        float gsum = 0.f;  // segment pass: log M_s of channel i
        int u0 = t0;
        // The loop's control flow depends on nothing a wait returns: a wait that
        // gives up raises the abort flag, every later wait returns at once, and
        // the windows (at least one token each) still run to the segment's end,
        // so the warp-collective TMEM accesses stay convergent.
        for (int w = 0;; ++w) {
            if (u0 >= t1) {
                if (i == 0) *win_n = 0;
                tc_fence_before();
                mbar_arrive(bar_op);
                break;
            }
            // ---- the window's 128 rows of q, k, v by TMA (raw, into the operand
            // tiles, transformed in place below) and of g (fp32, row-major, into
            // the mask(A) and St tiles, free until the products need them); the
            // previous window's products have all completed (bar_s).
            if (i == 0) {
                const uint64_t pol = l2_policy_evict_first();
                const int row = b * p.T + u0;
                mbar_arrive_expect_tx(bar_ld, uint32_t((OUT ? 3 : 2) * kTile + kD * kD * 4));
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    tma_load_2d(sK + cc * 16384, &tmK, bar_ld, h * kD + cc * 64, row, pol);
                    tma_load_2d(sV + cc * 16384, &tmV, bar_ld, h * kD + cc * 64, row, pol);
                    if (OUT) tma_load_2d(sQ + cc * 16384, &tmQ, bar_ld, h * kD + cc * 64, row, pol);
                }
                tma_load_2d(sA, &tmG, bar_ld, h * kD, row, pol);
            }
            mbar_wait(bar_ld, w & 1, wc, (kKernLinear << 8) | kSiteLinLoad);
            const float* gs = reinterpret_cast<const float*>(smem + kOffA) + i;  // g of row r: gs[r * kD]
            // ---- window end: before the first token that widens a channel's range
            // of b beyond kWindowRange (the window's first token always counts)
            const int cap = min(u0 + kD, t1);
            // the range mx - mn of the running sums never shrinks, so the rows
            // before the first violation are those where it is still in bounds
            int end;
            {
                float cum = 0.f, mx = 0.f, mn = 0.f;
                int in_range = 0;
#pragma unroll 8
                for (int r = 0; r < kD; ++r) {
                    cum += clamp_g(gs[r * kD]);
                    mx = fmaxf(mx, cum);
                    mn = fminf(mn, cum);
                    in_range += (r == 0 || mx - mn <= kWindowRange) ? 1 : 0;
                }
                end = min(u0 + in_range, cap);
            }
            end = __reduce_min_sync(0xffffffffu, end);
            if (lane == 0) wmin[warp] = end;
            named_bar_sync(1, 128);
            const int u1 = min(min(wmin[0], wmin[1]), min(wmin[2], wmin[3]));
            const int n = u1 - u0;
            // ---- the window's range of b for channel i: centre c and end value
            float bend = 0.f, c = 0.f;
            {
                float cum = 0.f, mx = 0.f, mn = 0.f;
#pragma unroll 8
                for (int r = 0; r < kD; ++r) {
                    const float gr = clamp_g(gs[r * kD]);
                    if (r < n) {
                        cum += gr;
                        mx = fmaxf(mx, cum);
                        mn = fminf(mn, cum);
                    }
                }
                bend = cum;
                c = 0.5f * (mx + mn);
            }
            gsum += bend;
            // ---- operands in place, row r = token u0 + r; rows past the window are
            // zero.  Rows go in batches of 16 whose raw q, k and g are read first,
            // so the shared-memory loads of a batch are in flight together.
            {
                unsigned short* tQ = reinterpret_cast<unsigned short*>(smem + kOffQ);
                unsigned short* tK = reinterpret_cast<unsigned short*>(smem + kOffK);
                unsigned short* tKh = reinterpret_cast<unsigned short*>(smem + kOffKh);
                unsigned short* tV = reinterpret_cast<unsigned short*>(smem + kOffV);
                // element (row r, column i) of a 128 x 128 bf16 tile of two 64-column SW128
                // chunks: chunk i / 64, then row r, 16-byte granule (i % 64) / 8 swizzled by r
                const uint32_t o0 = uint32_t(i >> 6) * 16384u + uint32_t(i & 7) * 2u;
                const int gi = (i & 63) >> 3;
                const float ehc = fast_exp2((bend - c) * kLog2e);
                float cum = 0.f;
#pragma unroll 1
                for (int r0 = 0; r0 < kD; r0 += 16) {
                    unsigned short kraw[16], qraw[16];
                    float gr[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        const uint32_t o = (o0 + sw128_offset(r0 + r, gi)) >> 1;
                        kraw[r] = tK[o];
                        if constexpr (OUT) qraw[r] = tQ[o];
                        gr[r] = clamp_g(gs[(r0 + r) * kD]);
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        const uint32_t o = (o0 + sw128_offset(r0 + r, gi)) >> 1;
                        const bool in = r0 + r < n;
                        cum += in ? gr[r] : 0.f;
                        const float ek = fast_exp2((c - cum) * kLog2e);  // e^{c - b}
                        const float kv = __uint_as_float(uint32_t(kraw[r]) << 16);
                        tKh[o] = in ? bf16_bits(kv * (ek * ehc)) : (unsigned short)0;  // e^{b_end - b}
                        if constexpr (OUT) {
                            const float qv = __uint_as_float(uint32_t(qraw[r]) << 16);
                            tQ[o] = in ? bf16_bits(qv * fast_exp2((cum - c) * kLog2e)) : (unsigned short)0;
                            tK[o] = in ? bf16_bits(kv * ek) : (unsigned short)0;
                        }
                        if (!in) tV[o] = 0;
                    }
                }
            }
            named_bar_sync(1, 128);  // every thread is done with g before St overwrites it
            if constexpr (OUT) {
                // St row i = e^{c} P[i][:] (P: the state before the window, in TMEM)
                const float ec = fast_exp2(c * kLog2e);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[32];
                    tmem_ld32(tS + lane_off + q * 32, x);
                    store_row32_bf16(sS, i, q, x, ec);
                }
            } else {
                // segment pass: scale the state now (no product reads it before MMA_S)
                const float e = fast_exp2(bend * kLog2e);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[32];
                    tmem_ld32(tS + lane_off + q * 32, x);
#pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4) x[e4] *= e;
                    tmem_st16(tS + lane_off + q * 32, x);
                    tmem_st16(tS + lane_off + q * 32 + 16, x + 16);
                }
                tmem_wait_st();
            }
            if (i == 0) *win_n = n;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_op);

            if constexpr (OUT) {
                // ---- mask(A) row t = i: keep s <= t; then scale the state
                mbar_wait(bar_a, w & 1, wc, (kKernLinear << 8) | kSiteLinScores);
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[32];
                    tmem_ld32(tA + lane_off + q * 32, x);
#pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4)
                        if (q * 32 + e4 > i) x[e4] = 0.f;
                    store_row32_bf16(sA, i, q, x, 1.f);
                }
                {
                    const float e = fast_exp2(bend * kLog2e);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float x[32];
                        tmem_ld32(tS + lane_off + q * 32, x);
#pragma unroll
                        for (int e4 = 0; e4 < 32; ++e4) x[e4] *= e;
                        tmem_st16(tS + lane_off + q * 32, x);
                        tmem_st16(tS + lane_off + q * 32 + 16, x + 16);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar_at);
                // ---- outputs of the window: token row t = i of O
                mbar_wait(bar_o, w & 1, wc, (kKernLinear << 8) | kSiteLinOut);
                tc_fence_after();
                // O row t = i (all 128 value columns) straight to global memory.  The
                // TMEM loads are warp-collective: every lane takes part, only the
                // rows of the window are stored.
                {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t(b) * p.T + u0 + i) * tok + size_t(h) * kD);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float x[32];
                        tmem_ld32(tO + lane_off + q * 32, x);
#pragma unroll
                        for (int g8 = 0; g8 < 4; ++g8) {
                            uint4 v4;
                            v4.x = pack_bf16x2(x[8 * g8] * p.scale, x[8 * g8 + 1] * p.scale);
                            v4.y = pack_bf16x2(x[8 * g8 + 2] * p.scale, x[8 * g8 + 3] * p.scale);
                            v4.z = pack_bf16x2(x[8 * g8 + 4] * p.scale, x[8 * g8 + 5] * p.scale);
                            v4.w = pack_bf16x2(x[8 * g8 + 6] * p.scale, x[8 * g8 + 7] * p.scale);
                            if (i < n) dst[4 * q + g8] = v4;
                        }
                    }
                }
            }
            mbar_wait(bar_s, w & 1, wc, (kKernLinear << 8) | kSiteLinState);
            tc_fence_after();
            u0 += n;
        }
        if constexpr (!OUT) {
            // h_s (the end state from zero) and log M_s
            float* dst = p.hs + ((size_t(seg) * p.B + b) * p.H + h) * kD * kD + size_t(i) * kD;
#pragma unroll
            for (int cc = 0; cc < kD / 16; ++cc) {
                float x[16];
                tmem_ld16(tS + lane_off + cc * 16, x);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(dst + cc * 16 + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            }
            p.logm[((size_t(seg) * p.B + b) * p.H + h) * kD + i] = gsum;
        }
    } else if (warp == 4) {
        // ===================== MMA issuer (the whole warp runs the loop)
        const bool leader = elect_one();
        // K-major operand: rows = M (or N) index, 64-column chunks of K; a K step
        // of 16 moves 32 bytes inside a chunk.  MN-major operand: rows = K index,
        // 64-column chunks of M (or N) 16 KB apart; a K step moves 16 rows.
        auto kmaj = [](uint32_t tile, int kk) {
            return make_sdesc_sw128(tile, 16, 1024) + uint64_t(uint32_t((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        };
        auto mnmaj = [](uint32_t tile, int kk) {
            return make_sdesc_sw128(tile, 16384, 1024) + uint64_t(uint32_t(kk * 2048) >> 4);
        };
        constexpr uint32_t id_kk = make_idesc_bf16(128, 128, false, false);
        constexpr uint32_t id_km = make_idesc_bf16(128, 128, false, true);
        constexpr uint32_t id_mm = make_idesc_bf16(128, 128, true, true);
        bool ok = true;
        for (int w = 0;; ++w) {
            ok = mbar_wait(bar_op, w & 1, wc, (kKernLinear << 8) | kSiteLinOperands) && ok;
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const int n = __shfl_sync(0xffffffffu, *win_n, 0);
            if (n == 0 || !ok) break;
            __syncwarp();
            if constexpr (OUT) {
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)  // A[t][s] = sum_i Qt[t][i] Kt[s][i]
                        umma_bf16(tA, kmaj(sQ, kk), kmaj(sK, kk), id_kk, kk > 0 ? 1u : 0u);
                    umma_commit(bar_a);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)  // O[t][j] = sum_i Qt[t][i] St[i][j]
                        umma_bf16(tO, kmaj(sQ, kk), mnmaj(sS, kk), id_km, kk > 0 ? 1u : 0u);
                }
                __syncwarp();
                ok = mbar_wait(bar_at, w & 1, wc, (kKernLinear << 8) | kSiteLinMasked) && ok;
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                __syncwarp();
                if (leader) {
                    if (ok) {
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk)  // O[t][j] += sum_s mask(A)[t][s] V[s][j]
                            umma_bf16(tO, kmaj(sA, kk), mnmaj(sV, kk), id_km, 1u);
                    }
                    umma_commit(bar_o);
                }
            }
            if (leader) {
                if (ok) {
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)  // S[i][j] += sum_s Kh[s][i] V[s][j]
                        umma_bf16(tS, mnmaj(sKh, kk), mnmaj(sV, kk), id_mm, 1u);
                }
                umma_commit(bar_s);
            }
            __syncwarp();
        }
        // every MMA issued above completes before TMEM is released
        if (leader) umma_commit(bar_drain);
        __syncwarp();
        mbar_drain(bar_drain, 0, p.timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t linear_attn_tc_smem() { return size_t(kSmemTc); }

cudaError_t launch_linear_attn_tc(const LinearAttnPlan& lp, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, const CUtensorMap& tmG, const void* q, const void* k,
                                  const void* v,
                                  const float* g, void* out, void* workspace, float scale, uint64_t timeout_ns,
                                  cudaStream_t stream) {
    (void)q;
    (void)k;
    (void)v;
    (void)g;
    LaTcParams p;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.hs = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.hs_off);
    p.logm = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.logm_off);
    p.status = static_cast<uint32_t*>(workspace);
    p.timeout_ns = timeout_ns;
    p.B = lp.B; p.T = lp.T; p.H = lp.H; p.N = lp.N; p.L = lp.L;
    p.scale = scale;
    cudaError_t e;
    if ((e = ensure_smem_attr(reinterpret_cast<const void*>(gla_tc_kernel<false>), kSmemTc)) != cudaSuccess ||
        (e = ensure_smem_attr(reinterpret_cast<const void*>(gla_tc_kernel<true>), kSmemTc)) != cudaSuccess)
        return e;
    p.clear_status = 1;
    if (lp.N > 1) {
        gla_tc_kernel<false><<<dim3(lp.N - 1, lp.H, lp.B), kTcThreads, kSmemTc, stream>>>(p, tmQ, tmK, tmV, tmG);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        p.clear_status = 0;
        if ((e = launch_linear_combine(lp, workspace, stream)) != cudaSuccess) return e;
    }
    gla_tc_kernel<true><<<dim3(lp.N, lp.H, lp.B), kTcThreads, kSmemTc, stream>>>(p, tmQ, tmK, tmV, tmG);
    return cudaGetLastError();
}

}  // namespace sk
