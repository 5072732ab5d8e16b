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
// One CTA per (segment, head, sequence); 288 threads: warps 0-7 are operand
// warps (TMEM lane i % 128 is key channel i % 128 of the state and token row
// i % 128 of the scores and outputs; its two threads take 64 columns each),
// warp 8 issues the MMAs from one elected lane.  A window's q, k, v rows
// arrive by TMA in the operand tiles' layout and are turned into the decayed
// operands in place; its log decays arrive by TMA as a row-major fp32 block.
// Every wait is bounded.
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
constexpr int kMathWarps = 8;         // operand / softmax-free elementwise warps; warp 8 issues the MMAs
constexpr int kMathThreads = 32 * kMathWarps;
constexpr int kTcThreads = kMathThreads + 32;
constexpr int kTile = kD * kD * 2;   // one 128 x 128 bf16 operand tile, two 64-column SW128 chunks
constexpr int kOffQ = 0;             // Qt [t][i]
constexpr int kOffK = kTile;         // Kt [s][i]
constexpr int kOffKh = 2 * kTile;    // Kh [s][i]
constexpr int kOffV = 3 * kTile;     // V  [s][j]
constexpr int kOffA = 4 * kTile;     // mask(A) [t][s]
constexpr int kOffS = 5 * kTile;     // St [i][j]
constexpr int kOffMisc = 6 * kTile;  // window ends, barriers, TMEM address, flags
constexpr int kSmemTc = kOffMisc + 3072 + 1024;  // + misc + alignment slack
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
    int inject_stall;  // test hook: the MMA warp first waits on a barrier nothing signals
};

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
    float* cs = reinterpret_cast<float*>(smem + kOffMisc + 1024);  // [128] window centre c per channel
    float* ehs = cs + kD;                                          // [128] e^{b_end - c} per channel
    float* bnd = cs + 2 * kD;                                      // [128] b_end per channel
    volatile int* win_n = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 20);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc + 24);
    const uint32_t bars = base + kOffMisc + 64;
    const uint32_t bar_op = bars, bar_at = bars + 8, bar_a = bars + 16, bar_o = bars + 24, bar_s = bars + 32,
                   bar_drain = bars + 40, bar_ld = bars + 48, bar_ldv = bars + 56, bar_never = bars + 64;

    if (threadIdx.x == 0) {
        if (p.clear_status && seg == 0 && h == 0 && b == 0) *p.status = 0u;
        mbar_init(bar_op, kMathThreads);
        mbar_init(bar_at, kMathThreads);
        mbar_init(bar_a, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_ld, 1);
        mbar_init(bar_ldv, 1);
        mbar_init(bar_never, 1);
        *abort_flag = 0;
        *win_n = 0;
        fence_mbar_init();
    }
    if (warp == kMathWarps) {
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
    // The next kernel on the stream (the combine, or the output pass) may be
    // scheduled now; it waits for this grid's completion before it reads.
    griddep_launch_dependents();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tA = tmem, tO = tmem + 128, tS = tmem + 256;  // A, O, S: 128 columns each
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp < kMathWarps) {
        // ===================== operand warps.  TMEM lane li = i % 128 belongs to
        // warps w and w + 4 (lane quarter w % 4); thread i takes the 64 columns
        // [64 half, 64 half + 64) of lane li's rows (half = i / 128).  The scans
        // over the rows of a key channel run in the threads of half 0.
        const int i = threadIdx.x;
        const int li = i & 127, half = i >> 7;
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const size_t tok = size_t(p.H) * kD;  // elements between tokens

        // The first window's copies: the inputs are not written by the kernel
        // this grid may overlap (the combine), so they go before the wait below.
        const uint64_t pol = l2_policy_evict_first();
        auto issue_qkg = [&](int ustart) {
            const int row = b * p.T + ustart;
            mbar_arrive_expect_tx(bar_ld, uint32_t((OUT ? 2 : 1) * kTile + kD * kD * 4));
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                tma_load_2d(sK + cc * 16384, &tmK, bar_ld, h * kD + cc * 64, row, pol);
                if (OUT) tma_load_2d(sQ + cc * 16384, &tmQ, bar_ld, h * kD + cc * 64, row, pol);
            }
            tma_load_2d(sA, &tmG, bar_ld, h * kD, row, pol);
        };
        auto issue_v = [&](int ustart) {
            const int row = b * p.T + ustart;
            mbar_arrive_expect_tx(bar_ldv, uint32_t(kTile));
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) tma_load_2d(sV + cc * 16384, &tmV, bar_ldv, h * kD + cc * 64, row, pol);
        };
        if (i == 0 && t0 < t1) {
            issue_qkg(t0);
            issue_v(t0);
        }
        // The incoming states are the previous kernel's output.
        griddep_wait();

        // The state in TMEM: S_in(s) (output pass, s > 0) or zero.
        {
            const float* src = (OUT && seg > 0)
                                   ? p.hs + ((size_t(seg) * p.B + b) * p.H + h) * kD * kD + size_t(li) * kD + 64 * half
                                   : nullptr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float4 v4 = src ? *reinterpret_cast<const float4*>(src + c * 16 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[e] = v4.x; x[e + 1] = v4.y; x[e + 2] = v4.z; x[e + 3] = v4.w;
                }
                tmem_st16(tS + lane_off + 64 * half + c * 16, x);
            }
            tmem_wait_st();
        }

        // Later windows' copies: q (output pass), k and g, whose tiles free up once
        // a window's scores and output products are done, and v, whose tile frees
        // up with the state update; each set is issued as soon as its tiles are
        // free (the next window's start is known by then).
        float gsum = 0.f;  // segment pass: log M_s of channel li (half 0)
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
            // ---- the window's 128 rows of q, k (raw, into the operand tiles,
            // transformed in place below), g (fp32, row-major, into the mask(A)
            // and St tiles, free until the products need them) and v, by TMA
            mbar_wait(bar_ld, w & 1, wc, (kKernLinear << 8) | kSiteLinLoad);
            // ---- running sums b_r of channel li over the 128 rows, in place of g,
            // and the window end: before the first token that widens a channel's
            // range of b beyond kWindowRange (the window's first token always
            // counts).  The range max - min of the running sums never shrinks, so
            // the rows before the first violation are those where it is in bounds.
            const int cap = min(u0 + kD, t1);
            float* gs = reinterpret_cast<float*>(smem + kOffA) + li;  // g of row r: gs[r * kD]
            float mx_all = 0.f, mn_all = 0.f;                          // over the rows before cap
            if (half == 0) {
                float cum = 0.f, mx = 0.f, mn = 0.f;
                int in_range = 0;
#pragma unroll 16
                for (int r = 0; r < kD; ++r) {
                    cum += clamp_g(gs[r * kD]);
                    gs[r * kD] = cum;
                    if (u0 + r < cap) {
                        mx = fmaxf(mx, cum);
                        mn = fminf(mn, cum);
                    }
                    in_range += (r == 0 || mx - mn <= kWindowRange) ? 1 : 0;
                }
                mx_all = mx;
                mn_all = mn;
                int end = min(u0 + in_range, cap);
                end = __reduce_min_sync(0xffffffffu, end);
                if (lane == 0) wmin[warp] = end;
            }
            named_bar_sync(1, kMathThreads);
            const int u1 = min(min(wmin[0], wmin[1]), min(wmin[2], wmin[3]));
            const int n = u1 - u0;
            if (i == kMathThreads - 1 && u1 < t1) {
                // The next window starts at u1: its rows into L2 now, so that its
                // copies, issued once this window's products free the tiles, hit L2.
                const int row = b * p.T + u1;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    tma_prefetch_l2_2d(&tmK, h * kD + cc * 64, row);
                    tma_prefetch_l2_2d(&tmV, h * kD + cc * 64, row);
                    if (OUT) tma_prefetch_l2_2d(&tmQ, h * kD + cc * 64, row);
                }
                tma_prefetch_l2_2d(&tmG, h * kD, row);
            }
            // ---- the window's range of b for channel li (0 included): centre c,
            // end value; when no channel cut the window short it is the range above
            if (half == 0) {
                const float bend = gs[(n - 1) * kD];
                float mx = mx_all, mn = mn_all;
                if (u1 < cap) {
                    float mx8[8], mn8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx8[e] = mn8[e] = 0.f;
#pragma unroll 16
                    for (int r = 0; r < kD; ++r) {
                        const float b_r = gs[r * kD];
                        if (r < n) {
                            mx8[r & 7] = fmaxf(mx8[r & 7], b_r);
                            mn8[r & 7] = fminf(mn8[r & 7], b_r);
                        }
                    }
                    mx = mx8[0];
                    mn = mn8[0];
#pragma unroll
                    for (int e = 1; e < 8; ++e) {
                        mx = fmaxf(mx, mx8[e]);
                        mn = fminf(mn, mn8[e]);
                    }
                }
                const float c = 0.5f * (mx + mn);
                gsum += bend;
                cs[li] = c;
                ehs[li] = fast_exp2((bend - c) * kLog2e);
                bnd[li] = bend;
            }
            named_bar_sync(1, kMathThreads);
            // ---- operands in place, row r = token u0 + r; rows past the window are
            // zero.  Here a thread takes 8 channels (one 16-byte granule of a row,
            // cg = i % 16) of rows i / 16 + 16 m: 16-byte shared accesses.
            {
                const int cg = i & 15, rsub = i >> 4;
                float c8[8], eh8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    c8[e] = cs[8 * cg + e];
                    eh8[e] = ehs[8 * cg + e];
                }
                const uint32_t chunk = uint32_t(cg >> 3) * 16384u;
                const float* brow = reinterpret_cast<const float*>(smem + kOffA) + 8 * cg;
#pragma unroll 2
                for (int m = 0; m < kD / 16; ++m) {
                    const int r = rsub + 16 * m;
                    const uint32_t off = chunk + sw128_offset(r, cg & 7);
                    const bool in = r < n;
                    uint4 kraw, qraw = make_uint4(0u, 0u, 0u, 0u);
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(kraw.x), "=r"(kraw.y), "=r"(kraw.z), "=r"(kraw.w) : "r"(sK + off));
                    if constexpr (OUT)
                        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(qraw.x), "=r"(qraw.y), "=r"(qraw.z), "=r"(qraw.w) : "r"(sQ + off));
                    const float4 b0 = *reinterpret_cast<const float4*>(brow + r * kD);
                    const float4 b1 = *reinterpret_cast<const float4*>(brow + r * kD + 4);
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    const uint32_t kw[4] = {kraw.x, kraw.y, kraw.z, kraw.w};
                    const uint32_t qw[4] = {qraw.x, qraw.y, qraw.z, qraw.w};
                    uint32_t oh[4], ok_[4], oq[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        float kh[2], kt[2], qt[2];
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int e = 2 * e2 + h2;
                            const float kv = __uint_as_float(h2 ? (kw[e2] & 0xFFFF0000u) : (kw[e2] << 16));
                            const float ek = fast_exp2((c8[e] - bv[e]) * kLog2e);  // e^{c - b}
                            kh[h2] = kv * (ek * eh8[e]);                            // k e^{b_end - b}
                            kt[h2] = kv * ek;
                            if constexpr (OUT) {
                                const float qv = __uint_as_float(h2 ? (qw[e2] & 0xFFFF0000u) : (qw[e2] << 16));
                                qt[h2] = qv * fast_exp2((bv[e] - c8[e]) * kLog2e);  // q e^{b - c}
                            } else {
                                qt[h2] = 0.f;
                            }
                        }
                        oh[e2] = in ? pack_bf16x2(kh[0], kh[1]) : 0u;
                        ok_[e2] = in ? pack_bf16x2(kt[0], kt[1]) : 0u;
                        oq[e2] = in ? pack_bf16x2(qt[0], qt[1]) : 0u;
                    }
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sKh + off), "r"(oh[0]), "r"(oh[1]),
                                 "r"(oh[2]), "r"(oh[3]) : "memory");
                    if constexpr (OUT) {
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sK + off), "r"(ok_[0]),
                                     "r"(ok_[1]), "r"(ok_[2]), "r"(ok_[3]) : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sQ + off), "r"(oq[0]),
                                     "r"(oq[1]), "r"(oq[2]), "r"(oq[3]) : "memory");
                    }
                }
                // v rows past the window: zero (0 x Inf would be NaN in the products)
                mbar_wait(bar_ldv, w & 1, wc, (kKernLinear << 8) | kSiteLinLoad);
#pragma unroll 2
                for (int m = 0; m < kD / 16; ++m) {
                    const int r = rsub + 16 * m;
                    if (r >= n)
                        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sV + chunk + sw128_offset(r, cg & 7)),
                                     "r"(0u)
                                     : "memory");
                }
            }
            named_bar_sync(1, kMathThreads);  // every thread is done with g before St overwrites it
            const float bend_l = bnd[li];
            if constexpr (!OUT) {
                // the raw k and g of this window are consumed: the next window's come now
                if (i == 0 && u0 + n < t1) issue_qkg(u0 + n);
            }
            if constexpr (OUT) {
                // St row li = e^{c} P[li][:] (P: the state before the window, in TMEM)
                const float ec = fast_exp2(cs[li] * kLog2e);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int q = 2 * half + q2;
                    float x[32];
                    tmem_ld32(tS + lane_off + q * 32, x);
                    store_row32_bf16(sS, li, q, x, ec);
                }
            } else {
                // segment pass: scale the state now (no product reads it before MMA_S)
                const float e = fast_exp2(bend_l * kLog2e);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int q = 2 * half + q2;
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
                // ---- mask(A) row t = li: keep s <= t; then scale the state
                mbar_wait(bar_a, w & 1, wc, (kKernLinear << 8) | kSiteLinScores);
                tc_fence_after();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int q = 2 * half + q2;
                    float x[32];
                    tmem_ld32(tA + lane_off + q * 32, x);
#pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4)
                        if (q * 32 + e4 > li) x[e4] = 0.f;
                    store_row32_bf16(sA, li, q, x, 1.f);
                }
                {
                    const float e = fast_exp2(bend_l * kLog2e);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const int q = 2 * half + q2;
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
                // ---- outputs of the window: token row t = li of O, this thread's 64
                // value columns straight to global memory.  The TMEM loads are
                // warp-collective: every lane takes part, only the window's rows
                // are stored.
                mbar_wait(bar_o, w & 1, wc, (kKernLinear << 8) | kSiteLinOut);
                tc_fence_after();
                // the scores and output products are done with Qt, Kt, mask(A), St
                if (i == 0 && u0 + n < t1) issue_qkg(u0 + n);
                {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t(b) * p.T + u0 + li) * tok + size_t(h) * kD);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const int q = 2 * half + q2;
                        float x[32];
                        tmem_ld32(tO + lane_off + q * 32, x);
#pragma unroll
                        for (int g8 = 0; g8 < 4; ++g8) {
                            uint4 v4;
                            v4.x = pack_bf16x2(x[8 * g8] * p.scale, x[8 * g8 + 1] * p.scale);
                            v4.y = pack_bf16x2(x[8 * g8 + 2] * p.scale, x[8 * g8 + 3] * p.scale);
                            v4.z = pack_bf16x2(x[8 * g8 + 4] * p.scale, x[8 * g8 + 5] * p.scale);
                            v4.w = pack_bf16x2(x[8 * g8 + 6] * p.scale, x[8 * g8 + 7] * p.scale);
                            if (li < n) dst[4 * q + g8] = v4;
                        }
                    }
                }
            }
            mbar_wait(bar_s, w & 1, wc, (kKernLinear << 8) | kSiteLinState);
            tc_fence_after();
            if (i == 0 && u0 + n < t1) issue_v(u0 + n);  // the state update is done with V
            u0 += n;
        }
        if constexpr (!OUT) {
            // h_s (the end state from zero) and log M_s
            float* dst = p.hs + ((size_t(seg) * p.B + b) * p.H + h) * kD * kD + size_t(li) * kD + 64 * half;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float x[16];
                tmem_ld16(tS + lane_off + 64 * half + cc * 16, x);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(dst + cc * 16 + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            }
            if (half == 0) p.logm[((size_t(seg) * p.B + b) * p.H + h) * kD + li] = gsum;
        }
    } else if (warp == kMathWarps) {
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
        if (p.inject_stall) {
            // gives up first (half the limit), so the status names this wait
            const WaitCtl wc_half{wc.abort_flag, wc.status, wc.limit_ns / 2};
            ok = mbar_wait(bar_never, 0, wc_half, (kKernLinear << 8) | kSiteInjected);
            ok = __all_sync(0xffffffffu, ok);
        }
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
    if (warp == kMathWarps) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t linear_attn_tc_smem() { return size_t(kSmemTc); }

cudaError_t launch_linear_attn_tc(const LinearAttnPlan& lp, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, const CUtensorMap& tmG, const void* q, const void* k,
                                  const void* v,
                                  const float* g, void* out, void* workspace, float scale, uint64_t timeout_ns,
                                  int inject_stall, cudaStream_t stream) {
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
    p.inject_stall = inject_stall;
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
    if (lp.N > 1)  // a programmatic dependent of the combine: its first copies overlap the combine
        return launch_pdl(reinterpret_cast<const void*>(gla_tc_kernel<true>), dim3(lp.N, lp.H, lp.B),
                          dim3(kTcThreads), kSmemTc, stream, p, tmQ, tmK, tmV, tmG);
    gla_tc_kernel<true><<<dim3(lp.N, lp.H, lp.B), kTcThreads, kSmemTc, stream>>>(p, tmQ, tmK, tmV, tmG);
    return cudaGetLastError();
}

}  // namespace sk
