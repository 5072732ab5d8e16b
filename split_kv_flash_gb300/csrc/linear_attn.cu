// linear_attn.cu -- chunk-parallel gated linear attention (inclusionAI/cuLA
// issue #11: each (sequence, head) is split along T into N segments that run in
// parallel CTAs and are merged by an affine combine (M, h_ext)).
//
// Recurrence (per sequence b and head h; dk = dv = 128, fp32 state):
//   S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t,   S_0 = 0
// Segment s covers tokens [s L, min((s + 1) L, T)), L = ceil(T / N).  Started
// from S_in it ends at M_s S_in + h_s with M_s = Diag(exp(sum of g over the
// segment)) and h_s its end state from a zero start.  Three launches:
//   1. gla_segment_kernel  -- one CTA per (segment, head, sequence): h_s and
//      log M_s (the sum of g) for every segment but the last;
//   2. gla_combine_kernel  -- the affine combine S_in(s + 1) = M_s S_in(s) + h_s,
//      S_in(0) = 0, done in place over the h_s buffer (element-parallel);
//   3. gla_output_kernel   -- one CTA per segment again: re-runs the segment
//      from S_in(s) and writes o_t.
// The per-token work is a rank-1 update of the state (no dense contraction), so
// it runs on the FMA pipes: 512 threads hold the 128 x 128 state as 8 x 4
// blocks, thread (rg = tid % 16, cg = tid / 16) owning rows 4 rg .. 4 rg + 3 and
// 64 + 4 rg .. 64 + 4 rg + 3 (consecutive lanes read consecutive 16-byte words:
// no bank conflicts) and columns 4 cg .. 4 cg + 3, so a token costs each thread
// 7 16-byte shared loads
// (k, the decays and q of its rows, v of its columns) and the output's sum
// over rows is a reduction over the 16 lanes of a half-warp.  Tokens
// are staged in shared memory 32 at a time (k, v, q converted to fp32), the
// next chunk's loads in flight in registers meanwhile; within a chunk the state
// is carried rescaled by the chunk's cumulative decay (see Stage), so a token
// costs one FMA per state element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fwd_common.cuh"
#include "linear_attn.h"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kD = kLinearAttnDim;   // 128 = dk = dv
constexpr int kThreads = 512;
constexpr int kTC = 32;              // tokens per staged chunk
constexpr int kR = 8;                // state rows per thread
constexpr int kC = 4;                // state columns per thread
constexpr int kS = kR * kC;

struct LaParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    __nv_bfloat16* out;
    float* hs;     // [N][B][H][dk][dv]: h_s, then (after the combine) S_in(s)
    float* logm;   // [N][B][H][dk]
    uint32_t* status;  // workspace header word: this path has no bounded wait, so it only clears it
    int B, T, H, N, L;
    float scale;
    int clear_status;  // 1 on the call's first launch: CTA (0, 0, 0) zeroes the status word
};

// Shared-memory staging of one chunk: fp32 k, exp(g), v and (output pass) q.
// With cum_t = sum of g over the chunk's tokens up to t (per key channel), the
// state is carried as S'_t = S_t / exp(cum_t) inside a chunk, so a token costs
// one FMA per state element: S'_t = S'_{t-1} + (k_t exp(-cum_t)) v_t^T, and
// o_t = scale * S'_t^T (q_t exp(cum_t)); at the chunk's end S = S' exp(cum_end).
// A chunk in which some cum_t leaves [kCumFloor, -kCumFloor] (exp(-cum_t) would
// approach the ends of the fp32 range) runs the plain update S = exp(g) S + k v^T.
constexpr float kCumFloor = -60.f;

struct Stage {
    float k[kTC][kD];    // k, then (rescaled chunks) k exp(-cum)
    float q[kTC][kD];    // q, then (rescaled chunks) q exp(cum)
    float v[kTC][kD];
    float g[kTC][kD];    // raw log decays
    float a[kTC][kD];    // exp(g) (plain chunks)
    float ecend[kD];     // exp(cum at the chunk's last token)
};

// Register copy of one chunk's raw inputs for thread tid (loaded ahead of use).
struct Raw {
    uint4 k, v, q;   // 8 bf16 each: token tid / 16, columns 8 (tid % 16) ..
    float4 g[2];     // 4 floats each: tokens (tid + 512 u) / 32, channels 4 ((tid + 512 u) % 32) ..
};

// State row of thread-local row i (0..7) for row group rg.
__device__ __forceinline__ int state_row(int rg, int i) { return (i < 4 ? 0 : 64 - 4) + 4 * rg + i; }

__device__ __forceinline__ size_t tok_row(const LaParams& p, int b, int t, int h) {
    return (size_t(b) * p.T + t) * p.H + h;
}

__device__ __forceinline__ void load_raw(const LaParams& p, int b, int h, int t0, int t1, bool with_q, Raw& r) {
    const int tid = threadIdx.x;
    const int tk = tid >> 4, c8 = (tid & 15) * 8;
    const int t = t0 + tk;
    r.k = r.v = r.q = make_uint4(0, 0, 0, 0);
    if (t < t1) {
        const size_t off = tok_row(p, b, t, h) * kD + c8;
        r.k = __ldg(reinterpret_cast<const uint4*>(p.k + off));
        r.v = __ldg(reinterpret_cast<const uint4*>(p.v + off));
        if (with_q) r.q = __ldg(reinterpret_cast<const uint4*>(p.q + off));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + kThreads * u;
        const int tg = t0 + e / 32, c4 = (e % 32) * 4;
        r.g[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tg < t1) r.g[u] = __ldg(reinterpret_cast<const float4*>(p.g + tok_row(p, b, tg, h) * kD + c4));
    }
}

__device__ __forceinline__ void bf8_to_f32(uint4 w, float* dst) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[2 * i] = __uint_as_float(x[i] << 16);
        dst[2 * i + 1] = __uint_as_float(x[i] & 0xffff0000u);
    }
}

// Raw -> shared stage; also adds this thread's four channels of g to gsum.
__device__ __forceinline__ void store_stage(const Raw& r, Stage& s, bool with_q, float* gsum) {
    const int tid = threadIdx.x;
    const int tk = tid >> 4, c8 = (tid & 15) * 8;
    float f[8];
    bf8_to_f32(r.k, f);
    *reinterpret_cast<float4*>(&s.k[tk][c8]) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(&s.k[tk][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    bf8_to_f32(r.v, f);
    *reinterpret_cast<float4*>(&s.v[tk][c8]) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(&s.v[tk][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    if (with_q) {
        bf8_to_f32(r.q, f);
        *reinterpret_cast<float4*>(&s.q[tk][c8]) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(&s.q[tk][c8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + kThreads * u;
        const int tg = e / 32, c4 = (e % 32) * 4;
        const float gv[4] = {r.g[u].x, r.g[u].y, r.g[u].z, r.g[u].w};
        *reinterpret_cast<float4*>(&s.g[tg][c4]) = r.g[u];
        *reinterpret_cast<float4*>(&s.a[tg][c4]) = make_float4(__expf(gv[0]), __expf(gv[1]), __expf(gv[2]), __expf(gv[3]));
#pragma unroll
        for (int i = 0; i < 4; ++i) gsum[i] += gv[i];
    }
}

// After the chunk is staged: channel c = tid (tid < 128) accumulates cum over
// the chunk's n tokens; unless some channel's cum leaves [kCumFloor, -kCumFloor]
// (then the chunk takes the plain update, which this returns to every thread),
// each channel rescales its k (and q) column.
template <bool OUT>
__device__ __forceinline__ bool rescale_chunk(Stage& s, int n) {
    const int c = threadIdx.x;
    bool out_of_range = false;
    if (c < kD) {
        float cum = 0.f;
        for (int t = 0; t < n; ++t) {
            cum += s.g[t][c];
            out_of_range |= cum < kCumFloor || cum > -kCumFloor;
        }
    }
    const bool plain = __syncthreads_or(out_of_range) != 0;
    if (!plain) {
        if (c < kD) {
            float cum = 0.f;
            for (int t = 0; t < n; ++t) {
                cum += s.g[t][c];
                s.k[t][c] *= __expf(-cum);
                if (OUT) s.q[t][c] *= __expf(cum);
            }
            s.ecend[c] = __expf(cum);
        }
        __syncthreads();
    }
    return plain;
}

// One pass over tokens [t0, t1) of (b, h) on the state S held in registers;
// with OUT the outputs o_t go to global memory (staged per chunk).
template <bool OUT>
__device__ __forceinline__ void run_tokens(const LaParams& p, int b, int h, int t0, int t1, float (&S)[kS],
                                           Stage& s, float* gsum, __nv_bfloat16 (*osm)[kD]) {
    const int tid = threadIdx.x;
    const int rg = tid & 15, cg = tid >> 4;
    const int nch = (t1 - t0 + kTC - 1) / kTC;
    Raw raw;
    if (nch > 0) load_raw(p, b, h, t0, t1, OUT, raw);
    for (int c = 0; c < nch; ++c) {
        store_stage(raw, s, OUT, gsum);
        __syncthreads();
        const int c0 = t0 + c * kTC;
        const int n = min(kTC, t1 - c0);
        if (c + 1 < nch) load_raw(p, b, h, c0 + kTC, t1, OUT, raw);  // next chunk, in flight during this one
        const bool plain = rescale_chunk<OUT>(s, n);
        // Two tokens per iteration: the next token's state update overlaps this
        // token's output reduction.
#pragma unroll 2
        for (int t = 0; t < n; ++t) {
            const float4 v4 = *reinterpret_cast<const float4*>(&s.v[t][kC * cg]);
            const float vv[kC] = {v4.x, v4.y, v4.z, v4.w};
            float kk[kR];
            *reinterpret_cast<float4*>(&kk[0]) = *reinterpret_cast<const float4*>(&s.k[t][4 * rg]);
            *reinterpret_cast<float4*>(&kk[4]) = *reinterpret_cast<const float4*>(&s.k[t][64 + 4 * rg]);
            if (plain) {
                float aa[kR];
                *reinterpret_cast<float4*>(&aa[0]) = *reinterpret_cast<const float4*>(&s.a[t][4 * rg]);
                *reinterpret_cast<float4*>(&aa[4]) = *reinterpret_cast<const float4*>(&s.a[t][64 + 4 * rg]);
#pragma unroll
                for (int i = 0; i < kR; ++i)
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) S[i * kC + jj] = fmaf(aa[i], S[i * kC + jj], kk[i] * vv[jj]);
            } else {
#pragma unroll
                for (int i = 0; i < kR; ++i)
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) S[i * kC + jj] = fmaf(kk[i], vv[jj], S[i * kC + jj]);
            }
            if (OUT) {
                float qq[kR];
                *reinterpret_cast<float4*>(&qq[0]) = *reinterpret_cast<const float4*>(&s.q[t][4 * rg]);
                *reinterpret_cast<float4*>(&qq[4]) = *reinterpret_cast<const float4*>(&s.q[t][64 + 4 * rg]);
                float o[kC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < kR; ++i)
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) o[jj] = fmaf(qq[i], S[i * kC + jj], o[jj]);
#pragma unroll
                for (int m = 1; m < 16; m <<= 1)
#pragma unroll
                    for (int jj = 0; jj < kC; ++jj) o[jj] += __shfl_xor_sync(0xffffffffu, o[jj], m);
                if (rg == 0) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o[0] * p.scale, o[1] * p.scale);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(o[2] * p.scale, o[3] * p.scale);
                    *reinterpret_cast<__nv_bfloat162*>(&osm[t][kC * cg]) = lo;
                    *reinterpret_cast<__nv_bfloat162*>(&osm[t][kC * cg + 2]) = hi;
                }
            }
        }
        if (!plain) {
            // back from S' to S: rows scaled by exp(cum at the chunk's end)
#pragma unroll
            for (int i = 0; i < kR; ++i) {
                const float e = s.ecend[state_row(rg, i)];
#pragma unroll
                for (int jj = 0; jj < kC; ++jj) S[i * kC + jj] *= e;
            }
        }
        __syncthreads();
        if (OUT) {
            // the chunk's outputs: n tokens x 128 bf16, one 16-byte store per thread
            const int tk = tid >> 4, c8 = (tid & 15) * 8;
            if (tk < n)
                *reinterpret_cast<uint4*>(p.out + tok_row(p, b, c0 + tk, h) * kD + c8) =
                    *reinterpret_cast<const uint4*>(&osm[tk][c8]);
        }
    }
}

// State block of thread tid in a [dk][dv] fp32 array: rows state_row(rg, 0..7), columns 4 cg ..
__device__ __forceinline__ void store_state(float* dst, const float (&S)[kS]) {
    const int rg = threadIdx.x & 15, cg = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < kR; ++i)
        *reinterpret_cast<float4*>(dst + size_t(state_row(rg, i)) * kD + kC * cg) =
            make_float4(S[i * kC], S[i * kC + 1], S[i * kC + 2], S[i * kC + 3]);
}
__device__ __forceinline__ void load_state(const float* src, float (&S)[kS]) {
    const int rg = threadIdx.x & 15, cg = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < kR; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(src + size_t(state_row(rg, i)) * kD + kC * cg);
        S[i * kC] = x.x;
        S[i * kC + 1] = x.y;
        S[i * kC + 2] = x.z;
        S[i * kC + 3] = x.w;
    }
}

__global__ void __launch_bounds__(kThreads, 1) gla_segment_kernel(const __grid_constant__ LaParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Stage& st = *reinterpret_cast<Stage*>(smem_raw);
    float* gred = reinterpret_cast<float*>(smem_raw + sizeof(Stage));  // [16][128]
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    if (p.clear_status && s == 0 && h == 0 && b == 0 && threadIdx.x == 0) *p.status = 0u;
    const int t0 = s * p.L, t1 = min(p.T, (s + 1) * p.L);
    float S[kS];
#pragma unroll
    for (int i = 0; i < kS; ++i) S[i] = 0.f;
    float gsum[4] = {0.f, 0.f, 0.f, 0.f};
    run_tokens<false>(p, b, h, t0, t1, S, st, gsum, nullptr);
    const int tid = threadIdx.x;
    store_state(p.hs + ((size_t(s) * p.B + b) * p.H + h) * kD * kD, S);
    // log M_s: the 16 threads that share a channel group add their partial sums
    const int grp = tid & 31;  // channels 4 grp .. 4 grp + 3
#pragma unroll
    for (int i = 0; i < 4; ++i) gred[(tid >> 5) * kD + 4 * grp + i] = gsum[i];
    __syncthreads();
    if (tid < kD) {
        float acc = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) acc += gred[w * kD + tid];
        p.logm[((size_t(s) * p.B + b) * p.H + h) * kD + tid] = acc;
    }
}

// In place over hs: slot s goes from h_s to S_in(s).  One thread per state
// element, 256 elements per CTA; the segment loads do not depend on the chain
// and are issued 16 segments at a time, ahead of it.
__global__ void __launch_bounds__(256) gla_combine_kernel(const __grid_constant__ LaParams p) {
    const int e = blockIdx.x * 256 + threadIdx.x;   // element of the 128 x 128 state
    const int h = blockIdx.y, b = blockIdx.z;
    // Launched as a programmatic dependent of the segment pass: let the output
    // pass be scheduled, then wait for the segment pass's states.
    griddep_launch_dependents();
    griddep_wait();
    const int row = e / kD;
    const size_t stride = size_t(p.B) * p.H * kD * kD;   // between segments
    float* hp = p.hs + (size_t(b) * p.H + h) * kD * kD + e;
    const float* lm = p.logm + (size_t(b) * p.H + h) * kD + row;
    const size_t lstride = size_t(p.B) * p.H * kD;
    float acc = 0.f;   // S_in(s)
    constexpr int kU = 16;  // segments whose loads are in flight together
    for (int s0 = 0; s0 < p.N; s0 += kU) {
        float hv[kU], m[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int s = s0 + u;
            hv[u] = s < p.N - 1 ? hp[s * stride] : 0.f;
            m[u] = s < p.N - 1 ? lm[s * lstride] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int s = s0 + u;
            if (s < p.N) {
                hp[s * stride] = acc;
                acc = fmaf(__expf(m[u]), acc, hv[u]);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) gla_output_kernel(const __grid_constant__ LaParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Stage& st = *reinterpret_cast<Stage*>(smem_raw);
    auto osm = reinterpret_cast<__nv_bfloat16(*)[kD]>(smem_raw + sizeof(Stage));
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    if (p.clear_status && s == 0 && h == 0 && b == 0 && threadIdx.x == 0) *p.status = 0u;
    const int t0 = s * p.L, t1 = min(p.T, (s + 1) * p.L);
    float S[kS];
#pragma unroll
    for (int i = 0; i < kS; ++i) S[i] = 0.f;
    if (s > 0) load_state(p.hs + ((size_t(s) * p.B + b) * p.H + h) * kD * kD, S);
    float gsum[4] = {0.f, 0.f, 0.f, 0.f};
    run_tokens<true>(p, b, h, t0, t1, S, st, gsum, osm);
}

}  // namespace

size_t linear_attn_smem_segment() { return sizeof(Stage) + 16 * kD * sizeof(float); }
size_t linear_attn_smem_output() { return sizeof(Stage) + kTC * kD * sizeof(__nv_bfloat16); }

cudaError_t launch_linear_attn(const LinearAttnPlan& lp, const void* q, const void* k, const void* v,
                               const float* g, void* out, void* workspace, float scale, cudaStream_t stream) {
    LaParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.g = g;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.hs = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.hs_off);
    p.logm = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.logm_off);
    p.status = static_cast<uint32_t*>(workspace);
    p.B = lp.B; p.T = lp.T; p.H = lp.H; p.N = lp.N; p.L = lp.L;
    p.scale = scale;
    p.clear_status = 1;
    const int smem_a = int(linear_attn_smem_segment()), smem_c = int(linear_attn_smem_output());
    cudaError_t e;
    if ((e = ensure_smem_attr(reinterpret_cast<const void*>(gla_segment_kernel), smem_a)) != cudaSuccess ||
        (e = ensure_smem_attr(reinterpret_cast<const void*>(gla_output_kernel), smem_c)) != cudaSuccess)
        return e;
    if (lp.N > 1) {
        gla_segment_kernel<<<dim3(lp.N - 1, lp.H, lp.B), kThreads, smem_a, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        p.clear_status = 0;
        gla_combine_kernel<<<dim3(kD * kD / 256, lp.H, lp.B), 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    gla_output_kernel<<<dim3(lp.N, lp.H, lp.B), kThreads, smem_c, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_linear_combine(const LinearAttnPlan& lp, void* workspace, cudaStream_t stream) {
    LaParams p = {};
    p.hs = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.hs_off);
    p.logm = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lp.logm_off);
    p.B = lp.B; p.T = lp.T; p.H = lp.H; p.N = lp.N; p.L = lp.L;
    return launch_pdl(reinterpret_cast<const void*>(gla_combine_kernel), dim3(kD * kD / 256, lp.H, lp.B), dim3(256),
                      0, stream, p);
}

}  // namespace sk
