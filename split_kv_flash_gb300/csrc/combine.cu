// combine.cu -- merges the per-split partial results (the stream-k fixup of the
// llama.cpp PR #21086 review; the separate combine kernel of the FlashAttention
// tiling chapter, section 5.1; the reduction kernel of "The Occupancy Awakening").
//
// For every output row with S_b > 1 splits holding (O_s, LSE_s):
//   M   = max_s LSE_s
//   LSE = M + ln sum_s exp(LSE_s - M)
//   O   = sum_s exp(LSE_s - LSE) * O_s         -> bf16
// All partials at -inf: O = 0, LSE = -inf.
//
// Two shapes of the same merge:
//  - many splits (S > 16; long-context decode: few rows, up to 128 splits):
//    one CTA of 8 warps per output row.  The row's partials are spread over
//    the warps (warp w takes splits w, w + 8, ...) and loaded together with
//    the LSEs, so a 64- or 128-wide row costs about one L2 round trip (a
//    512-wide row one per 32 splits);
//  - few splits (S <= 16; verify, batched decode: many rows, few splits): one
//    warp per row, 8 rows per CTA, lane s holding split s's LSE and lane c the
//    float4 columns c, c + 32, ... of the row, so a CTA is not launched for a
//    few loads.  The partials of up to 16 splits (8 or 4 for 64- or 512-wide
//    rows) are loaded at once, next to the LSEs: one L2 round trip.
// Rows are 64, 128 or 512 values wide (512: latent attention).
// Both are launched as programmatic dependents of the partial kernel: they are
// scheduled while the partial kernel runs and wait (griddepcontrol.wait) for
// that grid's completion and memory before they read anything.
#include <math.h>

#include "fwd_common.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634074f;

template <int HD, class Seqs>
__global__ void __launch_bounds__(32 * kWarps)
    combine_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ Seqs seqs) {
    constexpr int kCols4 = HD / 4;          // float4 columns of a row: 16, 32 or 128
    constexpr int kPer = (kCols4 + 31) / 32;  // per lane
    __shared__ float w_s[kMaxSplits];       // merge weight of each split
    __shared__ float4 part[kWarps][32 * kPer];  // per-warp partial sums
    __shared__ float lse_row;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long row = blockIdx.x;
    const int b = int(row / ((long long)p.Hq * p.sq));
    const int rem = int(row - (long long)b * p.Hq * p.sq);
    const int h = rem / p.sq;
    const int i = rem - h * p.sq;
    const int S = seqs.splits_of(b);
    griddep_launch_dependents();  // the next call's partial kernel may start its prologue
    griddep_wait();
    if (S <= 1) return;  // written directly by the partial kernel
    const size_t stride = (size_t)p.B * p.Hq * p.sq;  // between splits of one row
    const size_t base = ((size_t)b * p.Hq + h) * p.sq + i;

    // Warp w takes splits w, w + 8, ...; lane c the float4 columns c, c + 32, ...
    // A round loads kRound splits a warp (16 float4 a lane); the first round is
    // issued before the LSE phase so that both loads are in flight together.
    constexpr int kRound = 16 / kPer;
    const float4* src0 = reinterpret_cast<const float4*>(p.o_part + base * HD);
    const size_t stride4 = stride * (HD / 4);
    float4 v[kRound][kPer];
    auto load_round = [&](int r) {
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            const int s = warp + (r * kRound + u) * kWarps;
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int c = t * 32 + lane;
                v[u][t] = (s < S && c < kCols4) ? __ldcg(src0 + c + s * stride4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    load_round(0);

    // 1. log-sum-exp over the splits (warp 0), weights into shared memory.
    if (warp == 0) {
        float l[kMaxSplits / 32];
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t) {
            const int s = t * 32 + lane;
            l[t] = (s < S) ? __ldcg(p.lse_part + s * stride + base) : -INFINITY;
            mx = fmaxf(mx, l[t]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t)
            sum += (l[t] == -INFINITY) ? 0.f : exp2f((l[t] - mx) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float lse = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t) {
            const int s = t * 32 + lane;
            if (s < S) w_s[s] = (l[t] == -INFINITY || lse == -INFINITY) ? 0.f : exp2f((l[t] - lse) * kLog2e);
        }
        if (lane == 0) lse_row = lse;
    }
    __syncthreads();

    // 2. weighted sum of this warp's splits, then across the warps.
    float4 acc[kPer];
#pragma unroll
    for (int t = 0; t < kPer; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int rounds = (S + kWarps * kRound - 1) / (kWarps * kRound);
    for (int r = 0; r < rounds; ++r) {
        if (r > 0) load_round(r);
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            const int s = warp + (r * kRound + u) * kWarps;
            const float ws = (s < S) ? w_s[s] : 0.f;
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                acc[t].x += ws * v[u][t].x;
                acc[t].y += ws * v[u][t].y;
                acc[t].z += ws * v[u][t].z;
                acc[t].w += ws * v[u][t].w;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kPer; ++t) part[warp][t * 32 + lane] = acc[t];
    __syncthreads();
    for (int c = threadIdx.x; c < kCols4; c += 32 * kWarps) {
        float4 t = part[0][c];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            const float4 u = part[w][c];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        uint2 packed;
        __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p.out + (((size_t)b * p.sq + i) * p.Hq + h) * HD + c * 4) = packed;
    }
    if (threadIdx.x == 0) p.lse[base] = lse_row;
}

constexpr int kRowsMaxSplits = 16;  // the warp-per-row shape handles up to this many splits

template <int HD, class Seqs>
__global__ void __launch_bounds__(32 * kWarps)
    combine_rows_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ Seqs seqs, long long rows) {
    constexpr int kCols4 = HD / 4;
    constexpr int kPer = (kCols4 + 31) / 32;
    // splits loaded together: at most 16 float4 a lane (8 for 64-wide rows, whose upper lanes idle)
    constexpr int kBatch = kPer == 1 ? (HD >= 128 ? kRowsMaxSplits : 8) : 4;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + warp;
    griddep_launch_dependents();  // the next call's partial kernel may start its prologue
    griddep_wait();
    if (row >= rows) return;
    const int b = int(row / ((long long)p.Hq * p.sq));
    const int rem = int(row - (long long)b * p.Hq * p.sq);
    const int h = rem / p.sq;
    const int i = rem - h * p.sq;
    const int S = seqs.splits_of(b);
    if (S <= 1) return;  // written directly by the partial kernel
    const size_t stride = (size_t)p.B * p.Hq * p.sq;  // between splits of one row
    const size_t base = ((size_t)b * p.Hq + h) * p.sq + i;

    // lane s holds split s's LSE; lane c the float4 columns c, c + 32, ... of
    // every split's O partial.  The O loads of kBatch splits are issued together,
    // the first batch next to the LSE load, so a row with S <= kBatch costs one
    // L2 round trip.
    const float l = (lane < S) ? __ldcg(p.lse_part + lane * stride + base) : -INFINITY;
    const float4* src = reinterpret_cast<const float4*>(p.o_part + base * HD) + lane;
    const size_t stride4 = stride * (HD / 4);
    float4 v[kBatch][kPer];
    auto load_batch = [&](int s0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
            for (int t = 0; t < kPer; ++t)
                v[u][t] = (s0 + u < S && t * 32 + lane < kCols4) ? __ldcg(src + t * 32 + (s0 + u) * stride4)
                                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load_batch(0);

    // log-sum-exp over the splits
    float mx = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = (l == -INFINITY) ? 0.f : exp2f((l - mx) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float lse = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    const float w = (l == -INFINITY || lse == -INFINITY) ? 0.f : exp2f((l - lse) * kLog2e);

    // weighted sum of the O partials (lanes >= S carry weight 0)
    float4 acc[kPer];
#pragma unroll
    for (int t = 0; t < kPer; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0;;) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float ws = __shfl_sync(0xffffffffu, w, s0 + u);
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                acc[t].x += ws * v[u][t].x;
                acc[t].y += ws * v[u][t].y;
                acc[t].z += ws * v[u][t].z;
                acc[t].w += ws * v[u][t].w;
            }
        }
        s0 += kBatch;
        if (s0 >= S) break;
        load_batch(s0);
    }
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
        const int c = t * 32 + lane;
        if (c < kCols4) {
            uint2 packed;
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[t].x, acc[t].y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[t].z, acc[t].w);
            packed.x = *reinterpret_cast<uint32_t*>(&lo);
            packed.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(p.out + (((size_t)b * p.sq + i) * p.Hq + h) * HD + c * 4) = packed;
        }
    }
    if (lane == 0) p.lse[base] = lse;
}

template <int HD, class Seqs>
cudaError_t launch_c(const Plan& plan, const FwdParams& p, const Seqs& seqs, cudaStream_t stream) {
    const long long rows = (long long)plan.B * plan.Hq * plan.sq;
    if (rows <= 0) return cudaSuccess;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (plan.num_splits <= kRowsMaxSplits) {
        cfg.gridDim = dim3(unsigned((rows + kWarps - 1) / kWarps));
        return cudaLaunchKernelEx(&cfg, combine_rows_kernel<HD, Seqs>, p, seqs, rows);
    }
    cfg.gridDim = dim3(unsigned(rows));
    return cudaLaunchKernelEx(&cfg, combine_kernel<HD, Seqs>, p, seqs);
}

}  // namespace

template <class Seqs>
cudaError_t launch_width(const Plan& plan, const FwdParams& p, const Seqs& seqs, cudaStream_t stream) {
    switch (plan.dv) {
        case 64: return launch_c<64>(plan, p, seqs, stream);
        case 128: return launch_c<128>(plan, p, seqs, stream);
        case 512: return launch_c<512>(plan, p, seqs, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const Plan& plan, const FwdParams& p, cudaStream_t stream) {
    if (plan.num_splits > kMaxSplits) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return launch_width(plan, p, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    return launch_width(plan, p, v, stream);
}

}  // namespace sk
