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
// One CTA of 8 warps per output row.  The row's partials are spread over the
// warps (warp w takes splits w, w + 8, ...), so every load of the row is in
// flight at once and the merge costs about one L2 round trip; lane c holds the
// float4 columns c (and c + 32 when d = 256 ...) of the row.  The kernel is
// launched as a programmatic dependent of the partial kernel: it is scheduled
// while the partial kernel runs and waits (griddepcontrol.wait) for that
// grid's completion and memory before it reads anything.
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
    constexpr int kCols4 = HD / 4;       // float4 columns of a row: 32 (d=128) or 16 (d=64)
    __shared__ float w_s[kMaxSplits];    // merge weight of each split
    __shared__ float4 part[kWarps][32];  // per-warp partial sums
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

    // 2. weighted sum of the O partials, splits spread over the warps.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < kCols4) {
        const float4* src = reinterpret_cast<const float4*>(p.o_part + base * HD) + lane;
        const size_t stride4 = stride * (HD / 4);
        constexpr int kUnroll = kMaxSplits / kWarps;  // 16
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int s = warp + u * kWarps;
            v[u] = (s < S) ? __ldcg(src + s * stride4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int s = warp + u * kWarps;
            const float ws = (s < S) ? w_s[s] : 0.f;
            acc.x += ws * v[u].x;
            acc.y += ws * v[u].y;
            acc.z += ws * v[u].z;
            acc.w += ws * v[u].w;
        }
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && lane < kCols4) {
        float4 t = part[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            const float4 u = part[w][lane];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        uint2 packed;
        __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p.out + (((size_t)b * p.sq + i) * p.Hq + h) * HD + lane * 4) = packed;
        if (lane == 0) p.lse[base] = lse_row;
    }
}

template <int HD, class Seqs>
cudaError_t launch_c(const Plan& plan, const FwdParams& p, const Seqs& seqs, cudaStream_t stream) {
    const long long rows = (long long)plan.B * plan.Hq * plan.sq;
    if (rows <= 0) return cudaSuccess;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(rows));
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<HD, Seqs>, p, seqs);
}

}  // namespace

cudaError_t launch_combine(const Plan& plan, const FwdParams& p, cudaStream_t stream) {
    if (plan.num_splits > kMaxSplits) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return plan.d == 128 ? launch_c<128>(plan, p, u, stream) : launch_c<64>(plan, p, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    return plan.d == 128 ? launch_c<128>(plan, p, v, stream) : launch_c<64>(plan, p, v, stream);
}

}  // namespace sk
