// combine.cu -- merges the per-split partial results (the stream-k fixup of the
// llama.cpp PR #21086 review; the separate combine kernel of the FlashAttention
// tiling chapter, section 5.1; the reduction kernel of "The Occupancy Awakening").
//
// For every output row with S_b > 1 splits holding (O_s, LSE_s):
//   M   = max_s LSE_s
//   LSE = M + ln sum_s exp(LSE_s - M)
//   O   = sum_s exp(LSE_s - LSE) * O_s         -> bf16
// All partials at -inf: O = 0, LSE = -inf.  One warp per row; lane c holds
// d / 32 consecutive output columns.
#include <math.h>

#include "fwd_common.cuh"

namespace sk {
namespace {

constexpr int kRowsPerBlock = 8;
constexpr int kMaxSplitRegs = 4;  // 4 x 32 lanes = up to 128 splits
constexpr float kLog2e = 1.4426950408889634074f;

template <int HD, class Seqs>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    combine_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ Seqs seqs) {
    constexpr int kPer = HD / 32;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const long long rows = (long long)p.B * p.Hq * p.sq;
    if (row >= rows) return;
    const int b = int(row / ((long long)p.Hq * p.sq));
    const int rem = int(row - (long long)b * p.Hq * p.sq);
    const int h = rem / p.sq;
    const int i = rem - h * p.sq;
    const int S = seqs.splits_of(b);
    if (S <= 1) return;  // written directly by the partial kernel
    const size_t stride = (size_t)p.B * p.Hq * p.sq;  // between splits of one row
    const size_t base = ((size_t)b * p.Hq + h) * p.sq + i;

    float lse_s[kMaxSplitRegs];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < kMaxSplitRegs; ++t) {
        const int s = t * 32 + lane;
        lse_s[t] = (s < S) ? __ldg(p.lse_part + s * stride + base) : -INFINITY;
        mx = fmaxf(mx, lse_s[t]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
    float lse_out = -INFINITY;
    if (mx != -INFINITY) {
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxSplitRegs; ++t)
            sum += (lse_s[t] == -INFINITY) ? 0.f : exp2f((lse_s[t] - mx) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        lse_out = mx + logf(sum);
        float w[kMaxSplitRegs];
#pragma unroll
        for (int t = 0; t < kMaxSplitRegs; ++t)
            w[t] = (lse_s[t] == -INFINITY) ? 0.f : exp2f((lse_s[t] - lse_out) * kLog2e);
        const float* src = p.o_part + base * HD + lane * kPer;
#pragma unroll
        for (int t = 0; t < kMaxSplitRegs; ++t) {
            if (t * 32 >= S) break;
            const int n = min(32, S - t * 32);
#pragma unroll 4
            for (int s2 = 0; s2 < n; ++s2) {
                const float ws = __shfl_sync(0xffffffffu, w[t], s2);
                if (ws == 0.f) continue;
                const float* sp = src + (size_t)(t * 32 + s2) * stride * HD;
                if constexpr (kPer == 4) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(sp));
                    acc[0] += ws * v.x; acc[1] += ws * v.y; acc[2] += ws * v.z; acc[3] += ws * v.w;
                } else {
                    const float2 v = __ldg(reinterpret_cast<const float2*>(sp));
                    acc[0] += ws * v.x; acc[1] += ws * v.y;
                }
            }
        }
    }
    __nv_bfloat16* dst = p.out + (((size_t)b * p.sq + i) * p.Hq + h) * HD + lane * kPer;
#pragma unroll
    for (int c = 0; c < kPer; ++c) dst[c] = __float2bfloat16_rn(acc[c]);
    if (lane == 0) p.lse[base] = lse_out;
}

template <int HD, class Seqs>
cudaError_t launch_c(const Plan& plan, const FwdParams& p, const Seqs& seqs, cudaStream_t stream) {
    const long long rows = (long long)plan.B * plan.Hq * plan.sq;
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    combine_kernel<HD, Seqs><<<dim3(unsigned(blocks)), 32 * kRowsPerBlock, 0, stream>>>(p, seqs);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const Plan& plan, const FwdParams& p, cudaStream_t stream) {
    if (plan.num_splits > 32 * kMaxSplitRegs) return cudaErrorInvalidValue;
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return plan.d == 128 ? launch_c<128>(plan, p, u, stream) : launch_c<64>(plan, p, u, stream);
    }
    VarlenSeqs v;
    fill_varlen(plan, &v);
    return plan.d == 128 ? launch_c<128>(plan, p, v, stream) : launch_c<64>(plan, p, v, stream);
}

}  // namespace sk
