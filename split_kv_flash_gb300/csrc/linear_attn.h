// linear_attn.h -- host plan and launcher of the chunk-parallel gated linear
// attention (linear_attn.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sk {

constexpr int kLinearAttnDim = 128;        // dk = dv
constexpr int kLinearAttnMinSegment = 64;        // tokens per segment when the count is chosen (recurrent)
constexpr int kLinearAttnMinSegmentChunk = 128;  // the same for the tensor-core windows

struct LinearAttnPlan {
    int B = 0, T = 0, H = 0;
    int N = 1;  // segments per (sequence, head)
    int L = 0;  // tokens per segment (the last may be shorter)
    size_t hs_off = 0, logm_off = 0, ws_bytes = 256;
};

// Segments: n_req > 0 asks for that many (at most T); 0 fills one wave of SMs
// with (segment, head, sequence) CTAs while every segment keeps at least
// min_segment tokens.  Empty trailing segments are dropped.
inline void make_linear_attn_plan(int B, int T, int H, int n_req, int sms, LinearAttnPlan* p,
                                  int min_segment = kLinearAttnMinSegment) {
    p->B = B;
    p->T = T;
    p->H = H;
    long long n = n_req;
    if (n <= 0) {
        const long long bh = (long long)B * H;
        n = bh >= sms ? 1 : sms / bh;
        const long long by_len = (T + min_segment - 1) / min_segment;
        if (n > by_len) n = by_len;
    }
    if (n > T) n = T;
    if (n < 1) n = 1;
    p->L = T > 0 ? int((T + n - 1) / n) : 0;
    p->N = p->L > 0 ? (T + p->L - 1) / p->L : 1;
    const size_t per = size_t(p->N) * B * H;
    p->hs_off = 256;
    p->logm_off = p->hs_off + (p->N > 1 ? per * kLinearAttnDim * kLinearAttnDim * 4 : 0);
    p->ws_bytes = p->logm_off + (p->N > 1 ? ((per * kLinearAttnDim * 4 + 255) / 256) * 256 : 0);
}

size_t linear_attn_smem_segment();
size_t linear_attn_smem_output();
size_t linear_attn_tc_smem();
// Token-by-token passes on the FMA pipes (linear_attn.cu).
cudaError_t launch_linear_attn(const LinearAttnPlan& lp, const void* q, const void* k, const void* v,
                               const float* g, void* out, void* workspace, float scale, cudaStream_t stream);
// Window passes on the tensor cores (linear_attn_tc.cu); bounded waits report
// through the workspace's status word.
// q, k, v also come as 2-D maps [B * T][H * 128] (boxes of 128 rows x 64 columns,
// 128-byte swizzle) and g as a 2-D fp32 map of the same shape (boxes of 128 x 128,
// no swizzle) for the window copies.
cudaError_t launch_linear_attn_tc(const LinearAttnPlan& lp, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, const CUtensorMap& tmG, const void* q, const void* k,
                                  const void* v,
                                  const float* g, void* out, void* workspace, float scale, uint64_t timeout_ns,
                                  int inject_stall, cudaStream_t stream);
// The affine combine over the segments' (log M, h) in the workspace (both paths).
cudaError_t launch_linear_combine(const LinearAttnPlan& lp, void* workspace, cudaStream_t stream);

}  // namespace sk
