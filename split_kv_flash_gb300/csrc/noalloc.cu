// noalloc.cu -- sk_attn_fwd_noalloc: the attention forward without a caller
// workspace.  The scratch the split kernels need (status header, plan echo,
// per-split partial O and LSE) lives in one file-scope device array instead.
//
// Who needs this: code that must not call cudaMalloc/cudaFree (or any
// allocator) around the attention call -- cudaMalloc and cudaFree can
// synchronise the whole device, so latency-critical decode loops, callers that
// only own a fixed memory pool handed out by another runtime, and code paths that
// are forbidden to allocate (for example while other work is being recorded)
// cannot obtain a workspace buffer on demand.
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>
#include <string>

#include "../../include/sk_attn.h"
#include "plan.h"

namespace sk {
void set_last_error(const std::string& msg);  // api.cu: text for sk_attn_last_error()
}

namespace {

void note(const std::string& msg) { sk::set_last_error(msg); }

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(SK_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_sk_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call on
// a device resolves it (cudaGetSymbolAddress, with that device current) and
// caches it; later calls only read the cache.
sk_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        note(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
        return SK_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        note("device index out of range");
        return SK_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_sk_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            note(std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            return SK_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return SK_OK;
}

}  // namespace

extern "C" sk_status sk_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                         float* lse, int B, int Hq, int Hkv, int q_len,
                                         const int* kv_len_host, int d, float scale, int causal,
                                         int window_left, void* cuda_stream,
                                         const sk_attn_opts* opts) {
    sk_attn_plan_info info;
    sk_status s = sk_attn_plan(B, Hq, Hkv, q_len, kv_len_host, d, causal, window_left, opts, &info);
    if (s != SK_OK) return s;  // sk_attn_last_error() holds the reason
    if (info.workspace_bytes > kNoallocScratchBytes) {
        note("problem needs " + std::to_string(info.workspace_bytes) +
             " bytes of scratch; the built-in scratch holds " + std::to_string(kNoallocScratchBytes) +
             " (use sk_attn_fwd with a workspace)");
        return SK_ERR_WORKSPACE_TOO_SMALL;
    }
    void* scratch = nullptr;
    s = scratch_address(&scratch);
    if (s != SK_OK) return s;
    // The status word at the start of the header must read zero when the
    // kernels start; a previous call may have left a timeout code there.
    cudaError_t e = cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) {
        note(std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
        return SK_ERR_CUDA;
    }
    return sk_attn_fwd(q, k, v, out, lse, B, Hq, Hkv, q_len, kv_len_host, d, scale, causal,
                       window_left, scratch, kNoallocScratchBytes, cuda_stream, opts);
}

// Status of the last sk_attn_fwd_noalloc call on this device: the same word
// sk_attn_workspace_status reads from a caller workspace, here in the built-in
// scratch.  Read it before the next sk_attn_fwd_noalloc call, which clears it.
extern "C" sk_status sk_attn_noalloc_status(void* cuda_stream, int* where) {
    if (where) *where = 0;
    void* scratch = nullptr;
    sk_status s = scratch_address(&scratch);
    if (s != SK_OK) return s;
    return sk_attn_workspace_status(scratch, cuda_stream, where);
}
