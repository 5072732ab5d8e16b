// api.cu -- the C ABI declared in include/sk_attn.h: argument checks, the host
// plan, TMA tensor maps for K and V, and the launches of the partial kernel and
// the combine kernel on the caller's stream (standard and latent attention).
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "../../include/sk_attn.h"
#include "fwd_common.cuh"
#include "linear_attn.h"
#include "plan.h"

namespace sk {

namespace {

thread_local std::string g_last_error;

sk_status fail(sk_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

sk_status fail_cuda(cudaError_t e, const char* what) {
    return fail(SK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// K or V as a 2-D bf16 tensor [rows][Hkv * d]; boxes of 128 rows x 64 columns
// (128 bytes, the swizzle width), 128-byte swizzle, zero fill past the end.
bool make_kv_map(CUtensorMap* m, const void* base, int Hkv, int d, long long rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(Hkv) * cuuint64_t(d), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(Hkv) * cuuint64_t(d) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Latent rows [rows][576] as a 3-D bf16 tensor (64 columns, rows, 9 column
// chunks): the chunk dimension has a 128-byte stride, so a box of
// (64, 128, z) is z consecutive 64-column chunks of 128 rows, laid out in
// shared memory chunk after chunk, each [128 rows][128 bytes] with the
// 128-byte swizzle.  One copy then moves z x 16 KB (larger copies stream
// faster than 16 KB ones).
bool make_latent_map(CUtensorMap* m, const void* base, long long rows, int z, int box_rows = 128) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, cuuint64_t(rows), cuuint64_t(kLatentDqk / 64)};
    cuuint64_t strides[2] = {cuuint64_t(kLatentDqk) * 2, 128};
    cuuint32_t box[3] = {64, cuuint32_t(box_rows), cuuint32_t(z)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Q [B * q_len][Hq][d] as a 4-D bf16 tensor (d, gp, Hq / gp, B * q_len): a box
// of (64, gp, 1, 128 / gp) is 128 rows of 128 bytes in packed-row order
// (query position major, the gp query heads of a group minor), 128-byte
// swizzle, zero fill past the end.
bool make_q_map(CUtensorMap* m, const void* q, long long rows, int Hq, int d, int gp) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(gp), cuuint64_t(Hq / gp), cuuint64_t(rows)};
    cuuint64_t strides[3] = {cuuint64_t(d) * 2, cuuint64_t(gp) * cuuint64_t(d) * 2, cuuint64_t(Hq) * cuuint64_t(d) * 2};
    cuuint32_t box[4] = {64, cuuint32_t(gp), 1, cuuint32_t(128 / gp)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// O [B][q_len][Hq][d] as a 5-D bf16 tensor (d, gp, Hq / gp, q_len, B): the same
// packed-row boxes as the Q map, with the sequence as its own dimension so that
// a store clips the rows past q_len instead of writing into the next sequence.
bool make_o_map(CUtensorMap* m, void* o, int B, int q_len, int Hq, int d, int gp) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[5] = {cuuint64_t(d), cuuint64_t(gp), cuuint64_t(Hq / gp), cuuint64_t(q_len), cuuint64_t(B)};
    const cuuint64_t row = cuuint64_t(Hq) * cuuint64_t(d) * 2;
    cuuint64_t strides[4] = {cuuint64_t(d) * 2, cuuint64_t(gp) * cuuint64_t(d) * 2, row, row * cuuint64_t(q_len)};
    cuuint32_t box[5] = {64, cuuint32_t(gp), 1, cuuint32_t(128 / gp), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, o, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Log decays g [rows][H * 128] fp32 as a 2-D tensor; boxes of 128 rows x 128
// columns (512 bytes) without swizzle, row-major in shared memory.
bool make_g_map(CUtensorMap* m, const float* base, int H, long long rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(H) * kLinearAttnDim, cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(H) * kLinearAttnDim * 4};
    cuuint32_t box[2] = {kLinearAttnDim, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct DeviceInfo {
    int dev = 0, sms = 0, major = 0, minor = 0;
};

sk_status current_device(DeviceInfo* di) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && have[dev]) {
        *di = cache[dev];
        return SK_OK;
    }
    DeviceInfo d;
    d.dev = dev;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return fail_cuda(e, "cudaDeviceGetAttribute");
    if (dev >= 0 && dev < 64) {
        cache[dev] = d;
        have[dev] = true;
    }
    *di = d;
    return SK_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- per-thread cache of plans and tensor maps
struct CallKey {
    int dev, B, Hq, Hkv, q_len, d, dv, latent, causal, window_left;
    int policy, force_num_splits, force_pack_gqa, force_path, max_splits, num_sms, combine_mode, prefill_schedule;
    int tile_map;
    const void *q, *k, *v, *out;
};

struct CallEntry {
    CallKey key;
    Plan plan;  // plan.kv_len holds the lengths the entry was made for
    CUtensorMap tmK, tmV, tmQ, tmO;
    bool q_tma = false, o_tma = false;
    int q_gp = 1;
};

constexpr int kCallCacheSize = 64;

struct CallCache {
    CallEntry entries[kCallCacheSize];
    bool used[kCallCacheSize] = {};
    int next = 0;   // round-robin replacement
    int last = -1;  // most recent hit or insert, checked first
};

thread_local CallCache g_calls;

bool same_call(const CallEntry& e, const CallKey& k, const int* kv_len) {
    if (memcmp(&e.key, &k, sizeof k) != 0) return false;
    return memcmp(e.plan.kv_len.data(), kv_len, sizeof(int) * size_t(k.B)) == 0;
}

const CallEntry* lookup_call(const CallKey& k, const int* kv_len) {
    CallCache& c = g_calls;
    if (k.B <= 0) return nullptr;
    if (c.last >= 0 && c.used[c.last] && same_call(c.entries[c.last], k, kv_len)) return &c.entries[c.last];
    for (int i = 0; i < kCallCacheSize; ++i)
        if (c.used[i] && same_call(c.entries[i], k, kv_len)) {
            c.last = i;
            return &c.entries[i];
        }
    return nullptr;
}

const CallEntry* insert_call(const CallKey& k, CallEntry&& e) {
    CallCache& c = g_calls;
    const int i = c.next;
    c.next = (c.next + 1) % kCallCacheSize;
    c.entries[i] = std::move(e);
    c.entries[i].key = k;
    c.used[i] = true;
    c.last = i;
    return &c.entries[i];
}

}  // namespace

void set_last_error(const std::string& msg) { g_last_error = msg; }

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({kernel, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({kernel, dev});
    return e;
}

}  // namespace sk

using namespace sk;

extern "C" {

sk_status sk_attn_plan(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int causal,
                       int window_left, const sk_attn_opts* opts, sk_attn_plan_info* info) {
    g_last_error.clear();
    if (!info) return fail(SK_ERR_INVALID_ARG, "info is NULL");
    int sms = 0;
    if (!opts || opts->num_sms <= 0) {
        DeviceInfo di;
        sk_status s = current_device(&di);
        if (s != SK_OK) return s;
        sms = di.sms;
    }
    Plan p;
    std::string why;
    sk_status s = make_plan(B, Hq, Hkv, q_len, kv_len_host, d, causal, window_left, opts, sms, &p, &why);
    if (s != SK_OK) return fail(s, why);
    plan_to_info(p, info);
    return SK_OK;
}

sk_status sk_attn_plan_ranges(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d, int causal,
                              int window_left, const sk_attn_opts* opts, int32_t* ranges_host,
                              size_t n_int32) {
    g_last_error.clear();
    if (!ranges_host) return fail(SK_ERR_INVALID_ARG, "ranges_host is NULL");
    int sms = 0;
    if (!opts || opts->num_sms <= 0) {
        DeviceInfo di;
        sk_status s = current_device(&di);
        if (s != SK_OK) return s;
        sms = di.sms;
    }
    Plan p;
    std::string why;
    sk_status s = make_plan(B, Hq, Hkv, q_len, kv_len_host, d, causal, window_left, opts, sms, &p, &why);
    if (s != SK_OK) return fail(s, why);
    if (n_int32 < size_t(p.num_ctas) * 4) return fail(SK_ERR_INVALID_ARG, "ranges_host too small");
    plan_ranges(p, ranges_host);
    return SK_OK;
}

}  // extern "C"

namespace {

// Both forward entry points.  Latent attention: one KV head (Hkv = 1) of width
// d whose rows are the keys and whose first dv columns are the values (k == v).
sk_status fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                   int q_len, const int* kv_len_host, int d, int dv, bool latent, float scale, int causal,
                   int window_left, void* workspace, size_t ws_bytes, void* cuda_stream, const sk_attn_opts* opts) {
    sk_attn_opts o;
    memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    if (!(scale > 0.f) || !isfinite(scale)) return fail(SK_ERR_INVALID_ARG, "scale must be finite and > 0");
    DeviceInfo di;
    sk_status s = current_device(&di);
    if (s != SK_OK) return s;
    if (!(di.major == 10 && di.minor == 3))
        return fail(SK_ERR_UNSUPPORTED, "this library runs on sm_103 (GB300) only");
    // The plan and the tensor maps depend only on the problem, the options and
    // the q / k / v / out addresses: a decode loop that repeats a call reuses
    // them from the per-thread cache instead of planning and encoding again.
    CallKey key;
    memset(&key, 0, sizeof key);
    key.dev = di.dev; key.B = B; key.Hq = Hq; key.Hkv = Hkv; key.q_len = q_len; key.d = d;
    key.dv = dv; key.latent = latent ? 1 : 0;
    key.causal = causal ? 1 : 0; key.window_left = window_left < 0 ? -1 : window_left;
    key.policy = o.policy; key.force_num_splits = o.force_num_splits; key.force_pack_gqa = o.force_pack_gqa;
    key.force_path = o.force_path; key.max_splits = o.max_splits; key.num_sms = o.num_sms;
    key.combine_mode = o.combine_mode;
    key.prefill_schedule = o.prefill_schedule;
    key.tile_map = o.tile_map;
    key.q = q; key.k = k; key.v = v; key.out = out;
    const CallEntry* ce = kv_len_host ? lookup_call(key, kv_len_host) : nullptr;
    if (!ce) {
        CallEntry fresh;
        std::string why;
        s = latent ? make_plan_latent(B, Hq, q_len, kv_len_host, d, dv, causal, window_left, &o, di.sms,
                                      &fresh.plan, &why)
                   : make_plan(B, Hq, Hkv, q_len, kv_len_host, d, causal, window_left, &o, di.sms, &fresh.plan,
                               &why);
        if (s != SK_OK) return fail(s, why);
        const Plan& p = fresh.plan;
        if (p.num_ctas == 0) return SK_OK;  // q_len == 0: nothing to compute
        const long long total_kv = p.kv_off[size_t(B)];
        if (!q || !out) return fail(SK_ERR_INVALID_ARG, "NULL q, out, lse or workspace");
        if (total_kv > 0 && (!k || !v)) return fail(SK_ERR_INVALID_ARG, "NULL k or v");
        if (!aligned(q, 16) || !aligned(out, 16) || (total_kv > 0 && (!aligned(k, 16) || !aligned(v, 16))))
            return fail(SK_ERR_MISALIGNED, "q, k, v and out must be 16-byte aligned");
        if (total_kv >= (1LL << 31)) return fail(SK_ERR_UNSUPPORTED, "at most 2^31 - 1 KV rows in total");
        // K/V tensor maps.  With no KV rows at all no tile is ever loaded; the
        // map then points at `out` only so that it is well formed.
        const void* kb = total_kv > 0 ? k : out;
        const void* vb = total_kv > 0 ? v : out;
        const long long rows = total_kv > 0 ? total_kv : 1;
        if (latent) {
            // K: three 64-column chunks per copy; V: one 128-column group per copy.
            if (!make_latent_map(&fresh.tmK, kb, rows, kLatentKChunksPerCopy) ||
                !make_latent_map(&fresh.tmV, vb, rows, 2))
                return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (latent)");
        } else if (!make_kv_map(&fresh.tmK, kb, Hkv, d, rows) || !make_kv_map(&fresh.tmV, vb, Hkv, d, rows)) {
            return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        }
        // Prefill tiles take Q by TMA when a 128-row half is whole row groups of
        // the map (128 % gp == 0) and every row index fits the copy's int32
        // coordinate.  Final prefill outputs (one split per sequence) leave
        // through the same boxes.
        memset(&fresh.tmQ, 0, sizeof fresh.tmQ);
        memset(&fresh.tmO, 0, sizeof fresh.tmO);
        fresh.q_gp = p.pack_gqa ? p.G : 1;
        const long long q_rows = (long long)B * q_len;
        fresh.q_tma = p.path == SK_PATH_PREFILL && 128 % fresh.q_gp == 0 && q_rows < (1LL << 31);
        if (fresh.q_tma && !make_q_map(&fresh.tmQ, q, q_rows, Hq, d, fresh.q_gp))
            return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (Q)");
        if (latent) {
            // Q rows [B * q_len * Hq][576]: a tile's packed rows are consecutive
            // rows of this tensor, so its Q^T arrives as three boxes of
            // (64, kBlockM, 3).
            const long long rows_q = (long long)B * q_len * Hq;
            if (rows_q >= (1LL << 31)) return fail(SK_ERR_UNSUPPORTED, "latent: B * q_len * Hq must be < 2^31");
            if (!make_latent_map(&fresh.tmQ, q, rows_q, 3, p.kBlockM))
                return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (latent Q)");
        }
        fresh.o_tma = fresh.q_tma && !p.needs_combine && !p.persistent;
        if (fresh.o_tma && !make_o_map(&fresh.tmO, out, B, q_len, Hq, d, fresh.q_gp))
            return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (O)");
        ce = insert_call(key, std::move(fresh));
    }
    const Plan& p = ce->plan;
    if (!q || !out || !lse || !workspace) return fail(SK_ERR_INVALID_ARG, "NULL q, out, lse or workspace");
    if (!aligned(lse, 4)) return fail(SK_ERR_MISALIGNED, "lse must be 4-byte aligned");
    if (!aligned(workspace, 256)) return fail(SK_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (ws_bytes < p.ws_bytes) return fail(SK_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than plan.workspace_bytes");
    const CUtensorMap& tmK = ce->tmK;
    const CUtensorMap& tmV = ce->tmV;
    const CUtensorMap& tmQ = ce->tmQ;
    const CUtensorMap& tmO = ce->tmO;
    const bool q_tma = ce->q_tma, o_tma = ce->o_tma;
    const int q_gp = ce->q_gp;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    FwdParams fp;
    memset(&fp, 0, sizeof fp);
    fp.q = static_cast<const __nv_bfloat16*>(q);
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.o_part = reinterpret_cast<float*>(ws + p.o_off);
    fp.lse_part = reinterpret_cast<float*>(ws + p.lse_off);
    fp.echo = reinterpret_cast<int32_t*>(ws + p.echo_off);
    fp.counters = reinterpret_cast<uint32_t*>(ws + p.cnt_off);
    fp.fused_combine = p.fused_combine ? 1 : 0;

    fp.status = reinterpret_cast<uint32_t*>(ws);
    fp.B = B; fp.Hq = Hq; fp.Hkv = p.Hkv; fp.G = p.G; fp.sq = q_len; fp.d = d;
    fp.pack_gqa = p.pack_gqa ? 1 : 0;
    fp.rows = p.rows;
    fp.kBlockM = p.kBlockM; fp.kBlockN = p.kBlockN;
    fp.num_m_blocks = p.num_m_blocks; fp.num_splits = p.num_splits; fp.head_tiles = p.head_tiles;
    fp.win = p.win;
    fp.causal = p.causal;
    fp.window_left = p.window_left;
    fp.scale_log2 = float(double(scale) * 1.4426950408889634074);
    fp.reverse_m = p.reverse_m ? 1 : 0;
    fp.echo_plan = o.debug_echo_plan ? 1 : 0;
    fp.inject_stall = o.debug_inject_stall ? 1 : 0;
    fp.timeout_ns = (unsigned long long)(o.wait_timeout_us > 0 ? o.wait_timeout_us : 2000000) * 1000ull;
    fp.q_tma = q_tma ? 1 : 0;
    fp.q_gp = q_gp;
    fp.o_tma = o_tma ? 1 : 0;
    fp.packed_grid = p.packed_grid ? 1 : 0;

    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e;
    if (o.event_begin && (e = cudaEventRecord(static_cast<cudaEvent_t>(o.event_begin), stream)) != cudaSuccess)
        return fail_cuda(e, "cudaEventRecord");
    if (p.path == SK_PATH_LATENT)
        e = launch_latent(p, fp, tmK, tmV, tmQ, stream);
    else if (p.path == SK_PATH_DECODE)
        e = launch_decode(p, fp, tmK, tmV, stream);
    else if (p.persistent && q_tma)
        e = launch_prefill_persistent(p, fp, tmK, tmV, tmQ, stream);
    else
        e = launch_prefill(p, fp, tmK, tmV, tmQ, tmO, stream);
    if (e != cudaSuccess) return fail_cuda(e, "partial kernel launch");
    if (o.event_end && (e = cudaEventRecord(static_cast<cudaEvent_t>(o.event_end), stream)) != cudaSuccess)
        return fail_cuda(e, "cudaEventRecord");
    if (p.needs_combine && !p.fused_combine) {
        e = launch_combine(p, fp, stream);
        if (e != cudaSuccess) return fail_cuda(e, "combine kernel launch");
    }
    return SK_OK;
}

}  // namespace

extern "C" {

sk_status sk_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                      int Hkv, int q_len, const int* kv_len_host, int d, float scale, int causal,
                      int window_left, void* workspace, size_t ws_bytes, void* cuda_stream,
                      const sk_attn_opts* opts) {
    g_last_error.clear();
    return fwd_impl(q, k, v, out, lse, B, Hq, Hkv, q_len, kv_len_host, d, d, false, scale, causal, window_left,
                    workspace, ws_bytes, cuda_stream, opts);
}

sk_status sk_attn_plan_latent(int B, int Hq, int q_len, const int* kv_len_host, int d_qk, int d_v, int causal,
                              int window_left, const sk_attn_opts* opts, sk_attn_plan_info* info) {
    g_last_error.clear();
    if (!info) return fail(SK_ERR_INVALID_ARG, "info is NULL");
    int sms = 0;
    if (!opts || opts->num_sms <= 0) {
        DeviceInfo di;
        sk_status s = current_device(&di);
        if (s != SK_OK) return s;
        sms = di.sms;
    }
    Plan p;
    std::string why;
    sk_status s = make_plan_latent(B, Hq, q_len, kv_len_host, d_qk, d_v, causal, window_left, opts, sms, &p, &why);
    if (s != SK_OK) return fail(s, why);
    plan_to_info(p, info);
    return SK_OK;
}

sk_status sk_attn_fwd_latent(const void* q, const void* kv, void* out, float* lse, int B, int Hq, int q_len,
                             const int* kv_len_host, int d_qk, int d_v, float scale, int causal, int window_left,
                             void* workspace, size_t ws_bytes, void* cuda_stream, const sk_attn_opts* opts) {
    g_last_error.clear();
    return fwd_impl(q, kv, kv, out, lse, B, Hq, 1, q_len, kv_len_host, d_qk, d_v, true, scale, causal,
                    window_left, workspace, ws_bytes, cuda_stream, opts);
}

namespace {
sk_status linear_plan(int B, int T, int H, int dk, int dv, int num_segments, const sk_attn_opts* opts,
                      sk::LinearAttnPlan* lp, int* path) {
    if (dk != kLinearAttnDim || dv != kLinearAttnDim)
        return fail(SK_ERR_UNSUPPORTED, "linear attention: dk = dv = 128 only");
    if (B <= 0 || H <= 0 || T < 0 || num_segments < 0) return fail(SK_ERR_INVALID_ARG, "bad B, H, T or segments");
    if ((long long)B * T * H >= (1LL << 31)) return fail(SK_ERR_UNSUPPORTED, "B * T * H must be < 2^31");
    const int fp = opts ? opts->force_path : SK_PATH_AUTO;
    if (fp != SK_PATH_AUTO && fp != SK_PATH_LINEAR_CHUNK && fp != SK_PATH_LINEAR_RECURRENT)
        return fail(SK_ERR_INVALID_ARG, "linear attention: force_path must be AUTO, LINEAR_CHUNK or LINEAR_RECURRENT");
    *path = fp == SK_PATH_LINEAR_RECURRENT ? int(SK_PATH_LINEAR_RECURRENT) : int(SK_PATH_LINEAR_CHUNK);
    int sms = opts && opts->num_sms > 0 ? opts->num_sms : 0;
    if (sms == 0) {
        DeviceInfo di;
        sk_status s = current_device(&di);
        if (s != SK_OK) return s;
        sms = di.sms;
    }
    make_linear_attn_plan(B, T, H, num_segments, sms, lp,
                          *path == SK_PATH_LINEAR_CHUNK ? kLinearAttnMinSegmentChunk : kLinearAttnMinSegment);
    return SK_OK;
}
}  // namespace

sk_status sk_linear_attn_plan(int B, int T, int H, int dk, int dv, int num_segments, const sk_attn_opts* opts,
                              sk_linear_attn_info* info) {
    g_last_error.clear();
    if (!info) return fail(SK_ERR_INVALID_ARG, "info is NULL");
    sk::LinearAttnPlan lp;
    int path = 0;
    sk_status s = linear_plan(B, T, H, dk, dv, num_segments, opts, &lp, &path);
    if (s != SK_OK) return s;
    memset(info, 0, sizeof *info);
    info->num_segments = lp.N;
    info->segment_len = lp.L;
    info->workspace_bytes = lp.ws_bytes;
    info->launches = lp.N > 1 ? 3 : 1;
    info->path = path;
    return SK_OK;
}

sk_status sk_linear_attn_fwd(const void* q, const void* k, const void* v, const float* g, void* out, int B, int T,
                             int H, int dk, int dv, float scale, int num_segments, void* workspace, size_t ws_bytes,
                             void* cuda_stream, const sk_attn_opts* opts) {
    g_last_error.clear();
    if (!isfinite(scale)) return fail(SK_ERR_INVALID_ARG, "scale must be finite");
    DeviceInfo di;
    sk_status s = current_device(&di);
    if (s != SK_OK) return s;
    if (!(di.major == 10 && di.minor == 3))
        return fail(SK_ERR_UNSUPPORTED, "this library runs on sm_103 (GB300) only");
    sk::LinearAttnPlan lp;
    int path = 0;
    s = linear_plan(B, T, H, dk, dv, num_segments, opts, &lp, &path);
    if (s != SK_OK) return s;
    if (T == 0) return SK_OK;
    if (!q || !k || !v || !g || !out || !workspace) return fail(SK_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(out, 16))
        return fail(SK_ERR_MISALIGNED, "q, k, v, g and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(SK_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (ws_bytes < lp.ws_bytes) return fail(SK_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than info.workspace_bytes");
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e;
    if (opts && opts->event_begin &&
        (e = cudaEventRecord(static_cast<cudaEvent_t>(opts->event_begin), stream)) != cudaSuccess)
        return fail_cuda(e, "cudaEventRecord");
    if (path == SK_PATH_LINEAR_CHUNK) {
        const uint64_t timeout_ns =
            uint64_t(opts && opts->wait_timeout_us > 0 ? opts->wait_timeout_us : 2000000) * 1000ull;
        CUtensorMap tmQ, tmK, tmV, tmG;
        const long long rows = (long long)B * T;
        if (!make_kv_map(&tmQ, q, H, kLinearAttnDim, rows) || !make_kv_map(&tmK, k, H, kLinearAttnDim, rows) ||
            !make_kv_map(&tmV, v, H, kLinearAttnDim, rows) || !make_g_map(&tmG, g, H, rows))
            return fail(SK_ERR_CUDA, "cuTensorMapEncodeTiled failed (linear attention)");
        e = launch_linear_attn_tc(lp, tmQ, tmK, tmV, tmG, q, k, v, g, out, workspace, scale, timeout_ns,
                                  opts ? opts->debug_inject_stall : 0, stream);
    } else {
        e = launch_linear_attn(lp, q, k, v, g, out, workspace, scale, stream);
    }
    if (e != cudaSuccess) return fail_cuda(e, "linear attention launch");
    if (opts && opts->event_end &&
        (e = cudaEventRecord(static_cast<cudaEvent_t>(opts->event_end), stream)) != cudaSuccess)
        return fail_cuda(e, "cudaEventRecord");
    return SK_OK;
}

sk_status sk_attn_read_plan_echo(const void* workspace, int32_t* ranges_host, size_t n_int32, void* cuda_stream) {
    g_last_error.clear();
    if (!workspace || !ranges_host) return fail(SK_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    e = cudaMemcpy(ranges_host, static_cast<const uint8_t*>(workspace) + 256, n_int32 * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpy");
    return SK_OK;
}

sk_status sk_attn_workspace_status(void* workspace, void* cuda_stream, int* where) {
    g_last_error.clear();
    if (where) *where = 0;
    if (!workspace) return fail(SK_ERR_INVALID_ARG, "NULL workspace");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpy(&word, workspace, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpy");
    if (word == 0) return SK_OK;
    if (where) *where = int(word);
    e = cudaMemset(workspace, 0, 4);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemset");
    return fail(SK_ERR_DEVICE_TIMEOUT, "a kernel gave up on a bounded wait (code " + std::to_string(word) + ")");
}

const char* sk_attn_status_string(sk_status s) {
    switch (s) {
        case SK_OK: return "SK_OK";
        case SK_ERR_INVALID_ARG: return "SK_ERR_INVALID_ARG";
        case SK_ERR_UNSUPPORTED: return "SK_ERR_UNSUPPORTED";
        case SK_ERR_WORKSPACE_TOO_SMALL: return "SK_ERR_WORKSPACE_TOO_SMALL";
        case SK_ERR_MISALIGNED: return "SK_ERR_MISALIGNED";
        case SK_ERR_CUDA: return "SK_ERR_CUDA";
        case SK_ERR_DEVICE_TIMEOUT: return "SK_ERR_DEVICE_TIMEOUT";
    }
    return "SK_ERR_UNKNOWN";
}

const char* sk_attn_last_error(void) { return g_last_error.c_str(); }

int sk_attn_version(void) { return 104; }

}  // extern "C"
