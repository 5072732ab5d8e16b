/*
 * sk_attn.h -- C ABI of the split-KV flash attention forward library for
 * GB300 (sm_103a).  Library: split_kv_flash_gb300/libskattn.so.
 *
 * Operation (what every entry point below computes or plans; the latent and
 * linear-attention entry points near the end state their own):
 *   tiled attention forward with online softmax, parallelised over the KV axis
 *   (flash-decoding).  For batch b, query head h and query row i:
 *     O[b,i,h,:] = sum_j softmax_j(scale * <Q[b,i,h,:], K[off_b+j, h/G, :]>) V[off_b+j, h/G, :]
 *     LSE[b,h,i] = ln sum_j exp(scale * <Q[b,i,h,:], K[off_b+j, h/G, :]>)
 *   over the visible keys j of row i.
 *   Sources: FlashAttention tiling strategy and scheduling chapter (分块策略与调度),
 *   section 1 (tiling), section 3 (block-level masking skip), section 5 (split-K /
 *   flash decoding with a separate combine step), section 6 (PackGQA); "The Occupancy
 *   Awakening" (KV-split partial kernel plus reduction kernel); llama.cpp PR #21086
 *   review (the stream-k fixup that merges partial tiles).
 *
 * Conventions shared by all entry points
 *   - G = Hq / Hkv; query head h reads KV head h / G (contiguous groups).
 *   - Q   [B, q_len, Hq, d]  bf16, row-major, device memory.
 *   - K,V [sum_b kv_len[b], Hkv, d] bf16, row-major, device memory, packed by
 *         sequence: sequence b starts at row off_b = kv_len[0] + ... + kv_len[b-1].
 *         For equal lengths this is [B, kv_len, Hkv, d].
 *   - O   [B, q_len, Hq, d]  bf16 output;  LSE [B, Hq, q_len] fp32 output (natural log).
 *   - kv_len_host: HOST array of B non-negative lengths (read during the call only).
 *   - causal != 0: query i sees keys j <= i + kv_len - q_len (bottom-right aligned,
 *     tiling chapter section 3.1).  window_left >= 0: query i also needs
 *     j >= i + kv_len - q_len - window_left (inclusive).  window_left < 0: no left
 *     bound.  With causal == 0 a window bounds the left side only.
 *   - A row with no visible key returns O = 0 and LSE = -inf.
 *   - Supported: bf16 only, d in {64, 128}, Hq % Hkv == 0, q/k/v/out 16-byte
 *     aligned, lse 4-byte aligned, workspace 256-byte aligned.  Anything else is
 *     rejected with an error; there is no fallback path.
 *   - Ownership: the caller owns every buffer.  The library allocates no device
 *     memory and keeps no per-call state.  Inputs are never written.
 *   - Errors are returned before any launch; no output is partly written by a
 *     call that returns an error.  sk_attn_last_error() gives a one-line reason.
 *   - Rows outside a sequence never affect its result.  The 128-row block that
 *     holds the end of a sequence also holds the first rows of the next one:
 *     their scores are masked and their V rows are zeroed in shared memory
 *     before they are multiplied, so Inf or NaN there cannot leak in.
 */
#ifndef SK_ATTN_H
#define SK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SK_OK = 0,
    SK_ERR_INVALID_ARG = 1,          /* a size, pointer or flag is out of range */
    SK_ERR_UNSUPPORTED = 2,          /* valid attention, but outside the supported domain */
    SK_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < sk_attn_plan_info.workspace_bytes */
    SK_ERR_MISALIGNED = 4,           /* a pointer violates the alignment rules above */
    SK_ERR_CUDA = 5,                 /* a CUDA runtime/driver call failed */
    SK_ERR_DEVICE_TIMEOUT = 6        /* a kernel gave up on a bounded wait (see sk_attn_workspace_status) */
} sk_status;

/* How the number of KV splits is chosen (sk_attn_opts.policy). */
typedef enum {
    SK_POLICY_DEFAULT = 0,      /* = SK_POLICY_FILL */
    SK_POLICY_FILL = 1,         /* smallest per-CTA KV chunk such that all CTAs fit in one wave */
    SK_POLICY_FA_HEURISTIC = 2, /* num_splits_heuristic, tiling chapter section 5.2 */
    SK_POLICY_FIXED_CHUNK = 3,  /* clamp(ceil(kv_len / 2048), 1, 32), "The Occupancy Awakening" */
    SK_POLICY_MIN_CHUNK = 4     /* 2 blocks per SM, each >= 256 keys, llama.cpp PR #21086 review */
} sk_split_policy;

/* Which kernel runs the partial (split) pass (sk_attn_opts.force_path / plan_info.path). */
typedef enum {
    SK_PATH_AUTO = 0,
    SK_PATH_DECODE = 1,   /* <= 64 packed query rows per tile: KV rows on the MMA M axis */
    SK_PATH_PREFILL = 2,  /* 256-row tiles: two 128-row halves that share each K/V block; query rows on the MMA M axis */
    SK_PATH_LATENT = 3,   /* latent attention (sk_attn_fwd_latent only): 16 or 32 packed rows per tile, keys on the MMA M axis */
    SK_PATH_LINEAR_RECURRENT = 4, /* linear attention: the segments run token by token on the FMA pipes */
    SK_PATH_LINEAR_CHUNK = 5      /* linear attention: the segments run in windows of <= 128 tokens as four
                                     128 x 128 x 128 tensor-core products each (the default) */
} sk_path;

/* How the split partials are merged (sk_attn_opts.combine_mode; the stream-k
 * fixup of the llama.cpp PR #21086 review, the combine step of the tiling
 * chapter section 5.1). */
typedef enum {
    SK_COMBINE_AUTO = 0,      /* the library chooses (currently SK_COMBINE_KERNEL, the faster one) */
    SK_COMBINE_KERNEL = 1,    /* a second kernel merges every split row */
    SK_COMBINE_IN_KERNEL = 2  /* one launch: the last split CTA of a tile to finish merges the
                                 tile's partials (decode path, when they fit its shared memory;
                                 otherwise the second kernel is used) */
} sk_combine_mode;

/* How the prefill kernel's CTAs take tiles (sk_attn_opts.prefill_schedule;
 * tiling chapter section 4.2 single-tile and section 4.4 dynamic persistent
 * schedulers). */
typedef enum {
    SK_SCHEDULE_AUTO = 0,        /* the library chooses (currently one CTA per tile, measured faster) */
    SK_SCHEDULE_ONE_TILE = 1,    /* one CTA per tile */
    SK_SCHEDULE_PERSISTENT = 2   /* one CTA per SM, tiles from an atomic counter, longest first,
                                    in L2 sections of heads; needs Q rows that are whole groups of
                                    the 128-row TMA box (128 % heads per group == 0), else one tile
                                    per CTA */
} sk_prefill_schedule;

/* How the decode kernel's grid maps to tiles when the sequences of a batch have
 * different split counts (sk_attn_opts.tile_map; tiling chapter section 4.5,
 * the varlen scheduler's warp prefix sum over per-sequence tile counts). */
typedef enum {
    SK_TILE_MAP_AUTO = 0,    /* the library chooses (currently the grid) */
    SK_TILE_MAP_GRID = 1,    /* grid (m blocks, head tiles x grid splits, sequences); a CTA whose
                                split index is past its sequence's split count exits at once */
    SK_TILE_MAP_PACKED = 2   /* one-dimensional grid over the CTAs that have work, in the grid's
                                order without the empty ones: sequence b owns head_tiles x
                                splits_b x num_m_blocks consecutive CTAs, and each CTA finds its
                                sequence by a warp prefix sum over the split counts.  Decode path,
                                batches of more than one sequence with different split counts */
} sk_tile_map;

/* Options; an all-zero struct (or NULL) selects the defaults. */
typedef struct {
    int policy;            /* sk_split_policy */
    int force_num_splits;  /* > 0: exactly this many splits (clipped to the KV block count) */
    int force_pack_gqa;    /* 0: should_pack_gqa heuristic; 1: pack; -1: do not pack */
    int force_path;        /* sk_path */
    int max_splits;        /* 0: 128 */
    int num_sms;           /* 0: the current device's SM count; > 0: plan for this many SMs */
    int debug_echo_plan;   /* 1: each CTA writes its KV block range into the workspace */
    int wait_timeout_us;   /* 0: 2,000,000 us; bound on every device-side wait */
    int debug_inject_stall;/* 1: one kernel wait targets a barrier nothing signals (tests the
                              timeout path; the kernel reports SK_ERR_DEVICE_TIMEOUT) */
    void* event_begin;     /* optional cudaEvent_t recorded just before the partial kernel */
    void* event_end;       /* optional cudaEvent_t recorded just after it */
    int combine_mode;      /* sk_combine_mode */
    int prefill_schedule;  /* sk_prefill_schedule */
    int tile_map;          /* sk_tile_map */
} sk_attn_opts;

/* The host scheduler's decisions for one problem. */
typedef struct {
    int path;                 /* sk_path actually used */
    int kBlockM;              /* packed query rows per tile */
    int kBlockN;              /* keys per KV block */
    int pack_gqa;             /* 1: the G query heads of a KV head share one tile */
    int head_tiles;           /* Hkv if pack_gqa else Hq */
    int rows_per_head_tile;   /* q_len * G if pack_gqa else q_len */
    int num_m_blocks;         /* ceil(rows_per_head_tile / kBlockM) */
    int num_splits;           /* grid splits = max over sequences of the per-sequence count */
    int num_splits_policy;    /* the count the policy chose before per-sequence sizing */
    int num_n_blocks_max;     /* ceil(max kv_len / kBlockN) */
    int grid_x, grid_y, grid_z; /* partial kernel grid: (num_m_blocks, head_tiles*num_splits, B), or
                                   (num_ctas, 1, 1) with the packed tile map */
    long long num_ctas;       /* grid_x * grid_y * grid_z */
    int needs_combine;        /* 1: some sequence has more than one split */
    size_t workspace_bytes;   /* bytes of device workspace sk_attn_fwd needs */
    size_t echo_offset;       /* byte offset of the plan echo in the workspace */
    size_t lse_part_offset;   /* byte offset of LSE partials [S][B][Hq][q_len] fp32 */
    size_t o_part_offset;     /* byte offset of O partials [S][B][Hq][q_len][d] fp32 (d_v wide for latent) */
    int combine_in_kernel;    /* 1: the partial kernel merges the splits itself (no second launch) */
    size_t counter_offset;    /* byte offset of the counters: per-tile arrivals (in-kernel merge) or
                                 the persistent scheduler's next-tile and finished-CTA counts */
    int persistent;           /* 1: the prefill kernel runs persistent CTAs */
    int persistent_ctas;      /* CTAs of the persistent launch (<= SM count) */
    int l2_section_heads;     /* head tiles per L2 section of the persistent tile order */
    int tile_map;             /* SK_TILE_MAP_GRID or SK_TILE_MAP_PACKED (then grid = (num_ctas, 1, 1)
                                 and the plan echo lists only the CTAs that have work) */
} sk_attn_plan_info;

/* Plan only (host, no device work).  Fills *info.  Same argument meaning as
 * sk_attn_fwd.  With opts->num_sms > 0 it needs no GPU. */
sk_status sk_attn_plan(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d,
                       int causal, int window_left, const sk_attn_opts* opts,
                       sk_attn_plan_info* info);

/* The host plan's KV block range of every CTA of the partial kernel, in launch
 * order (x fastest, then y, then z): 4 int32 per CTA = {n_block_min, n_block_max,
 * split word (low 16 bits split index, high 16 bits the sequence's split count),
 * 1 if the CTA has work else 0}.  n_int32 must be >= 4 * num_ctas.  Tiling chapter
 * sections 3.2 and 5.3. */
sk_status sk_attn_plan_ranges(int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d,
                              int causal, int window_left, const sk_attn_opts* opts,
                              int32_t* ranges_host, size_t n_int32);

/* Attention forward.  Asynchronous on cuda_stream (a cudaStream_t; NULL = legacy
 * default stream).  workspace: device buffer of >= info.workspace_bytes bytes,
 * 256-byte aligned, zero-filled once before its first use (every call leaves its
 * status word at zero unless a kernel timed out); it may be reused by consecutive
 * calls on the same stream, but calls that overlap on the GPU need separate
 * workspaces.  After a call that reported SK_ERR_DEVICE_TIMEOUT the workspace
 * must be zero-filled again before its next use.  Returns SK_OK once the
 * kernels are enqueued. */
sk_status sk_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d,
                      float scale, int causal, int window_left,
                      void* workspace, size_t ws_bytes, void* cuda_stream,
                      const sk_attn_opts* opts);

/* Latent attention (absorbed multi-head latent attention, MLA): "The Occupancy
 * Awakening", the verify attention of a speculative-decoding engine for Kimi
 * K2.6, whose absorbed KV representation is one latent head of Dl = 512 columns
 * plus Dr = 64 rotary columns shared by every query head.  For batch b, query
 * head h and query row i:
 *     s_j          = scale * <Q[b,i,h,0:576], KV[off_b+j, 0:576]>
 *     O[b,i,h,:]   = sum_j softmax_j(s_j) KV[off_b+j, 0:512]
 *     LSE[b,h,i]   = ln sum_j exp(s_j)
 * over the visible keys j of row i (causal / window rules as above; the verify
 * workload is q_len = drafts + 1 rows at the end of a prefix, causal).
 *   - q   [B, q_len, Hq, d_qk] bf16;  kv [sum_b kv_len[b], d_qk] bf16, packed by
 *         sequence like K above (the values are the first d_v columns of each row,
 *         read in place);  out [B, q_len, Hq, d_v] bf16;  lse [B, Hq, q_len] fp32.
 *   - Supported: d_qk = 576 and d_v = 512 only, any Hq >= 1; the alignment,
 *     workspace, ownership and error rules of sk_attn_fwd.  The query heads are
 *     packed into the tiles (PackGQA with one KV head); opts.force_path,
 *     force_pack_gqa, combine_mode and prefill_schedule are ignored.
 *   - The plan reports path SK_PATH_LATENT; the O partials in the workspace are
 *     d_v wide. */
sk_status sk_attn_plan_latent(int B, int Hq, int q_len, const int* kv_len_host, int d_qk, int d_v,
                              int causal, int window_left, const sk_attn_opts* opts,
                              sk_attn_plan_info* info);
sk_status sk_attn_fwd_latent(const void* q, const void* kv, void* out, float* lse,
                             int B, int Hq, int q_len, const int* kv_len_host, int d_qk, int d_v,
                             float scale, int causal, int window_left,
                             void* workspace, size_t ws_bytes, void* cuda_stream,
                             const sk_attn_opts* opts);

/* Chunk-parallel linear attention (inclusionAI/cuLA issue #11: each (sequence,
 * head) is split along T into N segments that run in parallel and are merged
 * by an affine combine (M, h_ext)).  The issue does not print the recurrence;
 * this library computes gated linear attention with one decay per key channel,
 * for every sequence b and head h:
 *     S_0 = 0,  S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T  (dk x dv, fp32)
 *     o_t = scale * S_t^T q_t
 * A segment started from S_in ends at M S_in + h_ext with M = Diag(exp(sum of g
 * over the segment)) and h_ext its end state from a zero start; segment s covers
 * tokens [s L, min((s + 1) L, T)), L = ceil(T / N).
 *   - q, k [B, T, H, dk] bf16;  v [B, T, H, dv] bf16;  g [B, T, H, dk] fp32 log
 *     decays (<= 0);  out [B, T, H, dv] bf16.  dk = dv = 128 only.
 *   - num_segments: 0 = one wave of SMs over the (segment, head, sequence) CTAs
 *     with at least 64 tokens per segment (128 on the chunk path); > 0 = that
 *     many (at most T).
 *   - opts->force_path: SK_PATH_LINEAR_CHUNK (also for SK_PATH_AUTO) runs each
 *     segment in windows of at most 128 tokens on the tensor cores: inside a
 *     window the state, the intra-window scores and the outputs are dense
 *     products (bf16 operands, fp32 accumulation, the state kept in fp32); a
 *     window ends before a key channel's summed log decay would span more than
 *     60, and log decays are clamped to [-100, 100].  SK_PATH_LINEAR_RECURRENT
 *     runs the recurrence token by token in fp32 on the FMA pipes.  Other values
 *     are SK_ERR_INVALID_ARG.
 *   - workspace: >= info.workspace_bytes, 256-byte aligned, caller-owned (the
 *     segments' h_ext / incoming states and log M); q, k, v, g, out 16-byte
 *     aligned.  Same error rules as sk_attn_fwd.  The chunk path's device waits
 *     are bounded by opts->wait_timeout_us; one that gives up leaves its code in
 *     the workspace's status word (sk_attn_workspace_status).  On both paths the
 *     call's first kernel clears that word, so the workspace needs no zero fill
 *     (the token-by-token path has no bounded wait and leaves it at zero).  The
 *     state is never returned. */
typedef struct {
    int num_segments;        /* N actually used */
    int segment_len;         /* L */
    size_t workspace_bytes;
    int launches;            /* 1 (N = 1) or 3 (segment pass, combine, output pass) */
    int path;                /* SK_PATH_LINEAR_CHUNK or SK_PATH_LINEAR_RECURRENT */
} sk_linear_attn_info;

sk_status sk_linear_attn_plan(int B, int T, int H, int dk, int dv, int num_segments,
                              const sk_attn_opts* opts, sk_linear_attn_info* info);
sk_status sk_linear_attn_fwd(const void* q, const void* k, const void* v, const float* g, void* out,
                             int B, int T, int H, int dk, int dv, float scale, int num_segments,
                             void* workspace, size_t ws_bytes, void* cuda_stream,
                             const sk_attn_opts* opts);

/* Copy n_int32 int32 of the plan echo (written when opts.debug_echo_plan = 1;
 * same layout as sk_attn_plan_ranges) to host memory.  Synchronises cuda_stream. */
sk_status sk_attn_read_plan_echo(const void* workspace, int32_t* ranges_host, size_t n_int32,
                                 void* cuda_stream);

/* Synchronise cuda_stream and read the workspace's device status word.  Returns
 * SK_OK, or SK_ERR_DEVICE_TIMEOUT when a kernel gave up on a bounded wait since
 * the last check (the word is then cleared).  *where (optional) receives the code
 * of the wait that expired. */
sk_status sk_attn_workspace_status(void* workspace, void* cuda_stream, int* where);

/* Attention forward for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for this
 * library's users.  Code that must not call cudaMalloc / cudaFree (they can
 * synchronise the device, so hot decode loops avoid them; some callers only
 * own memory handed out by another runtime's pool) has no way to obtain the
 * workspace that sk_attn_fwd wants.  This variant takes no workspace: the split
 * kernels use one scratch array compiled into the library, of
 * SK_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads the library (held until
 * the process exits).  It allocates no device memory and calls no allocating
 * routine.
 *   - Arguments, layouts, results and errors are those of sk_attn_fwd.
 *   - A problem whose plan needs more than SK_NOALLOC_SCRATCH_BYTES of workspace
 *     (sk_attn_plan_info.workspace_bytes) is rejected with
 *     SK_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - The first call on each device looks up the scratch array's device address
 *     (with that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the one array and it keeps the previous call's contents;
 *     the call clears the status header it needs at zero (an asynchronous memset
 *     on cuda_stream) before the kernels.  Calls whose work overlaps on the GPU
 *     (different streams, or several host threads without ordering) race on the
 *     scratch and give wrong results: order them on one stream.
 *   - A kernel that gives up on a bounded wait leaves its code in the built-in
 *     scratch; read it with sk_attn_noalloc_status before the next call on the
 *     device (which clears it).
 *   - The cached address belongs to the device's current context: after
 *     cudaDeviceReset the library must be reloaded before this entry point is
 *     used again. */
#define SK_NOALLOC_SCRATCH_BYTES (16u << 20)
sk_status sk_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int Hq, int Hkv, int q_len, const int* kv_len_host, int d,
                              float scale, int causal, int window_left, void* cuda_stream,
                              const sk_attn_opts* opts);

/* sk_attn_workspace_status for the built-in scratch of sk_attn_fwd_noalloc on
 * the current device: synchronises cuda_stream, returns SK_OK or
 * SK_ERR_DEVICE_TIMEOUT (then clears the word; *where, optional, receives the
 * code of the wait that expired).  The pages have no counterpart to this entry
 * point either; it lets callers of sk_attn_fwd_noalloc see device timeouts. */
sk_status sk_attn_noalloc_status(void* cuda_stream, int* where);

const char* sk_attn_status_string(sk_status s);
/* One-line reason for the last error returned on this thread ("" if none). */
const char* sk_attn_last_error(void);
/* Library ABI version: 100 * major + minor. */
int sk_attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SK_ATTN_H */
