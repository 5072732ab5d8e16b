// fwd_common.cuh -- parameters shared by the partial (split) kernels and the
// combine kernel, and the launch entry points implemented in the .cu files.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "block_range.h"
#include "plan.h"

namespace sk {

// Status-word codes: (kernel << 8) | wait site.
enum : uint32_t {
    kKernDecode = 1,
    kKernPrefill = 2,
    kSiteProducerEmpty = 1,
    kSiteMmaQ = 2,
    kSiteMmaFull = 3,
    kSiteMmaSEmpty = 4,
    kSiteMmaPFull = 5,
    kSiteSoftmaxSFull = 6,
    kSiteSoftmaxODone = 7,
    kSiteInjected = 8,
    kSiteSmemAlign = 9,
    kSiteMerge = 10,
};

struct FwdParams {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    float* lse;
    float* o_part;     // [S][B][Hq][sq][d]
    float* lse_part;   // [S][B][Hq][sq]
    int32_t* echo;     // 4 int32 per CTA
    uint32_t* counters;  // per tile: split CTAs that have written their partial (in-kernel merge)
    uint32_t* status;  // workspace header word
    int B, Hq, Hkv, G, sq, d;
    int pack_gqa;
    int rows;          // packed rows per head tile
    int kBlockM, kBlockN, num_m_blocks, num_splits, head_tiles;
    KeyWindow win;     // which keys a row sees (block ranges)
    int causal;        // element-level mask
    int window_left;   // < 0: none
    float scale_log2;  // softmax scale * log2(e)
    int reverse_m;
    int echo_plan;
    int inject_stall;
    unsigned long long timeout_ns;
    int q_tma;         // prefill: Q halves arrive by TMA through the 4-D Q map
    int q_gp;          // query heads per row group of that map (G with PackGQA, else 1)
    int o_tma;         // prefill: final O halves leave by TMA through the 5-D O map
    int fused_combine; // decode: the last split CTA of a tile merges the tile's partials
    int packed_grid;   // decode, varlen: 1-D grid over the CTAs with work (packed_tile_of_cta)
};

// Per-sequence lengths, offsets and split counts.  Equal lengths need no table.
struct UniformSeqs {
    int len;
    int splits;
    __device__ __forceinline__ int seq_len(int) const { return len; }
    __device__ __forceinline__ int seq_off(int b) const { return b * len; }
    __device__ __forceinline__ int splits_of(int) const { return splits; }
};

struct VarlenSeqs {
    int off[kMaxVarlenBatch + 1];
    unsigned short splits[kMaxVarlenBatch];
    __device__ __forceinline__ int seq_len(int b) const { return off[b + 1] - off[b]; }
    __device__ __forceinline__ int seq_off(int b) const { return off[b]; }
    __device__ __forceinline__ int splits_of(int b) const { return splits[b]; }
};

// Packed tile map (tiling chapter section 4.5: the varlen scheduler finds a
// tile's sequence by a warp prefix sum over the sequences' tile counts).  The
// grid is one-dimensional over the CTAs that have work, in the order of the
// rectangular grid without its empty CTAs: sequence b owns head_tiles x
// splits_b x num_m_blocks consecutive CTAs (head tile, then split, then m
// block fastest).  Called by whole warps; every lane returns the same tile.
template <class Seqs>
__device__ __forceinline__ TileCoord packed_tile_of_cta(int cta, const FwdParams& p, const Seqs& seqs) {
    const int lane = threadIdx.x & 31;
    const int unit = p.head_tiles * p.num_m_blocks;  // CTAs per split of one sequence
    const int slot = cta / unit;                      // the CTA's split slot over all sequences
    const int chunk = (p.B + 31) >> 5;                // sequences per lane
    const int b0 = min(lane * chunk, p.B), b1 = min(b0 + chunk, p.B);
    int mine = 0;
    for (int b = b0; b < b1; ++b) mine += seqs.splits_of(b);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int excl = incl - mine;
    const unsigned hit = __ballot_sync(0xffffffffu, slot >= excl && slot < incl);
    const int src = hit ? __ffs(hit) - 1 : 31;
    int base = __shfl_sync(0xffffffffu, excl, src);
    int b = min(src * chunk, p.B - 1);
    while (b < p.B - 1 && base + seqs.splits_of(b) <= slot) base += seqs.splits_of(b++);
    const int sb = max(seqs.splits_of(b), 1);
    const int l = cta - base * unit;  // index inside sequence b
    const int bx = l % p.num_m_blocks;
    const int rest = l / p.num_m_blocks;
    TileCoord t;
    t.m_block = p.reverse_m ? p.num_m_blocks - 1 - bx : bx;
    t.split = rest % sb;
    t.head_tile = rest / sb;
    t.batch = b;
    return t;
}

// Packed row r of head tile ht -> (query position i, query head h).
// Tiling chapter section 6.1/6.3: with PackGQA the G query heads of KV head ht
// share the tile, row r = i * G + g.
struct RowMap {
    int i, h;
};
__device__ __forceinline__ RowMap map_row(const FwdParams& p, int ht, int r) {
    RowMap m;
    if (p.pack_gqa) {
        m.i = r / p.G;
        m.h = ht * p.G + (r - m.i * p.G);
    } else {
        m.i = r;
        m.h = ht;
    }
    return m;
}

// Launchers (return a CUDA error code).
cudaError_t launch_decode(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t stream);
cudaError_t launch_prefill(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, const CUtensorMap& tmQ, const CUtensorMap& tmO,
                           cudaStream_t stream);
cudaError_t launch_prefill_persistent(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, const CUtensorMap& tmQ, cudaStream_t stream);
// tmK: latent rows as 3-D boxes of kLatentKChunksPerCopy 64-column chunks;
// tmV: the same rows as boxes of 2 chunks (one 128-column value group);
// tmQ: query rows as boxes of (64 columns, kBlockM rows, 3 chunks).
cudaError_t launch_latent(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmQ, cudaStream_t stream);
cudaError_t launch_combine(const Plan& plan, const FwdParams& p, cudaStream_t stream);

void fill_varlen(const Plan& plan, VarlenSeqs* v);

// Launch a kernel as a programmatic dependent of the previous work on the
// stream: it may be scheduled while that work drains and waits for it
// (griddepcontrol.wait) before touching global memory.  `args` are the kernel's
// parameters in order.
template <class... A>
cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, int smem, cudaStream_t stream, const A&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* ptrs[] = {const_cast<void*>(static_cast<const void*>(&args))...};
    return cudaLaunchKernelExC(&cfg, kernel, ptrs);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

}  // namespace sk
