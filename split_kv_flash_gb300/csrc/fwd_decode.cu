// fwd_decode.cu -- split-KV partial kernel for tiles of at most 64 packed query
// rows (decode, speculative verify, GQA decode), sm_103a.
//
// One CTA owns (KV head tile, split, sequence).  The KV block range comes from
// the block-range rules of the FlashAttention tiling chapter (section 3.2: causal /
// local bounds; section 5.3: the split's share of the range).  Because the query
// side is small, the MMAs put the 128 KV rows of a block on the tensor-core M
// axis and the packed query rows on N ("swap AB"):
//   S^T[128 keys x NP] = K_blk[128 x d] . Q^T              (tcgen05, TMEM)
//   O^T[d x NP]       += V_blk^T[d x 128] . P^T[128 x NP]   (tcgen05, TMEM)
// Online softmax (running max m, running sum l, fp32 accumulator) follows the
// flash-decode description of "The Occupancy Awakening"; each split writes its
// normalised partial O and log-sum-exp for the combine kernel, or the final
// output when the sequence has a single split.
//
// Warp roles (192 threads): warp 0 issues the TMA loads of K and V blocks into
// two multi-stage shared-memory rings; warp 1 owns TMEM and issues the MMAs;
// warps 2-5 (128 threads, thread t <-> TMEM lane t = key t of S^T and d-row t
// of O^T) do the softmax, the rescaling and the epilogue.
#include <math.h>

#include "fwd_common.cuh"
#include "kv_producer.cuh"
#include "sm103_ptx.cuh"

namespace sk {
namespace {

constexpr int kThreads = 192;  // producer, MMA, 4 softmax warps
constexpr int kDecodeL2Warm = 3;  // K and V blocks of a range prefetched into L2 before the grid dependency
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Maximum over the 32 lanes of a converged warp, one instruction
// (redux.sync on f32; NaN inputs are not expected here).
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int HD, int NP>
struct DecodeCfg {
    // Ring depths: the next QK^T waits on a K block, so K gets the deeper ring;
    // V has a softmax pass of slack.  Each (HD, NP) takes what shared memory allows.
    static constexpr int kStagesK = decode_stages_k(HD, NP);
    static constexpr int kStagesV = decode_stages_v(HD, NP);
    static constexpr int kKBytes = 128 * HD * 2;      // K block: 128 rows x HD
    static constexpr int kVBytes = 128 * 128 * 2;     // V block region: 128 rows x 128 (M = 128 for PV)
    static constexpr int kVLoadBytes = 128 * HD * 2;  // bytes actually loaded
    static constexpr int kQBytes = NP * HD * 2;
    static constexpr int kPBuf = NP * 128 * 2;             // one P^T buffer
    static constexpr int kPBufs = decode_p_bufs(HD, NP);
    static constexpr int kPBytes = kPBufs * kPBuf;
    static constexpr int kOffK = 0;                        // K ring: kStagesK slots
    static constexpr int kOffV = kStagesK * kKBytes;       // V ring: kStagesV slots
    static constexpr int kOffQ = kOffV + kStagesV * kVBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffRed = kOffP + kPBytes;            // float red[4][NP]
    static constexpr int kOffM = kOffRed + 4 * NP * 4;         // float m[NP]
    static constexpr int kOffAlpha = kOffM + NP * 4;           // float alpha[NP]
    static constexpr int kOffL = kOffAlpha + NP * 4;           // float l[NP]
    static constexpr int kOffDiag = kOffL + NP * 4;            // int diag[NP]
    static constexpr int kOffBars = (kOffDiag + NP * 4 + 7) / 8 * 8;
    static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 1;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;   // tmem base, abort flag, merge flag
    static constexpr int kRingBytes = kStagesK * kKBytes + kStagesV * kVBytes;
    static_assert(kRingBytes == decode_ring_bytes(HD, NP), "ring geometry shared with the scheduler");
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;       // slack to align the base to 1024
    static constexpr int kTmemCols = (3 * NP <= 32) ? 32 : (3 * NP <= 64) ? 64 : (3 * NP <= 128) ? 128 : 256;
    static_assert(kSmemAlloc <= 232448, "shared memory budget");
    static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPBuf % 1024 == 0 && kOffV % 1024 == 0,
                  "UMMA operands need 1024-byte alignment");
};

// In-kernel merge of a tile's split partials (the stream-k fixup of the
// llama.cpp PR #21086 review, done by the partial kernel itself): every split
// CTA of the tile has written its normalised partial rows (O_s, LSE_s); the
// last one to arrive on the tile's counter merges them,
//   LSE = M + ln sum_s exp(LSE_s - M),  O = sum_s exp(LSE_s - LSE) O_s,
// and writes the final bf16 O and LSE.  The tile's rows of one split are one
// contiguous run of the partial buffer (heads of the tile x query positions),
// so each split arrives by one bulk copy into the CTA's free K/V rings while
// the weights are computed from the LSE partials.  128 threads (the softmax
// warps); the scheduler only picks this mode when the staged partials fit the
// rings.  Writers publish with a fence before the counter increment; the
// merging CTA fences after it and before its bulk copies read the partials.
template <int HD, int NP>
__device__ __noinline__ void merge_tile(const FwdParams& p, int b, int ht, int sb, int rows, int sidx, int w4,
                                        int lane, uint8_t* ring, uint8_t* wbuf_raw, float* lse_row, uint32_t bar,
                                        volatile int* flag, const WaitCtl& wc) {
    const int tile = b * p.head_tiles + ht;  // decode tiles have one m block
    __threadfence();
    named_bar_sync(1, 128);
    if (sidx == 0) {
        const uint32_t prev = atomicAdd(p.counters + tile, 1u);
        *flag = (prev + 1u == uint32_t(sb)) ? 1 : 0;
    }
    named_bar_sync(1, 128);
    if (!*flag) return;
    __threadfence();
    // Rows of the tile in memory order: heads h0 .. h0 + nh - 1, each q_len rows.
    const int h0 = p.pack_gqa ? ht * p.G : ht;
    const int nh = p.pack_gqa ? p.G : 1;
    const size_t stride = size_t(p.B) * p.Hq * p.sq;  // rows between splits
    const size_t base = (size_t(b) * p.Hq + h0) * p.sq;
    const uint32_t bytes = uint32_t(rows) * HD * 4u;
    const uint32_t ring_s = smem_u32(ring);
    if (sidx == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(bar, bytes * uint32_t(sb));
        for (int s = 0; s < sb; ++s)
            bulk_copy_g2s(ring_s + uint32_t(s) * bytes, p.o_part + (size_t(s) * stride + base) * HD, bytes, bar);
    }
    // Weights w[r][s] (the P buffers are free) and the merged LSE per row; warp
    // w4 takes rows w4, w4 + 4, ...; lane t holds splits t, t + 32, ...
    float* wbuf = reinterpret_cast<float*>(wbuf_raw);
    constexpr float kLog2e = 1.4426950408889634074f;
    for (int r = w4; r < rows; r += 4) {
        const size_t rm = base + size_t(r % nh) * p.sq + r / nh;  // packed row r = i * nh + g
        float l[kMaxSplits / 32];
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t) {
            const int sp = t * 32 + lane;
            l[t] = sp < sb ? __ldcg(p.lse_part + size_t(sp) * stride + rm) : -INFINITY;
            mx = fmaxf(mx, l[t]);
        }
        mx = warp_max_f32(mx);
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t) sum += (l[t] == -INFINITY) ? 0.f : exp2f((l[t] - mx) * kLog2e);
        sum = warp_sum(sum);
        const float lse = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
#pragma unroll
        for (int t = 0; t < kMaxSplits / 32; ++t) {
            const int sp = t * 32 + lane;
            if (sp < sb) wbuf[r * sb + sp] = (l[t] == -INFINITY || lse == -INFINITY) ? 0.f : exp2f((l[t] - lse) * kLog2e);
        }
        if (lane == 0) lse_row[r] = lse;
    }
    named_bar_sync(1, 128);
    mbar_wait(bar, 0, wc, (kKernDecode << 8) | kSiteMerge);
    // O rows: item = (row r, float4 column c); splits summed from shared memory.
    constexpr int kC4 = HD / 4;
    for (int it = sidx; it < rows * kC4; it += 128) {
        const int r = it / kC4, c = it - r * kC4;
        const int g = r % nh, i = r / nh;
        const int rmem = g * p.sq + i;  // row in the staged (memory) order
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < sb; ++sp) {
            const float wgt = wbuf[r * sb + sp];
            const float4 v = *reinterpret_cast<const float4*>(ring + (size_t(sp) * rows + rmem) * HD * 4 + c * 16);
            acc.x += wgt * v.x;
            acc.y += wgt * v.y;
            acc.z += wgt * v.z;
            acc.w += wgt * v.w;
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x, acc.y);
        packed.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.out + ((size_t(b) * p.sq + i) * p.Hq + h0 + g) * HD + c * 4) = packed;
        if (c == 0) p.lse[(size_t(b) * p.Hq + h0 + g) * p.sq + i] = lse_row[r];
    }
    if (sidx == 0) p.counters[tile] = 0u;  // ready for the next call on this workspace
    mbar_drain(bar, 0, wc.limit_ns);        // no bulk copy may still be writing when the CTA exits
}

template <int HD, int NP, class Seqs>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_decode_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Seqs seqs) {
    using C = DecodeCfg<HD, NP>;
    constexpr int KST = C::kStagesK;
    constexpr int VST = C::kStagesV;
    constexpr int NB0 = 2 * KST + 2 * VST;  // first barrier after the rings
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- which tile
    const TileCoord tc = p.packed_grid ? packed_tile_of_cta(int(blockIdx.x), p, seqs)
                                       : tile_of_cta(blockIdx.x, blockIdx.y, blockIdx.z, p.num_m_blocks, p.num_splits,
                                                     p.reverse_m != 0);
    const int b = tc.batch;
    const int ht = tc.head_tile;
    const int sb = seqs.splits_of(b);
    const uint32_t word = split_word(tc.split, sb);
    const long long cta_lin =
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    if (tc.split >= sb) {
        griddep_launch_dependents();
        griddep_wait();
        if (p.echo_plan && threadIdx.x == 0) {
            int4 e = make_int4(0, 0, int(word), 0);
            *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = e;
        }
        return;
    }
    const int sk = seqs.seq_len(b);
    const int kv_off = seqs.seq_off(b);
    const BlockRange br =
        tile_key_blocks(p.sq, sk, tc.m_block, p.kBlockM, p.kBlockN, p.win, p.pack_gqa ? p.G : 1, word);
    const int nblocks = br.hi > br.lo ? br.hi - br.lo : 0;
    const int m0 = tc.m_block * p.kBlockM;
    const int rows_valid = min(p.kBlockM, p.rows - m0);

    // ---- shared memory carve-up
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ;
    const uint32_t sP = sbase + C::kOffP;
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* sm_m = reinterpret_cast<float*>(smem + C::kOffM);
    float* sm_alpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
    float* sm_l = reinterpret_cast<float*>(smem + C::kOffL);
    int* sm_diag = reinterpret_cast<int*>(smem + C::kOffDiag);
    const uint32_t bars = sbase + C::kOffBars;
    // barriers: kfull[KST] kempty[KST] vfull[VST] vempty[VST] sfull[2] sempty[2] pfull[2] odone[2] q never drain
    auto bar_kfull = [&](int s) { return bars + 8u * s; };
    auto bar_kempty = [&](int s) { return bars + 8u * (KST + s); };
    auto bar_vfull = [&](int s) { return bars + 8u * (2 * KST + s); };
    auto bar_vempty = [&](int s) { return bars + 8u * (2 * KST + VST + s); };
    auto bar_sfull = [&](int i) { return bars + 8u * (NB0 + i); };
    auto bar_sempty = [&](int i) { return bars + 8u * (NB0 + 2 + i); };
    auto bar_pfull = [&](int i) { return bars + 8u * (NB0 + 4 + i); };
    auto bar_odone = [&](int i) { return bars + 8u * (NB0 + 6 + i); };
    const uint32_t bar_qfull = bars + 8u * (NB0 + 8);
    const uint32_t bar_never = bars + 8u * (NB0 + 9);
    const uint32_t bar_drain = bars + 8u * (NB0 + 10);
    const uint32_t bar_merge = bars + 8u * (NB0 + 11);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    auto stage_k = [&](int s) { return sbase + C::kOffK + uint32_t(s) * C::kKBytes; };
    auto stage_v = [&](int s) { return sbase + C::kOffV + uint32_t(s) * C::kVBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(bar_vfull(s), 1);
            mbar_init(bar_vempty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull(i), 1);
            mbar_init(bar_sempty(i), 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_pfull(i), 128);
            mbar_init(bar_odone(i), 1);
        }
        mbar_init(bar_qfull, 128);
        mbar_init(bar_never, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_merge, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        // The range's first K and V blocks into L2 while the previous kernel on
        // the stream may still be running.  Only a hint: global writes land in
        // L2, so the copies issued after the wait below read current data.
        // Split calls only: back to back, their partial kernel starts during the
        // previous call's combine, which leaves the prefetch time to land (GQA
        // decode, 131072 keys: 49.2 -> 47.0 us a call).  After a single-split
        // call the grid starts only at that call's epilogue, and the prefetch
        // measured slower there (verify over 137 keys: 4.9 -> 5.2 us).
        const int kvh = p.pack_gqa ? ht : ht / p.G;
        const int npre = sb > 1 ? min(nblocks, kDecodeL2Warm) : 0;
        for (int j = 0; j < npre; ++j)
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                tma_prefetch_l2_2d(&tmK, kvh * HD + c * 64, kv_off + (br.lo + j) * 128);
                tma_prefetch_l2_2d(&tmV, kvh * HD + c * 64, kv_off + (br.lo + j) * 128);
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Everything above read only shared memory, TMEM and kernel parameters (the
    // L2 prefetch returns nothing).  Under programmatic dependent launch this
    // grid may start while the previous kernel on the stream is still running:
    // wait for it before any global access.
    griddep_wait();
    if (p.echo_plan && threadIdx.x == 0)
        *reinterpret_cast<int4*>(p.echo + cta_lin * 4) = make_int4(br.lo, br.hi, int(word), 1);
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS0 = tmem;           // S^T buffers: columns [0, NP), [NP, 2NP)
    const uint32_t tO = tmem + 2 * NP;   // O^T: columns [2NP, 3NP)
    WaitCtl wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ===================== TMA producer (K and V rings): the whole warp
        // runs the loop, one elected lane issues the copies.  (One warp per
        // tensor, with K never queued behind a V slot, measured no faster.)
        const bool leader = elect_one();
        const KvRing kr{stage_k(0), uint32_t(C::kKBytes), bar_kfull(0), bar_kempty(0), KST};
        const KvRing vr{stage_v(0), uint32_t(C::kVBytes), bar_vfull(0), bar_vempty(0), VST};
        const int kvh = p.pack_gqa ? ht : ht / p.G;
        produce_kv<HD>(&tmK, &tmV, kr, vr, nblocks, kvh * HD, kv_off + br.lo * 128, false, l2_policy_evict_first(), wc,
                       (kKernDecode << 8) | kSiteProducerEmpty, leader);
    } else if (warp == 1) {
        // ===================== MMA issuer
        // The whole warp runs the schedule (warp-uniform control flow and
        // descriptors); one elected lane issues every tcgen05 op, so its
        // commits track exactly the MMAs it issued.
        const bool leader = elect_one();
        constexpr uint32_t idesc_qk = make_idesc_bf16(128, NP, false, false);
        constexpr uint32_t idesc_pv = make_idesc_bf16(128, NP, true, true);
        // Descriptors built once; per MMA only a constant is added to the
        // start-address field (operands lie below 256 KB: no carry).
        const uint64_t kdesc0 = make_sdesc_sw128(stage_k(0), 16, 1024);
        const uint64_t vdesc0 = make_sdesc_sw128(stage_v(0), 16384, 1024);
        const uint64_t qdesc0 = make_sdesc_sw128(sQ, 16, 1024);
        // P^T: MN-major, no swizzle; core matrices of 8 keys x 8 rows, rows
        // adjacent (128 B apart), key groups (NP / 8) * 128 B apart.
        const uint64_t pdesc0 = make_sdesc_noswz(sP, (NP / 8) * 128, 128);
        bool ok = true;
        if (p.inject_stall) {
            // The injected stall gives up first (half the limit), so the status
            // names it rather than a wait that starves behind it.
            const WaitCtl wc_half{wc.abort_flag, wc.status, wc.limit_ns / 2};
            ok = mbar_wait(bar_never, 0, wc_half, (kKernDecode << 8) | kSiteInjected);
        }
        if (nblocks > 0)
            ok = mbar_wait(bar_qfull, 0, wc, (kKernDecode << 8) | kSiteMmaQ) && ok;
        auto issue_pv = [&](int jj) {
            bool good = mbar_wait(bar_pfull(jj & 1), (jj >> 1) & 1, wc, (kKernDecode << 8) | kSiteMmaPFull);
            const int s = jj % VST;
            good = mbar_wait(bar_vfull(s), (jj / VST) & 1, wc, (kKernDecode << 8) | kSiteMmaFull) && good;
            // The block that holds the end of the sequence also holds rows of
            // the next sequence: their P is 0, but 0 * (Inf or NaN) is NaN, so
            // those V rows are zeroed before the PV MMA reads the slot.
            const int tail_row = sk - (br.lo + jj) * 128;
            if (good && tail_row < 128) zero_rows<HD>(stage_v(s), tail_row, lane);
            tc_fence_after();
            __syncwarp();
            if (leader && good) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = vdesc0 + uint64_t((s * C::kVBytes + kk * 2048) >> 4);
                    const uint64_t bd =
                        pdesc0 + uint64_t(((jj % C::kPBufs) * C::kPBuf + kk * 2 * (NP / 8) * 128) >> 4);
                    umma_bf16(tO, a, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar_odone(jj & 1));
                umma_commit(bar_vempty(s));
            }
        };
        for (int j = 0; j < nblocks; ++j) {
            const int s = j % KST;
            bool good = mbar_wait(bar_kfull(s), (j / KST) & 1, wc, (kKernDecode << 8) | kSiteMmaFull);
            if (j >= 2)
                good = mbar_wait(bar_sempty(j & 1), ((j >> 1) - 1) & 1, wc,
                                 (kKernDecode << 8) | kSiteMmaSEmpty) && good;
            tc_fence_after();
            __syncwarp();
            if (leader && good && ok) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t a =
                        kdesc0 + uint64_t((s * C::kKBytes + (kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    const uint64_t bd = qdesc0 + uint64_t(((kk >> 2) * (NP * 128) + (kk & 3) * 32) >> 4);
                    umma_bf16(tS0 + (j & 1) * NP, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar_sfull(j & 1));
                umma_commit(bar_kempty(s));
            }
            if (j >= 1) issue_pv(j - 1);
        }
        if (nblocks >= 1) issue_pv(nblocks - 1);
        // Every issued MMA completes before TMEM is released.
        __syncwarp();
        if (leader) umma_commit(bar_drain);
        mbar_drain(bar_drain, 0, p.timeout_ns);
    } else {
        // ===================== softmax / correction / epilogue (128 threads)
        const int sidx = threadIdx.x - 64;            // 0..127 for cooperative loops
        const int kt = 32 * (warp & 3) + lane;        // TMEM lane owned by this thread
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const int diag_shift = sk - p.sq;

        // Q tile -> smem (K-major, 128B swizzle), padded rows zero.  All of a
        // thread's loads are issued before any store so that they overlap.
        {
            constexpr int kGran = HD / 8;  // 16-byte granules per row
            constexpr int kPer = (NP * kGran + 127) / 128;
            uint4 val[kPer];
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int idx = sidx + t * 128;
                const int r = idx / kGran;
                const int g16 = idx - r * kGran;
                val[t] = make_uint4(0, 0, 0, 0);
                if (idx < NP * kGran && r < rows_valid) {
                    const RowMap rm = map_row(p, ht, m0 + r);
                    val[t] = __ldg(reinterpret_cast<const uint4*>(
                        p.q + ((size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * HD + g16 * 8));
                }
            }
#pragma unroll
            for (int t = 0; t < kPer; ++t) {
                const int idx = sidx + t * 128;
                if (idx < NP * kGran) {
                    const int r = idx / kGran;
                    const int g16 = idx - r * kGran;
                    const uint32_t dst = sQ + (g16 >> 3) * (NP * 128) + sw128_offset(r, g16 & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(val[t].x), "r"(val[t].y),
                                 "r"(val[t].z), "r"(val[t].w)
                                 : "memory");
                }
            }
        }
        if (sidx < NP) {
            sm_m[sidx] = -INFINITY;
            sm_diag[sidx] = (sidx < rows_valid) ? map_row(p, ht, m0 + sidx).i + diag_shift : 0;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_qfull);
        named_bar_sync(1, 128);

        // Rows whose query sees the whole block need no element mask.
        const int diag_lo = (rows_valid > 0) ? sm_diag[0] : 0;
        const int diag_hi = (rows_valid > 0) ? sm_diag[rows_valid - 1] : 0;
        const bool has_causal = p.causal != 0;
        const bool has_window = p.window_left >= 0;

        // Per row q (identical in every thread): neg_m[q] = -(running max) in
        // log2 units, 0 while the row has seen no visible key; -1e30 for padding
        // rows, whose scores thereby fall to -1e30 and their P to 0.  The
        // running max itself lives in sm_m and is only read on the blocks that
        // raise it.  Until every valid row has a finite max, every block takes
        // the rescale path, which sets the max of the rows that start there.
        float l_t[NP];
        float neg_m[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            l_t[q] = 0.f;
            neg_m[q] = (q < rows_valid) ? 0.f : -1e30f;
        }
        bool unstarted = rows_valid > 0;
        const float sl2 = p.scale_log2;
        const uint32_t p_st = sP + uint32_t((kt >> 3) * (NP / 8) * 128 + (kt & 7) * 16);
        // The rows that see this thread's key, as bits (bit q: row q), from a
        // rolled loop over the rows: per-row tests unrolled over the NP rows
        // made the masked blocks' code so long that a CTA starting on a masked
        // block spent microseconds fetching it.
        auto visible_rows = [&](int key) -> unsigned long long {
            unsigned long long vis = 0ull;
            if (key < sk) {
#pragma unroll 4
                for (int q = 0; q < rows_valid; ++q) {
                    const int dg = sm_diag[q];
                    const bool ok = (!has_causal || key <= dg) && (!has_window || key >= dg - p.window_left);
                    vis |= (unsigned long long)ok << q;
                }
            }
            return vis;
        };

        for (int j = 0; j < nblocks; ++j) {
            const int n = br.lo + j;
            const uint32_t tS = tS0 + (j & 1) * NP + lane_off;
            float t[NP];  // scaled scores minus the running max, log2 units
            mbar_wait(bar_sfull(j & 1), (j >> 1) & 1, wc, (kKernDecode << 8) | kSiteSoftmaxSFull);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) tmem_ld16(tS + c * 16, t + c * 16);
            tmem_wait_ld();

            const int key = n * 128 + kt;
            const int blk_first = n * 128, blk_last = n * 128 + 127;
            const bool need_mask = (blk_last >= sk) || (has_causal && blk_last > diag_lo) ||
                                   (has_window && blk_first < diag_hi - p.window_left);
#pragma unroll
            for (int q = 0; q < NP; ++q) t[q] = fmaf(t[q], sl2, neg_m[q]);
            if (need_mask) {
                const unsigned long long vis = visible_rows(key);
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    if (!((vis >> q) & 1ull)) t[q] = -INFINITY;
            }
            bool need = unstarted;
#pragma unroll
            for (int q = 0; q < NP; ++q) need |= t[q] > kRescaleThreshold;
            if (named_bar_or(1, 128, need)) {
                // A row's max grew by more than 2^8, or a row may see its first
                // key here: take every row's block max (t - neg_m is the scaled
                // score; -inf where masked), move the running maxima and shift
                // the scores by the change.
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float v = warp_max_f32(t[q] - neg_m[q]);
                    if (lane == 0) red[(warp & 3) * NP + q] = v;
                }
                named_bar_sync(1, 128);
                bool still = false;  // a valid row without a visible key so far
                if (sidx < NP) {
                    const int q = sidx;
                    float a = 1.f;
                    if (q < rows_valid) {
                        const float bm = fmaxf(fmaxf(red[q], red[NP + q]), fmaxf(red[2 * NP + q], red[3 * NP + q]));
                        const float mo = sm_m[q];
                        const float mn = fmaxf(mo, bm);
                        a = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);  // l and O are 0 while mo = -inf
                        sm_m[q] = mn;
                        still = mn == -INFINITY;
                    }
                    sm_alpha[q] = a;
                }
                unstarted = named_bar_or(1, 128, still);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    if (q < rows_valid) {
                        const float mq = sm_m[q];
                        const float nm = (mq == -INFINITY) ? 0.f : -mq;
                        t[q] += nm - neg_m[q];
                        neg_m[q] = nm;
                    }
                    l_t[q] *= sm_alpha[q];
                }
                // Rescaling O needs the previous block's PV to be complete.
                if (j >= 1) {
                    mbar_wait(bar_odone((j - 1) & 1), ((j - 1) >> 1) & 1, wc,
                              (kKernDecode << 8) | kSiteSoftmaxODone);
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < NP / 16; ++c) {
                        float o[16];
                        tmem_ld16(tO + lane_off + c * 16, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] *= sm_alpha[c * 16 + e];
                        tmem_st16(tO + lane_off + c * 16, o);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_before();
            mbar_arrive(bar_sempty(j & 1));

            // P = 2^t, summed per row, packed as bf16 pairs of consecutive rows.
            uint32_t pk[NP / 2];
#pragma unroll
            for (int e = 0; e < NP / 2; ++e) {
                const float p0 = fast_exp2(t[2 * e]);
                const float p1 = fast_exp2(t[2 * e + 1]);
                l_t[2 * e] += p0;
                l_t[2 * e + 1] += p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            // P buffer j % kPBufs was last read by the PV of block j - kPBufs.
            if (j >= C::kPBufs) {
                const int jp = j - C::kPBufs;
                mbar_wait(bar_odone(jp & 1), (jp >> 1) & 1, wc, (kKernDecode << 8) | kSiteSoftmaxODone);
                tc_fence_after();
            }
            // P^T -> smem, MN-major without swizzle: key kt's 8 consecutive rows
            // form one 16-byte line of a core matrix ([key / 8][row / 8][key % 8][row % 8]).
            {
                const uint32_t dst = p_st + uint32_t((j % C::kPBufs) * C::kPBuf);
#pragma unroll
                for (int g = 0; g < NP / 8; ++g)
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + g * 128), "r"(pk[4 * g]),
                                 "r"(pk[4 * g + 1]), "r"(pk[4 * g + 2]), "r"(pk[4 * g + 3])
                                 : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_pfull(j & 1));
        }

        // Let the dependent grid (the combine, or the next call's partial kernel)
        // get scheduled; it waits for this grid's completion before reading.
        griddep_launch_dependents();
        // ---- epilogue: l across the 128 key lanes, then O^T / l
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const float v = warp_sum(l_t[q]);
            if (lane == 0) red[(warp & 3) * NP + q] = v;
        }
        named_bar_sync(1, 128);
        // One thread per row: the row's LSE, 1 / l (into sm_l) and the element
        // offset of its output row (into red, free once the sums are read).  The
        // stores below then carry no per-row index arithmetic: with every row
        // unrolled that arithmetic made the epilogue long enough that, run once
        // per CTA from a cold instruction cache, it took longer than the loop.
        const bool final_out = (sb == 1);
        long long* row_off = reinterpret_cast<long long*>(red);
        float l_row = 0.f;
        if (sidx < NP) l_row = red[sidx] + red[NP + sidx] + red[2 * NP + sidx] + red[3 * NP + sidx];
        named_bar_sync(1, 128);
        if (sidx < NP) {
            const int q = sidx;
            long long off = 0;
            if (q < rows_valid) {
                const RowMap rm = map_row(p, ht, m0 + q);
                const float lse = l_row > 0.f ? (sm_m[q] + log2f(l_row)) * kLn2 : -INFINITY;
                if (final_out) {
                    off = ((long long)(size_t(b) * p.sq + rm.i) * p.Hq + rm.h) * HD;
                    p.lse[(size_t(b) * p.Hq + rm.h) * p.sq + rm.i] = lse;
                } else {
                    const size_t prow = ((size_t(tc.split) * p.B + b) * p.Hq + rm.h) * p.sq + rm.i;
                    off = (long long)prow * HD;
                    p.lse_part[prow] = lse;
                }
            }
            row_off[q] = off;
            sm_l[q] = l_row > 0.f ? 1.f / l_row : 0.f;
        }
        named_bar_sync(1, 128);

        float o[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) o[q] = 0.f;
        if (nblocks >= 1) {
            mbar_wait(bar_odone((nblocks - 1) & 1), ((nblocks - 1) >> 1) & 1, wc,
                      (kKernDecode << 8) | kSiteSoftmaxODone);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) tmem_ld16(tO + lane_off + c * 16, o + c * 16);
            tmem_wait_ld();
        }
        if (kt < HD) {
            if (final_out) {
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    if (q < rows_valid) p.out[row_off[q] + kt] = __float2bfloat16_rn(o[q] * sm_l[q]);
            } else {
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    if (q < rows_valid) p.o_part[row_off[q] + kt] = o[q] * sm_l[q];
            }
        }
        if (!final_out && p.fused_combine)
            merge_tile<HD, NP>(p, b, ht, sb, rows_valid, sidx, warp & 3, lane, smem + C::kOffK, smem + C::kOffP, red,
                               bar_merge, merge_flag, wc);
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int HD, int NP, class Seqs>
cudaError_t launch_one(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const Seqs& seqs, cudaStream_t stream) {
    using C = DecodeCfg<HD, NP>;
    auto kern = fwd_decode_kernel<HD, NP, Seqs>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    return launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), C::kSmemAlloc, stream, p, tmK, tmV,
                      seqs);
}

template <int HD, class Seqs>
cudaError_t dispatch_np(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, const Seqs& seqs, cudaStream_t stream) {
    switch (plan.kBlockM) {
        case 16: return launch_one<HD, 16>(plan, p, tmK, tmV, seqs, stream);
        case 32: return launch_one<HD, 32>(plan, p, tmK, tmV, seqs, stream);
        case 48: return launch_one<HD, 48>(plan, p, tmK, tmV, seqs, stream);
        case 64: return launch_one<HD, 64>(plan, p, tmK, tmV, seqs, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

void fill_varlen(const Plan& plan, VarlenSeqs* v) {
    for (int b = 0; b <= plan.B && b <= kMaxVarlenBatch; ++b) v->off[b] = int(plan.kv_off[size_t(b)]);
    for (int b = 0; b < plan.B && b < kMaxVarlenBatch; ++b)
        v->splits[b] = (unsigned short)plan.splits_b[size_t(b)];
}

cudaError_t launch_decode(const Plan& plan, const FwdParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t stream) {
    if (!plan.varlen) {
        UniformSeqs u{plan.kv_len[0], plan.splits_b[0]};
        return plan.d == 128 ? dispatch_np<128>(plan, p, tmK, tmV, u, stream)
                             : dispatch_np<64>(plan, p, tmK, tmV, u, stream);
    }
    VarlenSeqs v;  // copied into the launch's parameter buffer at launch
    fill_varlen(plan, &v);
    return plan.d == 128 ? dispatch_np<128>(plan, p, tmK, tmV, v, stream)
                         : dispatch_np<64>(plan, p, tmK, tmV, v, stream);
}

}  // namespace sk
