// kv_producer.cuh -- the TMA producer shared by the partial kernels: K and V
// blocks of 128 rows stream through two separate shared-memory rings.  A K slot
// is refilled as soon as the QK^T MMA that read it has completed, a V slot as
// soon as its PV MMA has, so K runs ahead of V and the next QK^T never waits for
// a whole K+V load.  The MMA warp issues QK^T(j) before PV(j-1), so the slots
// free up in the order K(j), V(j-1), K(j+1), V(j), ...; the producer waits for
// them in exactly that order (bounded waits that suspend the thread).
#pragma once
#include "sm103_ptx.cuh"

namespace sk {

// The j-th block a CTA visits is block (j + rot) mod nblocks of its range.  The
// online softmax does not depend on the visiting order; CTAs that share K/V
// (the m blocks of one head) start at different blocks, so they do not all
// read the same few L2 lines at the same moment.
__device__ __forceinline__ int rotated_block(int j, int rot, int nblocks) {
    int b = j + rot;
    return b >= nblocks ? b - nblocks : b;
}

struct KvRing {
    uint32_t base;    // shared address of slot 0
    uint32_t stride;  // bytes between slots
    uint32_t full;    // shared address of full[0] (8 bytes apart)
    uint32_t empty;   // shared address of empty[0]
    int slots;
};

template <int HD>
__device__ __forceinline__ bool load_block(const CUtensorMap* tm, const KvRing& R, int j, int x0, int y0,
                                           int rot, int nblocks, uint64_t policy, const WaitCtl& wc, int where) {
    constexpr uint32_t kBytes = 128u * HD * 2u;
    const int s = j % R.slots, u = j / R.slots;
    if (u >= 1 && !mbar_wait(R.empty + 8u * s, (u - 1) & 1, wc, where)) return false;
    mbar_arrive_expect_tx(R.full + 8u * s, kBytes);
#pragma unroll
    for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(R.base + s * R.stride + c * 16384, tm, R.full + 8u * s, x0 + c * 64,
                    y0 + rotated_block(j, rot, nblocks) * 128, policy);
    return true;
}

// Loads K and V blocks of rows y0 + 128 * rotated_block(j), j in [0, nblocks),
// columns x0 .. x0 + HD (HD / 64 boxes of 64 columns, 16 KB apart in a slot).
template <int HD>
__device__ __forceinline__ void produce_kv(const CUtensorMap* tmK, const CUtensorMap* tmV, const KvRing& K,
                                           const KvRing& V, int nblocks, int x0, int y0, int rot, uint64_t policy,
                                           const WaitCtl& wc, int where) {
    int jk = 0, jv = 0;  // blocks issued on each ring
    if (nblocks > 0 && load_block<HD>(tmK, K, 0, x0, y0, rot, nblocks, policy, wc, where)) jk = 1;
    for (int j = 1; j <= nblocks && jk == j; ++j) {
        if (j < nblocks) {
            if (!load_block<HD>(tmK, K, j, x0, y0, rot, nblocks, policy, wc, where)) break;
            jk = j + 1;
        }
        if (!load_block<HD>(tmV, V, j - 1, x0, y0, rot, nblocks, policy, wc, where)) break;
        jv = j;
    }
    // Drain: the last load of every slot must land before the CTA exits.
    for (int j = jk - 1; j >= 0 && j >= jk - K.slots; --j)
        mbar_drain(K.full + 8u * (j % K.slots), (j / K.slots) & 1, wc.limit_ns);
    for (int j = jv - 1; j >= 0 && j >= jv - V.slots; --j)
        mbar_drain(V.full + 8u * (j % V.slots), (j / V.slots) & 1, wc.limit_ns);
}

// Cluster of two CTAs that need the same K/V blocks (two query heads of one KV
// head with the same block range): each CTA loads one 64-column half of every
// block and multicasts it to both.  A slot's full barrier expects the whole
// block (both halves); its empty barrier counts one release from each CTA.
template <int HD>
__device__ __forceinline__ bool load_block_pair(const CUtensorMap* tm, const KvRing& R, int j, int x0, int y0,
                                                int rot, int nblocks, uint32_t rank, uint64_t policy,
                                                const WaitCtl& wc, int where) {
    static_assert(HD == 128, "paired loads split a 128-column block into two halves");
    constexpr uint32_t kBytes = 128u * HD * 2u;
    const int s = j % R.slots, u = j / R.slots;
    if (u >= 1 && !mbar_wait(R.empty + 8u * s, (u - 1) & 1, wc, where)) return false;
    mbar_arrive_expect_tx(R.full + 8u * s, kBytes);
    tma_load_2d_mc(R.base + s * R.stride + rank * 16384, tm, R.full + 8u * s, x0 + int(rank) * 64,
                   y0 + rotated_block(j, rot, nblocks) * 128, uint16_t(0x3), policy);
    return true;
}

template <int HD>
__device__ __forceinline__ void produce_kv_pair(const CUtensorMap* tmK, const CUtensorMap* tmV, const KvRing& K,
                                                const KvRing& V, int nblocks, int x0, int y0, int rot,
                                                uint32_t rank, uint64_t policy, const WaitCtl& wc, int where) {
    int jk = 0, jv = 0;
    if (nblocks > 0 && load_block_pair<HD>(tmK, K, 0, x0, y0, rot, nblocks, rank, policy, wc, where)) jk = 1;
    for (int j = 1; j <= nblocks && jk == j; ++j) {
        if (j < nblocks) {
            if (!load_block_pair<HD>(tmK, K, j, x0, y0, rot, nblocks, rank, policy, wc, where)) break;
            jk = j + 1;
        }
        if (!load_block_pair<HD>(tmV, V, j - 1, x0, y0, rot, nblocks, rank, policy, wc, where)) break;
        jv = j;
    }
    for (int j = jk - 1; j >= 0 && j >= jk - K.slots; --j)
        mbar_drain(K.full + 8u * (j % K.slots), (j / K.slots) & 1, wc.limit_ns);
    for (int j = jv - 1; j >= 0 && j >= jv - V.slots; --j)
        mbar_drain(V.full + 8u * (j % V.slots), (j / V.slots) & 1, wc.limit_ns);
}

}  // namespace sk
