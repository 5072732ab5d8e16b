// kv_producer.cuh -- the TMA producer shared by the partial kernels: K and V
// blocks of 128 rows stream through two separate shared-memory rings.  A K slot
// is refilled as soon as the QK^T MMAs that read it have completed, a V slot as
// soon as its PV MMAs have, so K runs ahead of V and the next QK^T never waits
// for a whole K+V load.  The MMA warp issues QK^T(j) before the last PV(j-1),
// so the slots free up in the order K(j), V(j-1), K(j+1), V(j), ...; the
// producer waits for them in exactly that order (bounded waits that suspend the
// thread).
#pragma once
#include "sm103_ptx.cuh"

namespace sk {

// The j-th block a CTA visits: ascending, or descending from the last block of
// its range (causal and local tiles then meet their masked diagonal blocks
// first).  The online softmax does not depend on the visiting order.
__device__ __forceinline__ int visit_block(int j, int nblocks, bool desc) { return desc ? nblocks - 1 - j : j; }

struct KvRing {
    uint32_t base;    // shared address of slot 0
    uint32_t stride;  // bytes between slots
    uint32_t full;    // shared address of full[0] (8 bytes apart)
    uint32_t empty;   // shared address of empty[0]
    int slots;
};

// One block into ring slot j % slots.  With CL > 1 the CTA is rank `rank` of a
// cluster of CL CTAs that visit the same blocks: it loads rows
// [rank * 128 / CL, (rank + 1) * 128 / CL) of the block and multicasts them to
// every CTA of the cluster, so each block leaves L2 once per cluster.  Every
// CTA's full barrier expects the whole block (its own rows and the peers');
// every empty barrier counts one release from each CTA of the cluster.
template <int HD, int CL>
__device__ __forceinline__ bool load_block(const CUtensorMap* tm, const KvRing& R, int j, int x0, int y0,
                                           int nblocks, bool desc, uint32_t rank, uint64_t policy,
                                           const WaitCtl& wc, int where) {
    constexpr uint32_t kBytes = 128u * HD * 2u;
    constexpr int kRows = 128 / CL;  // rows per TMA box
    const int s = j % R.slots, u = j / R.slots;
    if (u >= 1 && !mbar_wait(R.empty + 8u * s, (u - 1) & 1, wc, where)) return false;
    mbar_arrive_expect_tx(R.full + 8u * s, kBytes);
    const int y = y0 + visit_block(j, nblocks, desc) * 128 + int(rank) * kRows;
#pragma unroll
    for (int c = 0; c < HD / 64; ++c) {
        const uint32_t dst = R.base + s * R.stride + c * 16384 + rank * uint32_t(kRows * 128);
        if constexpr (CL == 1)
            tma_load_2d(dst, tm, R.full + 8u * s, x0 + c * 64, y, policy);
        else
            tma_load_2d_mc(dst, tm, R.full + 8u * s, x0 + c * 64, y, uint16_t((1u << CL) - 1u), policy);
    }
    return true;
}

// Loads K and V blocks of rows y0 + 128 * visit_block(j), j in [0, nblocks),
// columns x0 .. x0 + HD (HD / 64 boxes of 64 columns, 16 KB apart in a slot).
template <int HD, int CL = 1>
__device__ __forceinline__ void produce_kv(const CUtensorMap* tmK, const CUtensorMap* tmV, const KvRing& K,
                                           const KvRing& V, int nblocks, int x0, int y0, bool desc,
                                           uint32_t rank, uint64_t policy, const WaitCtl& wc, int where) {
    int jk = 0, jv = 0;  // blocks issued on each ring
    if (nblocks > 0 && load_block<HD, CL>(tmK, K, 0, x0, y0, nblocks, desc, rank, policy, wc, where)) jk = 1;
    for (int j = 1; j <= nblocks && jk == j; ++j) {
        if (j < nblocks) {
            if (!load_block<HD, CL>(tmK, K, j, x0, y0, nblocks, desc, rank, policy, wc, where)) break;
            jk = j + 1;
        }
        if (!load_block<HD, CL>(tmV, V, j - 1, x0, y0, nblocks, desc, rank, policy, wc, where)) break;
        jv = j;
    }
    // Drain: the last load of every slot must land before the CTA exits.
    for (int j = jk - 1; j >= 0 && j >= jk - K.slots; --j)
        mbar_drain(K.full + 8u * (j % K.slots), (j / K.slots) & 1, wc.limit_ns);
    for (int j = jv - 1; j >= 0 && j >= jv - V.slots; --j)
        mbar_drain(V.full + 8u * (j % V.slots), (j / V.slots) & 1, wc.limit_ns);
    if constexpr (CL > 1) {
        // The peers' MMAs release this CTA's slots remotely: wait for the last
        // release of every slot, so none arrives after the CTA has left.
        for (int j = nblocks - 1; j >= 0 && j >= nblocks - K.slots; --j)
            mbar_drain(K.empty + 8u * (j % K.slots), (j / K.slots) & 1, wc.limit_ns);
        for (int j = nblocks - 1; j >= 0 && j >= nblocks - V.slots; --j)
            mbar_drain(V.empty + 8u * (j % V.slots), (j / V.slots) & 1, wc.limit_ns);
    }
}

}  // namespace sk
