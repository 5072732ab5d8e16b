// kv_producer.cuh -- the TMA producers of the partial kernels: K and V blocks
// of 128 rows stream through two separate shared-memory rings.  A K slot is
// refilled as soon as the QK^T MMAs that read it have completed, a V slot as
// soon as its PV MMAs have, so K runs ahead of V and the next QK^T never waits
// for a whole K+V load.
//
// One warp streams both: the MMA warp issues QK^T(j) before the last PV(j-1),
// so the slots free up in the order K(j), V(j-1), K(j+1), V(j), ...; the
// producer waits for them in exactly that order.
// All waits are bounded and suspend the thread.  The whole producer warp runs
// these loops (warp-uniform control flow); one elected lane, `leader`, issues
// the copies.  A ring position counts the blocks loaded so far: slot
// pos % slots, use pos / slots.
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

// One 128-row block (rows y .. y + 127, columns x0 .. x0 + HD) into ring position pos.
template <int HD>
__device__ __forceinline__ bool load_block(const CUtensorMap* tm, const KvRing& R, int pos, int x0, int y,
                                           uint64_t policy, const WaitCtl& wc, int where, bool leader) {
    constexpr uint32_t kBytes = 128u * HD * 2u;
    const int s = pos % R.slots, u = pos / R.slots;
    const bool ok = __all_sync(0xffffffffu, u < 1 || mbar_wait(R.empty + 8u * s, (u - 1) & 1, wc, where));
    if (!ok) return false;
    if (leader) {
        mbar_arrive_expect_tx(R.full + 8u * s, kBytes);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
            tma_load_2d(R.base + s * R.stride + c * 16384, tm, R.full + 8u * s, x0 + c * 64, y, policy);
    }
    return true;
}

// K and V blocks of rows y0 + 128 * visit_block(j), j in [0, nblocks), into
// ring positions g0 + j (K of j = 0 skipped when the caller has issued it).  kpos / vpos advance past every load issued, so the
// caller can drain exactly those; returns false once a wait has given up.
template <int HD>
__device__ __forceinline__ bool produce_kv_tile(const CUtensorMap* tmK, const CUtensorMap* tmV, const KvRing& K,
                                                const KvRing& V, int g0, int nblocks, int x0, int y0, bool desc,
                                                uint64_t policy, const WaitCtl& wc, int where, bool leader,
                                                int& kpos, int& vpos, bool k0_issued = false) {
    auto row = [&](int j) { return y0 + visit_block(j, nblocks, desc) * 128; };
    if (nblocks > 0) {
        if (!k0_issued && !load_block<HD>(tmK, K, g0, x0, row(0), policy, wc, where, leader)) return false;
        kpos = g0 + 1;
    }
    for (int j = 1; j <= nblocks; ++j) {
        if (j < nblocks) {
            if (!load_block<HD>(tmK, K, g0 + j, x0, row(j), policy, wc, where, leader)) return false;
            kpos = g0 + j + 1;
        }
        if (!load_block<HD>(tmV, V, g0 + j - 1, x0, row(j - 1), policy, wc, where, leader)) return false;
        vpos = g0 + j;
    }
    return true;
}

// Zero rows [first, 128) of a 128-row K/V block in shared memory (HD / 64
// chunks of 128 rows x 128 bytes; a whole row is zeroed, so its swizzle does
// not matter), by the 32 lanes of one warp, then make the zeros visible to the
// tensor cores (async proxy).  Called after the block's copy has completed.
template <int HD>
__device__ __forceinline__ void zero_rows(uint32_t slot, int first, int lane) {
    const int n16 = (128 - first) * 8;  // 16-byte granules per chunk
#pragma unroll
    for (int c = 0; c < HD / 64; ++c)
        for (int idx = lane; idx < n16; idx += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(slot + c * 16384 + first * 128 + idx * 16),
                         "r"(0u)
                         : "memory");
    fence_proxy_async_smem();
}

// Before the CTA exits: the last load of every slot (ring positions below
// `loaded`) must have landed.
__device__ __forceinline__ void drain_ring(const KvRing& R, int loaded, uint64_t limit_ns) {
    for (int pos = loaded - 1; pos >= 0 && pos >= loaded - R.slots; --pos)
        mbar_drain(R.full + 8u * (pos % R.slots), (pos / R.slots) & 1, limit_ns);
}

// Single-tile form: stream one range, then drain what was issued.
template <int HD>
__device__ __forceinline__ void produce_kv(const CUtensorMap* tmK, const CUtensorMap* tmV, const KvRing& K,
                                           const KvRing& V, int nblocks, int x0, int y0, bool desc,
                                           uint64_t policy, const WaitCtl& wc, int where, bool leader) {
    int kpos = 0, vpos = 0;
    produce_kv_tile<HD>(tmK, tmV, K, V, 0, nblocks, x0, y0, desc, policy, wc, where, leader, kpos, vpos);
    drain_ring(K, kpos, wc.limit_ns);
    drain_ring(V, vpos, wc.limit_ns);
}

}  // namespace sk
