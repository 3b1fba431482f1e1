// cta_pair.cuh -- the two CTAs of a cluster of two working as one tensor-core pair
// (tcgen05 cta_group::2): TMEM allocation for the pair, pair MMAs issued from the even CTA,
// TMA copies that complete on the even CTA's barrier, and the cluster-scope barrier waits
// and arrivals around them.  Plain inline PTX.
//
// A kernel uses either these tcgen05 forms or the cta_group::1 ones of tcgen05.cuh, never
// both.  The MMA is issued from the even CTA and reads its A rows and B columns from the
// shared memory of both (the same offsets in each), writing the D rows of each CTA to that
// CTA's TMEM.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace inkattn {

// Non-blocking test of a phase that other CTAs of the cluster complete (arrivals made with
// release at cluster scope, mbar_remote_arrive): cluster-scope acquire.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// mbar_wait for a phase completed from another CTA of the cluster (a remote arrival, or a
// tensor-core commit issued there).  It polls, with a short back-off: a thread suspended in
// try_wait is not woken promptly by such an arrival.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int32_t *status,
                                                  volatile int *abort, uint64_t limit_ns) {
    if (mbar_test_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_test_wait_cluster(bar, parity)) return true;
        __nanosleep(32);
        if ((n & 255u) == 0u) {
            if (abort && *abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                set_status(status, INKATTN_ERR_DEVICE_TIMEOUT);
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}

// One arrival, with release at cluster scope, on the mbarrier at `bar`'s offset in the
// shared memory of CTA `cta_rank` of the cluster.
__device__ __forceinline__ void mbar_remote_arrive(uint32_t bar, uint32_t cta_rank) {
    asm volatile("{\n\t.reg .b32 ra;\n\tmapa.shared::cluster.u32 ra, %0, %1;\n\t"
                 "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}"
                 :: "r"(bar), "r"(cta_rank) : "memory");
}

// As tma_load_2d, for a CTA pair: the box lands in this CTA's shared memory and its bytes
// complete on the mbarrier `bar_pair` of the even CTA of the pair (a shared::cluster
// address, from mapa), which counts the copies of both CTAs.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *map, int c0, int c1,
                                                 uint32_t bar_pair) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_pair)
        : "memory");
}

// The shared::cluster address of the object at `addr`'s offset in CTA `cta_rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t cta_rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta_rank));
    return r;
}

namespace tc {

// TMEM allocation for the pair: one warp of each of the two CTAs executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// One K = 64 stage of a pair GEMM tile (M = 256 over the two CTAs): four K = 16 MMAs over
// 128-byte-swizzled K-major A and B tiles (the k steps advance the start addresses by 32
// bytes, 2 in descriptor units), then, when `rel` is nonzero, a commit of them to the
// mbarrier at `rel_bar`'s offset in both CTAs, and, when `done` is nonzero, a second such
// commit to `done_bar`.  acc0 = 0 makes the first MMA overwrite D.  Warp-collective like
// mma_bf16_ss (one elected lane issues).
__device__ __forceinline__ void mma_pair_bf16_ss_k64_commit(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                                            uint32_t acc0, uint32_t rel_bar, uint32_t rel,
                                                            uint32_t done_bar, uint32_t done) {
    asm volatile("{\n\t.reg .pred e, p0, pt, pr, pd;\n\t.reg .b64 a1, b1;\n\t.reg .b16 m;\n\t"
                 "mov.b16 m, 3;\n\t"
                 "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.u32 pt, 0, 0;\n\t"
                 "setp.ne.b32 pr, %6, 0;\n\tsetp.ne.b32 pd, %8, 0;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\tand.pred pr, pr, e;\n\tand.pred pd, pd, e;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p0;\n\t"
                 "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, pt;\n\t"
                 "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, pt;\n\t"
                 "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, pt;\n\t"
                 "@pr tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%5], m;\n\t"
                 "@pd tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%7], m;\n\t}"
                 :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc0), "r"(rel_bar), "r"(rel), "r"(done_bar),
                    "r"(done)
                 : "memory");
}
// Arrives once on the local mbarrier when every pair MMA issued so far by the elected lane
// has completed.  Warp-collective.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 :: "r"(bar) : "memory");
}

}  // namespace tc
}  // namespace inkattn
