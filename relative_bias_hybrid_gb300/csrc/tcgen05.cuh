// tcgen05.cuh -- 5th-generation tensor-core helpers (sm_100 family, here sm_103a):
// TMEM allocation, shared-memory matrix descriptors, instruction descriptors,
// tcgen05.mma (operands in shared memory, or A in TMEM), commit to an mbarrier, and
// TMEM <-> register moves.  Plain inline PTX.
#pragma once

#include <stdint.h>

namespace inkattn {
namespace tc {

// ---------------------------------------------------------------- TMEM allocation

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
// Per-thread register budget of the calling warpgroup (all four of its warps execute it).
// The launch hands every thread the kernel's register count; a decrease returns registers
// to the CTA's pool and an increase waits until the pool holds enough, so the warpgroups'
// budgets must add up to no more than the threads times the launch count.
template <int N> __device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(N));
}
template <int N> __device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(N));
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading- and
// stride-dimension byte offsets (16-byte units), descriptor version 1 (bit 46),
// layout type 2 = SWIZZLE_128B (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// As sdesc_sw128, layout type 4 = SWIZZLE_64B (64-byte rows, 8-row atoms of 512 bytes).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;
    return d;
}

// Instruction descriptor: D fp32 (bits 4-5 = 1), A/B element format (bits 7-9, 10-12:
// 1 = bf16 for kind::f16), A/B major (bits 15, 16: 1 = MN-major),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc(int M, int N, uint32_t ab_format, int a_mn, int b_mn) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kFmtBF16 = 1;
constexpr uint32_t kFmtF16 = 0;

// ---------------------------------------------------------------- MMA + commit
// Warp-collective: all 32 lanes of a converged warp make the call with the same operands,
// and one lane, elected inside the instruction sequence, issues.  A lone thread issuing
// from a divergent branch (if (lane == 0)) spends several instructions of its own on every
// MMA; while the other warps of its SM sub-partition keep the issue port busy (softmax
// arithmetic), those delay each MMA past the 64 cycles the tensor pipe needs for an
// M = 128, N = 128, K = 16 step, and the step takes ~130 cycles instead.  With the operands
// warp-uniform the issue keeps up with the pipe.  The commits elect the same lane, so they
// track the MMAs that lane issued.

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 inputs), cta_group::1.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
// Arrives once on the mbarrier when every tcgen05 operation issued so far by the elected
// lane has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 :: "r"(bar) : "memory");
}

// A whole K = 128 step (eight K = 16 MMAs), a commit of it to `bar` and, when `rel` is
// nonzero, a second commit to `rel_bar` (in every CTA named in `rel_mask` when kMc), all in
// one instruction sequence with one election: the issuing lane spends no instructions of
// its own between them.  acc0 = 0 makes the first MMA overwrite D.  Warp-collective like
// the single forms.
//
// SS: A and B are 128-byte-swizzled K-major tiles stored as two 64-column halves 16 KB
// apart; the k-step start addresses advance by 32 bytes within a half (2 in the
// descriptor's 16-byte units) and by 16 KB (1024) to the second half.
#define INKATTN_MMA_SS_K128 \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t" \
    "add.s64 a1, %1, 2;\n\t" \
    "add.s64 b1, %2, 2;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 4;\n\t" \
    "add.s64 b1, %2, 4;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 6;\n\t" \
    "add.s64 b1, %2, 6;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 1024;\n\t" \
    "add.s64 b1, %2, 1024;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 1026;\n\t" \
    "add.s64 b1, %2, 1026;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 1028;\n\t" \
    "add.s64 b1, %2, 1028;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "add.s64 a1, %1, 1030;\n\t" \
    "add.s64 b1, %2, 1030;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t"

// TS: A (P, bf16) in TMEM, 8 columns per k step; B is a 128-byte-swizzled MN-major tile
// whose k steps (16 rows of 128 bytes) lie 2 KB apart (128 in 16-byte units).
#define INKATTN_MMA_TS_K128 \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t" \
    "add.u32 a1, %1, 8;\n\t" \
    "add.s64 b1, %2, 128;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 16;\n\t" \
    "add.s64 b1, %2, 256;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 24;\n\t" \
    "add.s64 b1, %2, 384;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 32;\n\t" \
    "add.s64 b1, %2, 512;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 40;\n\t" \
    "add.s64 b1, %2, 640;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 48;\n\t" \
    "add.s64 b1, %2, 768;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t" \
    "add.u32 a1, %1, 56;\n\t" \
    "add.s64 b1, %2, 896;\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t"

#define INKATTN_K128_PROLOGUE \
    "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.u32 pt, 0, 0;\n\tsetp.ne.b32 pr, %7, 0;\n\t" \
    "elect.sync _|e, 0xffffffff;\n\tand.pred pr, pr, e;\n\t"
#define INKATTN_K128_COMMITS(MC) \
    "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t" \
    "@pr tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster" MC ";\n\t}"

template <bool kMc>
__device__ __forceinline__ void mma_bf16_ss_k128_commit(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                                         uint32_t acc0, uint32_t bar, uint32_t rel_bar = 0,
                                                         uint32_t rel = 0, uint16_t rel_mask = 0) {
    if constexpr (kMc) {
        asm volatile("{\n\t.reg .pred e, p0, pt, pr;\n\t.reg .b64 a1, b1;\n\t" INKATTN_K128_PROLOGUE
                     INKATTN_MMA_SS_K128 INKATTN_K128_COMMITS(".multicast::cluster.b64 [%6], %8")
                     :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc0), "r"(bar), "r"(rel_bar), "r"(rel),
                        "h"(rel_mask) : "memory");
    } else {
        asm volatile("{\n\t.reg .pred e, p0, pt, pr;\n\t.reg .b64 a1, b1;\n\t" INKATTN_K128_PROLOGUE
                     INKATTN_MMA_SS_K128 INKATTN_K128_COMMITS(".b64 [%6]")
                     :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc0), "r"(bar), "r"(rel_bar), "r"(rel),
                        "h"(rel_mask) : "memory");
    }
}

template <bool kMc>
__device__ __forceinline__ void mma_bf16_ts_k128_commit(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                                         uint32_t acc0, uint32_t bar, uint32_t rel_bar = 0,
                                                         uint32_t rel = 0, uint16_t rel_mask = 0) {
    if constexpr (kMc) {
        asm volatile("{\n\t.reg .pred e, p0, pt, pr;\n\t.reg .b32 a1;\n\t.reg .b64 b1;\n\t" INKATTN_K128_PROLOGUE
                     INKATTN_MMA_TS_K128 INKATTN_K128_COMMITS(".multicast::cluster.b64 [%6], %8")
                     :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc0), "r"(bar), "r"(rel_bar), "r"(rel),
                        "h"(rel_mask) : "memory");
    } else {
        asm volatile("{\n\t.reg .pred e, p0, pt, pr;\n\t.reg .b32 a1;\n\t.reg .b64 b1;\n\t" INKATTN_K128_PROLOGUE
                     INKATTN_MMA_TS_K128 INKATTN_K128_COMMITS(".b64 [%6]")
                     :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc0), "r"(bar), "r"(rel_bar), "r"(rel),
                        "h"(rel_mask) : "memory");
    }
}

// ---------------------------------------------------------------- TMEM <-> registers
// 32x32b shape: thread i of the warp reads/writes TMEM lane (quarter base + i), 32
// consecutive 32-bit columns starting at the address's column.

__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace inkattn
