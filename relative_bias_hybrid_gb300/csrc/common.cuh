// common.cuh -- device helpers shared by the inkattn kernels (sm_103a).
//
// Everything here is plain PTX wrapped in inline functions: mbarriers with
// bounded waits, TMA tensor copies, clusters, mma.sync (fp16), bf16/fp16 packing, paired fp32.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/inkattn.h"
#include "internal.h"

namespace inkattn {

constexpr float kLog2e = 1.4426950408889634f;

// A device wait that has not completed after this many nanoseconds gives up,
// records INKATTN_ERR_DEVICE_TIMEOUT and lets the kernel wind down.  Kernels take the
// limit as an argument (this value unless a test of the failure path sets a shorter one).
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s
constexpr uint32_t kWaitSleepNs = 100000u;         // longest single suspension of a waiting thread

__device__ __forceinline__ void set_status(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch.  Every kernel of the library is launched so that it may
// start while the kernel before it on the stream is still running; grid_dep_wait() returns
// once that kernel has completed and its writes are visible (at once when there is none),
// and each kernel calls it before its first read of global memory.  grid_dep_launch() lets
// the next kernel on the stream be scheduled; the short HBM-bound kernels (prologue,
// attention-output conv) call it right after their wait, the attention kernels not at all
// (their successor launches when they exit), so a successor never takes SM room an
// attention CTA still needs.  Since a kernel triggers only after its own wait, a kernel
// that starts early still cannot overtake any work before its predecessor.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended (instead of returning at once) until
// the phase completes or about `ns` nanoseconds have passed, so a waiting warp takes no
// issue slots from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records a timeout) if it has not completed within limit_ns, or soon after *abort
// is set by another role of the same CTA.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *status,
                                          volatile int *abort, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (abort && *abort) return false;
        if (globaltimer() - t0 > limit_ns) {
            set_status(status, INKATTN_ERR_DEVICE_TIMEOUT);
            if (abort) *abort = 1;
            return false;
        }
    }
}

// Teardown wait for asynchronous work this CTA has already issued (TMA copies landing in
// its shared memory, tensor-core operations on its TMEM): unlike mbar_wait it does not
// stop when another role gives up, since the CTA may release neither while that work is in
// flight.  Still bounded by limit_ns: issued copies and MMAs complete in microseconds, and
// a phase that needs a copy nobody issued (a peer that gave up first) never completes.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, int32_t *status,
                                           uint64_t limit_ns) {
    return mbar_wait(bar, parity, status, nullptr, limit_ns);
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 1D bulk copy global -> shared: both addresses 16-byte aligned, bytes a multiple of 16;
// completes on the mbarrier's transaction count
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// As tma_load_2d, multicast: the box lands at the same shared-memory offset in every CTA
// of the cluster named in cta_mask, and each of those CTAs' mbarrier at `bar`'s offset
// receives the bytes that landed in that CTA.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void *map, int c0, int c1,
                                               uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of every CTA of the cluster; orders shared-memory writes (barrier
// initialisation included) before the peers' accesses after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- mma.sync and packing

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col)
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two floats -> packed fp16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 2^-k for the k that brings m (>= 0) to at most 2^15, 1 when m is below that: a scale by
// which values of magnitude <= m convert to fp16 without overflow (exact, being a power of 2)
__device__ __forceinline__ float fp16_prescale(float m) {
    const int e = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;   // floor(log2 m) for normal m
    const int k = e > 14 ? e - 14 : 0;
    return __uint_as_float((uint32_t)(127 - k) << 23);
}

// two floats -> packed bf16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- paired fp32 (sm_100 family)
// Two fp32 lanes per instruction (fma/add/mul .f32x2), each lane rounded to nearest even
// exactly like its scalar form.

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// max of three (one instruction on the sm_100 family)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------- 16-bit fixed-point bias
// The relative bias is staged in shared memory as 16-bit offset-binary fixed point,
// value = (u - 32768) * sigma, with sigma chosen per tile (or table row) from a bound on
// |bias|, so that the staged value keeps an absolute error of at most sigma / 2
// (16 bits over the bound) instead of fp16's 11 significant bits.
//
// Encoding: v = x / sigma must satisfy |v| < 32768.  Adding 1.5 * 2^23 + 32768 in fp32
// rounds v to the nearest integer (the spacing of floats there is 1) and leaves
// round(v) + 32768 in the low 16 bits of the result.
constexpr float kFixMagic = 12582912.0f + 32768.0f;
__device__ __forceinline__ float2 fix16_encode2(float2 x, float inv_sigma) {
    return ffma2(x, make_float2(inv_sigma, inv_sigma), make_float2(kFixMagic, kFixMagic));
}
__device__ __forceinline__ unsigned short fix16_bits(float encoded) {
    return (unsigned short)(__float_as_uint(encoded) & 0xFFFFu);
}
// The two values packed in w (low half first) as exact integers round(v): the bits are
// placed under the exponent of 2^23 (byte permute), giving 2^23 + u, and 2^23 + 32768 is
// subtracted exactly.
__device__ __forceinline__ float2 fix16_decode2(uint32_t w) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, %2, 0x7610;" : "=r"(lo) : "r"(w), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi) : "r"(w), "r"(0x4B000000u));
    return fadd2(make_float2(__uint_as_float(lo), __uint_as_float(hi)),
                 make_float2(-8421376.0f, -8421376.0f));
}

}  // namespace inkattn
