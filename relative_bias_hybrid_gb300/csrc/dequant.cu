// dequant.cu -- prefill over an E4M3 cache: the blocks a batch reads, expanded to bf16.
//
// [SGLang と Miles が Inkling を初日からサポート, §Relative Attention と FA4 経路] and
// [vLLM TML Inkling サポート, §フューチャーロードマップ]: FP8 for the global-attention layers'
// KV cache.  The cache format is that of fp8.cuh: E4M3 codes with one power-of-two scale
// per row (token, KV head).
//
// The bf16 prefill kernel loads K and V tiles by TMA straight into its tensor-core operands
// and has no shared memory left for a conversion stage.  So the blocks of an E4M3 cache that
// a batch reads, block_table[b][0 .. ceil(seqlen_k[b] / 64)), are first expanded into a bf16
// copy in the caller's workspace, in sequence order (block b * max_blocks_per_seq + j), with
// a block table of its own (-1 past each sequence's blocks); then the bf16 prefill runs on
// the copy.  code * scale is exact in bf16 (4 significant bits times a power of two inside
// bf16's range), so the prefill sees exactly the values the decode reads.  Rows past a
// sequence's end are written as zeros.  A row inside it whose scale lies outside
// [2^-24, 2^7] (or is NaN), or a block id out of range, is flagged as
// INKATTN_ERR_DEVICE_BOUNDS and written as zeros, as the decode reads it.
//
// One CTA per (block j of sequence b, stream K or V and KV head); 256 threads, thread =
// (row, quarter of the row's 128 codes): 32 codes in, 64 bytes of bf16 out.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace inkattn {

namespace {

constexpr int kDqThreads = 256;            // 64 rows x 4 quarters of 32 codes

// Two codes (byte 0 -> low half) times the row scale, as bf16x2: the E4M3 -> f16 conversion
// is exact, and so are the f32 product (a power of two) and the bf16 rounding of it.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes, float s) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
    __half2 h;
    *reinterpret_cast<__half2_raw *>(&h) = r;
    const float2 f = __half22float2(h);
    return pack_bf16(f.x * s, f.y * s);
}

}  // namespace

__global__ void __launch_bounds__(kDqThreads)
k_dequant_e4m3(const inkattn_attn_params p, inkattn_bf16 *k_out, inkattn_bf16 *v_out, int32_t *table_out) {
    grid_dep_wait();                                   // the cache: written by the prologue
    grid_dep_launch();
    const int j = blockIdx.x, b = blockIdx.y, z = blockIdx.z;
    const int stream = z / p.Hkv, hk = z - stream * p.Hkv;
    const int tid = threadIdx.x;
    const int T = p.seqlen_k[b];
    if (T < 0 || T > p.max_seqlen_k) {
        if (tid == 0 && j == 0 && z == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const bool inside = (long long)j * kBlock < T;
    const size_t nb = (size_t)b * p.max_blocks_per_seq + j;
    if (z == 0 && tid == 0) table_out[nb] = inside ? (int32_t)nb : -1;
    if (!inside) return;
    const int phys = __ldg(p.block_table + nb);
    const bool phys_ok = phys >= 0 && phys < p.num_blocks;
    if (!phys_ok && tid == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
    const int r = tid >> 2, qd = tid & 3;              // row of the block, quarter of the row
    uint4 o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_uint4(0, 0, 0, 0);
    if (phys_ok && (long long)j * kBlock + r < T) {
        const size_t src_row = ((size_t)phys * p.Hkv + hk) * kBlock + r;
        const float s = __ldg((stream == 0 ? p.k_scale : p.v_scale) + src_row);
        if (s >= 0x1p-24f && s <= 0x1p7f) {
            const unsigned char *codes =
                static_cast<const unsigned char *>(stream == 0 ? p.k_cache : p.v_cache) + src_row * kHeadDim + qd * 32;
            const uint4 c[2] = {__ldg(reinterpret_cast<const uint4 *>(codes)),
                                __ldg(reinterpret_cast<const uint4 *>(codes + 16))};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w[4] = {c[h].x, c[h].y, c[h].z, c[h].w};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t lo = w[2 * e], hi = w[2 * e + 1];
                    o[2 * h + e] = make_uint4(e4m3x2_to_bf16x2(lo, s), e4m3x2_to_bf16x2(lo >> 16, s),
                                              e4m3x2_to_bf16x2(hi, s), e4m3x2_to_bf16x2(hi >> 16, s));
                }
            }
        } else {
            set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>((stream == 0 ? k_out : v_out) +
                                           (((size_t)nb * p.Hkv + hk) * kBlock + r) * kHeadDim + qd * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = o[i];
}

cudaError_t launch_dequant_e4m3(const inkattn_attn_params &p, inkattn_bf16 *k_out, inkattn_bf16 *v_out,
                                int32_t *table_out, cudaStream_t stream) {
    dim3 grid(p.max_blocks_per_seq, p.B, 2 * p.Hkv);
    return launch_dependent(k_dequant_e4m3, grid, dim3(kDqThreads), 0, stream, 1, p, k_out, v_out, table_out);
}

}  // namespace inkattn
