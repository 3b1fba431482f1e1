// fp8.cuh -- KV-cache rows in OCP FP8 E4M3 with one power-of-two scale per row.
//
// [SGLang と Miles が Inkling を初日からサポート, §Relative Attention と FA4 経路]: the FA4
//  path runs in MXFP8; [vLLM TML Inkling サポート, §フューチャーロードマップ] and [vLLM hỗ trợ
//  TML Inkling ..., last section]: FP8 for the global-attention layers, to relieve compute
//  and the KV cache.
// A row of 128 values x is stored as codes c = E4M3(x / 2^k) (round to nearest even) and
// the scale 2^k, k the smallest integer >= -24 with 448 * 2^k >= max|x| (0 for a zero row);
// reading back gives c * 2^k exactly.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace inkattn {

// 2^k as fp32, k in [-126, 127]
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// The row exponent k.  With amax = m * 2^e, m in [1, 2), and 448 = 1.75 * 2^8:
// 448 * 2^k >= amax holds from k = e - 8 when m <= 1.75, from k = e - 7 otherwise.
__device__ __forceinline__ int e4m3_row_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    const uint32_t u = __float_as_uint(amax);
    const int e = (int)(u >> 23) - 127;            // a subnormal amax gives -127: clamped below
    const int k = e - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return k < -24 ? -24 : k;
}

// Eight codes of x * inv_scale (inv_scale = 2^-k, so the products are exact), byte e of the
// result = element e.
__device__ __forceinline__ uint2 e4m3_encode8(const float (&x)[8], float inv_scale) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = __nv_cvt_float2_to_fp8x2(make_float2(x[2 * i] * inv_scale, x[2 * i + 1] * inv_scale),
                                        __NV_SATFINITE, __NV_E4M3);
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Two codes (byte 0 -> low half) to f16, times an f16 scale held in both halves of s2.  The
// conversion is exact (E4M3 is a subset of f16); the product is exact unless it falls
// below f16's smallest subnormal.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t two_codes, __half2 s2) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
    __half2 h;
    *reinterpret_cast<__half2_raw *>(&h) = r;
    h = __hmul2(h, s2);
    return *reinterpret_cast<uint32_t *>(&h);
}

// The same expansion on the integer pipe: the E4M3 fields (exponent bias 7) moved into
// f16's (bias 15) give the code's value times 2^-8 for every finite code, subnormals
// included, so s2 must hold scale * 2^8.  `sel` picks the two code bytes of w
// (0x1404: bytes 0, 1; 0x3424: bytes 2, 3) and places them at bits 8-15 and 24-31.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled_bits(uint32_t w, uint32_t sel, __half2 s2_x256) {
    const uint32_t t = __byte_perm(w, 0u, sel);
    const uint32_t f = (t & 0x80008000u) | ((t >> 1) & 0x3F803F80u);
    __half2 h = *reinterpret_cast<const __half2 *>(&f);
    h = __hmul2(h, s2_x256);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace inkattn
