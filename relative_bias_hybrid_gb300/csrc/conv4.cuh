// conv4.cuh -- the W = 4 causal ShortConv of one channel, correctly rounded to bf16, and
// the bf16 row packing shared by the prologue and the attention-output conv.
//
// [SGLang と Miles が Inkling を初日からサポート, §ShortConv：4カ所に現れる短距離因果畳み込み]:
//  per-channel causal conv along the tokens over the current token and the W-1 = 3
//  previous positions of the same channel; the taps are ordered oldest first here
//  (w[0] weighs the token three back, w[3] the current token).
#pragma once
#include "common.cuh"

namespace inkattn {

__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z);
    x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]); u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]); u.w = pack_bf16(x[6], x[7]);
    return u;
}

// Exact-sum helpers for the conv: a*b = p + e exactly (fma), a + b = s + e exactly.
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
    p = a * b;
    e = fmaf(a, b, -p);
}
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// bf16 of the value hi + lo (|lo| <= half an fp32 ulp of hi), rounded to nearest even:
// rounding hi alone is right unless hi sits exactly on a bf16 tie, where lo decides.
__device__ __forceinline__ float round_pair_bf16(float hi, float lo) {
    const uint32_t u = __float_as_uint(hi);
    if ((u & 0xFFFFu) == 0x8000u && lo != 0.f) {
        const bool away = (lo > 0.f) == (hi > 0.f);
        return __uint_as_float(((u >> 16) + (away ? 1u : 0u)) << 16);
    }
    return __bfloat162float(__float2bfloat16_rn(hi));
}

// Correctly rounded bf16 of sum_{k=0..3} w[k]*x[k]: the products are split exactly and
// the running sum is carried as an unevaluated pair, so hi + lo equals the exact sum up
// to ~2^-47 of the largest term (fp32 accumulation alone can lose every bit of a
// strongly cancelling sum).
__device__ __forceinline__ float conv4_bf16(const float (&w)[4], const float (&x)[4]) {
    float s, c;
    two_prod(w[0], x[0], s, c);
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        float p, pe, t, te;
        two_prod(w[k], x[k], p, pe);
        two_sum(s, p, t, te);
        s = t;
        c += te + pe;
    }
    float hi, lo;
    two_sum(s, c, hi, lo);
    return round_pair_bf16(hi, lo);
}

// The same correctly rounded value, cheaply in almost every case: an fp32 multiply-add
// chain s is within 4u * sum|w_k x_k| of the exact sum (u = 2^-24), so when s is farther
// than 8u * sum|w_k x_k| from the nearest bf16 rounding boundary (the midpoint above or
// below it, or a quarter bf16 ulp when a power of two is near) its rounding is the exact
// sum's; otherwise the error-free path decides.
__device__ __forceinline__ float conv4_bf16_fast(const float (&w)[4], const float (&x)[4]) {
    const float s = fmaf(w[3], x[3], fmaf(w[2], x[2], fmaf(w[1], x[1], w[0] * x[0])));
    const float a = fmaf(fabsf(w[3]), fabsf(x[3]),
                         fmaf(fabsf(w[2]), fabsf(x[2]), fmaf(fabsf(w[1]), fabsf(x[1]), fabsf(w[0] * x[0]))));
    const float mid = __uint_as_float((__float_as_uint(s) & 0xFFFF0000u) | 0x8000u);
    if (fabsf(s - mid) * 2097152.f > a && fabsf(s) * 2048.f > a)        // 2^21, 2^11
        return __bfloat162float(__float2bfloat16_rn(s));
    return conv4_bf16(w, x);
}

// conv4_bf16_fast on two channels at once: the multiply-add chains and the sums of
// magnitudes run on paired fp32 instructions.
__device__ __forceinline__ void conv4_bf16_fast2(const float (&wa)[4], const float (&xa)[4],
                                                 const float (&wb)[4], const float (&xb)[4],
                                                 float &ya, float &yb) {
    float2 s = fmul2(make_float2(wa[0], wb[0]), make_float2(xa[0], xb[0]));
    // the sums of magnitudes in scalar form: the absolute values then ride on the
    // multiply-adds' operands instead of taking instructions of their own
    float2 a = make_float2(fabsf(s.x), fabsf(s.y));
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        s = ffma2(make_float2(wa[k], wb[k]), make_float2(xa[k], xb[k]), s);
        a.x = fmaf(fabsf(wa[k]), fabsf(xa[k]), a.x);
        a.y = fmaf(fabsf(wb[k]), fabsf(xb[k]), a.y);
    }
    // The exact sums lie within 2^-21 of the sums of magnitudes of s (the chain's error is
    // at most 4u of it, u = 2^-24; the margin also covers the rounding of the magnitudes'
    // own sum).  Rounding to nearest is monotonic, so when both ends of that interval
    // (computed rounding outwards) round to the same bf16, so does the exact sum: one
    // packed compare decides both channels.  Magnitudes below 2^-100 (where products can
    // lose bits to underflow) and anything non-finite take the error-free path.
    const float ea = a.x * 0x1p-21f, eb = a.y * 0x1p-21f;
    const uint32_t lo = pack_bf16(__fsub_rd(s.x, ea), __fsub_rd(s.y, eb));
    const uint32_t hi = pack_bf16(__fadd_ru(s.x, ea), __fadd_ru(s.y, eb));
    if (lo == hi && fminf(a.x, a.y) > 0x1p-100f) {
        ya = bf16_lo(lo);
        yb = bf16_hi(lo);
    } else {
        ya = conv4_bf16(wa, xa);
        yb = conv4_bf16(wb, xb);
    }
}

}  // namespace inkattn
