// decode.cu -- the split combine of the decode path.
//
// [vLLM TML Inkling サポート, §低レイテンシコレクティブとカーネル "FA4 Kernel"]: the decode
// attention splits the KV length and merges the partial results afterwards.  Each split s
// leaves, per (token, query head), its normalised output o_s and its natural-log LSE lse_s
// (decode_tc.cu); the merge is lse = ln sum_s e^{lse_s}, o = sum_s e^{lse_s - lse} o_s.
#include "common.cuh"
#include "internal.h"

namespace inkattn {

// One warp per (token, query head): lse = ln sum_s exp(lse_s), out = sum_s exp(lse_s - lse) o_s.
__global__ void __launch_bounds__(256)
k_combine(const inkattn_attn_params p, int S, const float *__restrict__ ws_o,
          const float *__restrict__ ws_lse) {
    grid_dep_wait();                                   // the partials of the decode before it
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)p.N_tok * p.Hq) return;
    const float *ls = ws_lse + row * S;
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, ls[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int s = 0; s < S; ++s) {
            const float w = __expf(ls[s] - mx);
            if (w == 0.f) continue;
            const float4 v = *reinterpret_cast<const float4 *>(ws_o + (row * S + s) * kHeadDim + lane * 4);
            acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
            wsum += w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (p.out_dtype == INKATTN_DTYPE_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * kHeadDim + lane * 4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        uint2 pk;
        pk.x = pack_bf16(acc.x * inv, acc.y * inv);
        pk.y = pack_bf16(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(static_cast<inkattn_bf16 *>(p.out) + row * kHeadDim + lane * 4) = pk;
    }
    if (p.lse && lane == 0) p.lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

cudaError_t launch_combine(const inkattn_attn_params &p, int num_splits, const float *ws_o,
                           const float *ws_lse, cudaStream_t stream) {
    const long long rows = (long long)p.N_tok * p.Hq;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    return launch_dependent(k_combine, dim3(blocks), dim3(256), 0, stream, 1, p, num_splits, ws_o, ws_lse);
}

}  // namespace inkattn
