// output_conv.cu -- the attention-output ShortConv with the residual add and the RMSNorm of
// the new residual stream, in one kernel.
//
// [SGLang と Miles が Inkling を初日からサポート, §ShortConv：4カ所に現れる短距離因果畳み込み]:
//  the third ShortConv of a layer follows the attention output.
// [same page, §ShortConv 最適化：融合、グラフキャプチャ、シャーディング]: it sits on the residual
//  stream, and in decode the residual add and the RMSNorm are folded into the same kernel.
// [vLLM hỗ trợ TML Inkling ..., §TP sharding nhận biết sconv]: the unfused order is
//  o_proj output -> sconv -> residual connection -> RMSNorm.
//
// HBM-bound: per token it reads y and the residual row and writes h and out (8 D bytes).
// Work split: one CTA per (4-token tile of one sequence), all D channels; a thread owns
// channel groups of 8 (one 16-byte vector per row), g = tid, tid + 256, ...  For each of
// its groups it requests all the tile's input rows at once (7 rows of y: the tile's 4 and
// the 3 before it, and 4 residual rows), so a thread waits on memory once per group, and
// accumulates each token's sum of squares of h.  One block reduction gives the tile's
// inverse RMS values; the thread then reads back the h it wrote (L2-resident) and writes
// out.  The halo rows of y are L2 hits (the neighbouring tile reads them too).
//
// Conv-state carry without races: tiles are aligned to sequence starts and hold at least 3
// tokens, so only tile 0 of a sequence reads the carried rows, and the same CTA writes the
// new state.  Every element of the state, of h and of the residual is read and written by
// one thread, in that order, so h_out may be the residual array itself.
#include "common.cuh"
#include "conv4.cuh"
#include "internal.h"

namespace inkattn {

constexpr int kOcTokens = 4;        // tokens of a CTA
constexpr int kOcThreads = 256;
constexpr int kOcWarps = kOcThreads / 32;
static_assert(kOcTokens >= 3, "only tile 0 of a sequence may read the carried rows");

__device__ __forceinline__ uint32_t word(const uint4 &u, int e) {
    return e == 0 ? u.x : e == 1 ? u.y : e == 2 ? u.z : u.w;
}

__global__ void __launch_bounds__(kOcThreads, 2) k_output_conv(const inkattn_output_conv_params p) {
    __shared__ float s_red[kOcWarps][kOcTokens];
    __shared__ float s_inv[kOcTokens];
    grid_dep_wait();                                   // inputs written by the work before
    grid_dep_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    const int tile = blockIdx.x;
    const int start = p.cu_seqlens_q[b];
    const int end = p.cu_seqlens_q[b + 1];
    if (start < 0 || end < start || end > p.N_tok || end - start > p.max_seqlen_q) {
        if (tid == 0 && tile == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const int q_len = end - start;
    const int t0 = tile * kOcTokens;
    if (t0 >= q_len) return;            // (an empty sequence keeps its state)
    const int slot = p.state_slot[b];
    if (slot < 0 || slot >= p.num_state_slots) {
        if (tid == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const int nt = min(kOcTokens, q_len - t0);
    const int G = p.D >> 3;                              // channel groups of 8
    const uint4 *y = reinterpret_cast<const uint4 *>(p.y) + (size_t)start * G;
    const uint4 *res = reinterpret_cast<const uint4 *>(p.residual) + (size_t)(start + t0) * G;
    uint4 *h_out = reinterpret_cast<uint4 *>(p.h_out) + (size_t)(start + t0) * G;
    uint4 *out = reinterpret_cast<uint4 *>(p.out) + (size_t)(start + t0) * G;
    uint4 *state = reinterpret_cast<uint4 *>(p.conv_state) + (size_t)slot * 3 * G;

    float ss[kOcTokens];
#pragma unroll
    for (int u = 0; u < kOcTokens; ++u) ss[u] = 0.f;

    for (int g = tid; g < G; g += kOcThreads) {
        // every input row of the group is requested before any is used: xs rows
        // t0 .. t0 + nt + 2 (carried rows where the xs index is below 3) and the residual rows
        uint4 xr[kOcTokens + 3], rv[kOcTokens];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int xi = t0 + i;
            xr[i] = xi < 3 ? state[(size_t)xi * G + g] : __ldg(y + (size_t)(xi - 3) * G + g);
        }
#pragma unroll
        for (int j = 0; j < kOcTokens; ++j) {
            if (j < nt) {
                xr[3 + j] = __ldg(y + (size_t)(t0 + j) * G + g);
                rv[j] = res[(size_t)j * G + g];
            }
        }
        // Channel pairs (2 e, 2 e + 1) = word e of every row: each row word is unpacked once
        // and serves the (up to) four tokens whose window holds it.  The pair's taps are
        // loaded one pair ahead (L1/L2 hits: every CTA reads the same taps).
        const float4 *wp = reinterpret_cast<const float4 *>(p.conv_w) + (size_t)g * 8;
        float4 wa = __ldg(wp), wb = __ldg(wp + 1);
        uint32_t hp[kOcTokens][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float4 na = wa, nb = wb;
            if (e < 3) { na = __ldg(wp + 2 * e + 2); nb = __ldg(wp + 2 * e + 3); }
            float xa[kOcTokens + 3], xb[kOcTokens + 3];
#pragma unroll
            for (int i = 0; i < kOcTokens + 3; ++i) {
                const uint32_t u = word(xr[i], e);
                xa[i] = __uint_as_float(u << 16);
                xb[i] = __uint_as_float(u & 0xffff0000u);
            }
            const float ta[4] = {wa.x, wa.y, wa.z, wa.w}, tb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int j = 0; j < kOcTokens; ++j) {
                if (j < nt) {
                    const float xja[4] = {xa[j], xa[j + 1], xa[j + 2], xa[j + 3]};
                    const float xjb[4] = {xb[j], xb[j + 1], xb[j + 2], xb[j + 3]};
                    float ca, cb;
                    conv4_bf16_fast2(ta, xja, tb, xjb, ca, cb);
                    const uint32_t ru = word(rv[j], e);
                    // two bf16 values: their fp32 sum rounds to the same bf16 as the exact
                    // sum (exact unless the exponents are 17+ apart, and then the smaller is
                    // far below half a bf16 ulp of the larger)
                    const uint32_t hw = pack_bf16(__uint_as_float(ru << 16) + ca,
                                                  __uint_as_float(ru & 0xffff0000u) + cb);
                    hp[j][e] = hw;
                    const float ha = __uint_as_float(hw << 16), hb = __uint_as_float(hw & 0xffff0000u);
                    ss[j] = fmaf(ha, ha, fmaf(hb, hb, ss[j]));
                }
            }
            wa = na;
            wb = nb;
        }
#pragma unroll
        for (int j = 0; j < kOcTokens; ++j)
            if (j < nt) h_out[(size_t)j * G + g] = make_uint4(hp[j][0], hp[j][1], hp[j][2], hp[j][3]);
        // the new state: the last 3 rows of xs (tile 0 only; its reads of the old rows above
        // came first, in this thread)
        if (tile == 0) {
            uint4 nv[3];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int xi = q_len + i;
                nv[i] = xi < 3 ? state[(size_t)xi * G + g] : __ldg(y + (size_t)(xi - 3) * G + g);
            }
#pragma unroll
            for (int i = 0; i < 3; ++i) state[(size_t)i * G + g] = nv[i];
        }
    }

    // the tile's sums of squares, over all D channels
#pragma unroll
    for (int u = 0; u < kOcTokens; ++u) {
        float v = ss[u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_red[warp][u] = v;
    }
    __syncthreads();
    if (tid < kOcTokens) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kOcWarps; ++i) t += s_red[i][tid];
        s_inv[tid] = rsqrtf(t / (float)p.D + p.eps);
    }
    __syncthreads();

    for (int g = tid; g < G; g += kOcThreads) {
        uint4 hv[kOcTokens];
#pragma unroll
        for (int j = 0; j < kOcTokens; ++j)
            if (j < nt) hv[j] = h_out[(size_t)j * G + g];   // written above by this thread
        float gw[8];
        {
            const float4 *gp = reinterpret_cast<const float4 *>(p.norm_w) + (size_t)g * 2;
            const float4 v0 = __ldg(gp), v1 = __ldg(gp + 1);
            gw[0] = v0.x; gw[1] = v0.y; gw[2] = v0.z; gw[3] = v0.w;
            gw[4] = v1.x; gw[5] = v1.y; gw[6] = v1.z; gw[7] = v1.w;
        }
#pragma unroll
        for (int j = 0; j < kOcTokens; ++j) {
            if (j < nt) {
                float x[8];
                unpack8(hv[j], x);
                const float inv = s_inv[j];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = x[e] * inv * gw[e];
                __stcs(out + (size_t)j * G + g, pack8(x));
            }
        }
    }
}

cudaError_t launch_output_conv(const inkattn_output_conv_params &p, cudaStream_t stream) {
    const int tiles = (p.max_seqlen_q + kOcTokens - 1) / kOcTokens;
    dim3 grid(tiles, p.B);
    return launch_dependent(k_output_conv, grid, dim3(kOcThreads), 0, stream, 1, p);
}

}  // namespace inkattn
