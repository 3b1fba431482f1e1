// prologue.cu -- the fused attention prologue: K/V ShortConv (W = 4) with conv-state
// carry, Q/K RMSNorm and the paged KV-cache write, in one kernel.
//
// [SGLang と Miles が Inkling を初日からサポート, §ShortConv 最適化：融合、グラフキャプチャ、
//  シャーディング]: K/V convolution, Q/K RMSNorm and the KV-cache write fused into one
//  attention-prologue kernel with no intermediate write-back.
// [same page, §ShortConv：4カ所に現れる短距離因果畳み込み]: per-channel causal conv along the
//  tokens over the current token and the W-1 = 3 previous positions.
// [vLLM hỗ trợ TML Inkling ..., §Quản lý bộ nhớ đệm sconv]: the state keeps the hidden
//  states of the last W-1 tokens.
//
// The conv sum of each channel is formed exactly (error-free products and sums in fp32)
// and rounded once to bf16, which is the correctly rounded value of the definition.
//
// Work split: two CTAs per (16-token tile of one sequence, KV head hk), neighbours in the
// grid.  One streams the tile's query rows of the g = Hq/Hkv query heads of hk (RMSNorm
// only; eight rows per half-warp in flight).  The other takes the K and V streams of head
// hk: it stages the tile's input rows and the three rows before it in shared memory once,
// then computes the conv (rounded to bf16), the K RMSNorm and the cache writes.  The
// latency-bound K/V work thus runs beside the bandwidth-bound query stream, four CTAs per
// SM.  Each 128-value row is owned by a half-warp: 16 lanes x 16 bytes, so every global
// access is a full 256-byte row, coalesced.

// Conv-state carry without races: tiles are aligned to sequence starts, so every read of
// the carried rows (tokens 0..2) happens in the K/V CTA of tile 0 of the sequence; that
// same CTA, after a block barrier, writes the new state for its own 128 channels.  No other
// CTA touches those channels of that state slot.
#include "common.cuh"
#include "conv4.cuh"
#include "fp8.cuh"
#include "internal.h"

namespace inkattn {

constexpr int kPrologueTokens = 16;      // tokens of a query-stream CTA
constexpr int kKvTilesMax = 4;           // query tiles per K/V CTA: 2, or 4 for large grids
constexpr int kKvTokens = kKvTilesMax * kPrologueTokens;   // most tokens of a K/V CTA
constexpr int kPrologueThreads = 256;
static_assert(kPrologueThreads == 256, "the row mapping assumes 16 half-warps per CTA");
constexpr int kQInFlight = 8;      // query rows a half-warp loads before it computes

__global__ void __launch_bounds__(kPrologueThreads, 4)
k_prologue(const inkattn_prologue_params p, const int kv_tiles) {
    __shared__ __align__(16) float s_wk[kHeadDim * 4];
    __shared__ __align__(16) float s_wv[kHeadDim * 4];
    __shared__ float s_gk[kHeadDim];
    // this head's K and V input rows [t0 - 3, t0 + nt) of [3 carried rows ; new rows]
    __shared__ uint4 s_x[2][kKvTokens + 3][16];
    grid_dep_wait();                                   // inputs written by the work before
    grid_dep_launch();                                 // the attention may be scheduled

    // Groups of kv_tiles + 1 neighbouring CTAs along x: the first kv_tiles stream the query
    // rows of one 16-token tile each (RMSNorm only); the last takes the K and V rows of the
    // group's 16 * kv_tiles tokens (conv, norm, cache write, state carry).  The
    // latency-bound K/V work thus runs beside the bandwidth-bound query stream.
    const int grp = blockIdx.x / (kv_tiles + 1), sub = blockIdx.x - grp * (kv_tiles + 1);
    const int role_kv = sub == kv_tiles, b = blockIdx.y, hk = blockIdx.z;
    const int tile = role_kv ? grp * kv_tiles : grp * kv_tiles + sub;
    const int tid = threadIdx.x;
    const int C = p.Hkv * kHeadDim;
    const int g = p.Hq / p.Hkv;

    const int start = p.cu_seqlens_q[b];
    const int end = p.cu_seqlens_q[b + 1];
    const int slot = p.state_slot[b];
    if (start < 0 || end < start || end > p.N_tok || end - start > p.max_seqlen_q ||
        slot < 0 || slot >= p.num_state_slots) {
        if (tid == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;   // uniform over the CTA
    }
    const int q_len = end - start;
    const int t0 = tile * kPrologueTokens;
    if (t0 >= q_len) return;   // (an empty sequence keeps its state unchanged)
    const int nt = min(role_kv ? kv_tiles * kPrologueTokens : kPrologueTokens, q_len - t0);

    const int half = tid >> 4;                // 16 half-warps per CTA
    const int lane16 = tid & 15;
    const int c0 = lane16 * 8;                // 8 channels per lane within the head

    if (!role_kv) {
        // ======================= query rows: RMSNorm, kQInFlight rows per lane in flight
        const int q_rows = nt * g;
        // the tile's query rows from one base: 32-bit offsets within the tile
        const size_t q_base = (size_t)(start + t0) * p.Hq * kHeadDim;
        const inkattn_bf16 *qb = p.q + q_base;
        inkattn_bf16 *ob = p.q_out + q_base;
        const int g_shift = (g & (g - 1)) == 0 ? __ffs(g) - 1 : -1;
        auto div_g = [&](int row) { return g_shift >= 0 ? row >> g_shift : row / g; };
        // the gains need only 4-byte alignment: scalar loads
        float2 gq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            gq[e] = make_float2(__ldg(p.q_norm_w + c0 + 2 * e), __ldg(p.q_norm_w + c0 + 2 * e + 1));
        for (int j0 = 0; j0 * 16 < q_rows; j0 += kQInFlight) {   // uniform over the CTA
            uint4 qraw[kQInFlight];
#pragma unroll
            for (int j = 0; j < kQInFlight; ++j) {
                const int row = half + 16 * (j0 + j);
                qraw[j] = make_uint4(0, 0, 0, 0);
                if (row < q_rows) {
                    const int tt = div_g(row), h = hk * g + (row - tt * g);
                    qraw[j] = __ldg(reinterpret_cast<const uint4 *>(
                        qb + (uint32_t)((tt * p.Hq + h) * kHeadDim + c0)));
                }
            }
#pragma unroll
            for (int j = 0; j < kQInFlight; ++j) {
                const int row = half + 16 * (j0 + j);
                float x[8];
                unpack8(qraw[j], x);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (row >= q_rows) continue;
                const int tt = div_g(row), h = hk * g + (row - tt * g);
                const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
                const float2 inv2 = make_float2(inv, inv);
                float y[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 v = fmul2(fmul2(make_float2(x[2 * e], x[2 * e + 1]), inv2), gq[e]);
                    y[2 * e] = v.x;
                    y[2 * e + 1] = v.y;
                }
                *reinterpret_cast<uint4 *>(ob + (uint32_t)((tt * p.Hq + h) * kHeadDim + c0)) =
                    pack8(y);
            }
        }
        return;
    }

    // ======================= K and V rows
    // conv weights and the K gains, interleaved by lane: channel c = 8 * lane + e, tap k at
    // [(e * 16 + lane) * 4 + k], so the 16 lanes of a half-warp read consecutive float4s.
    // Consecutive threads fill consecutive entries (no bank conflicts), each from the
    // channel and tap that entry holds.
    for (int j = tid; j < kHeadDim * 4; j += kPrologueThreads) {
        const int q = j >> 2, k = j & 3;
        const int c = ((q & 15) << 3) + (q >> 4);
        const size_t src = ((size_t)hk * kHeadDim + c) * 4 + k;
        s_wk[j] = p.conv_w_k[src];
        s_wv[j] = p.conv_w_v[src];
    }
    if (tid < kHeadDim) s_gk[tid] = p.k_norm_w[((tid & 15) << 3) + (tid >> 4)];
    // one 16-byte chunk of one row of both streams per step (no division by the row count)
    for (int i = tid; i < (nt + 3) * 16; i += kPrologueThreads) {
        const int r = i >> 4, chunk = i & 15;
        const int idx = t0 + r;               // index into [3 carried rows ; new rows]
        const size_t ch = (size_t)hk * kHeadDim + chunk * 8;
        uint4 vk, vv;
        if (idx < 3) {
            const size_t o = ((size_t)slot * 3 + idx) * C + ch;
            vk = *reinterpret_cast<const uint4 *>(p.conv_state_k + o);
            vv = *reinterpret_cast<const uint4 *>(p.conv_state_v + o);
        } else {
            const size_t o = ((size_t)start + idx - 3) * C + ch;
            vk = __ldg(reinterpret_cast<const uint4 *>(p.k + o));
            vv = __ldg(reinterpret_cast<const uint4 *>(p.v + o));
        }
        s_x[0][r][chunk] = vk;
        s_x[1][r][chunk] = vv;
    }
    // slot mapping of the rows this half-warp writes (tokens half&7 + 8u): lane u of the
    // half-warp fetches the one for step u before the barrier, so the cache write neither
    // waits for it nor selects it from a register array
    constexpr int kRowsPerHalf = kKvTokens / 8;
    static_assert(kRowsPerHalf <= 16, "one entry per lane of a half-warp");
    int sm_mine = 0;
    {
        const int tt = lane16 * 8 + (half & 7);
        if (lane16 < kRowsPerHalf && tt < nt) sm_mine = __ldg(p.slot_mapping + start + t0 + tt);
    }
    __syncthreads();

    // conv (rounded to bf16), K RMSNorm, cache write.  Half-warps 0-7 take the K stream and
    // 8-15 the V stream.
    const long long slot_limit = (long long)p.num_blocks * kBlock;
    const bool f8 = p.kv_dtype == INKATTN_KV_E4M3;
    const int stream = half >> 3;
    const float *wsm = stream == 0 ? s_wk : s_wv;
#pragma unroll 1
    for (int u = 0; u < kRowsPerHalf; ++u) {         // uniform trip count: all lanes shuffle
        if (u * 8 >= nt) break;                      // uniform over the CTA
        const int tt = u * 8 + (half & 7);
        const bool valid = tt < nt;
        const int ts = valid ? tt : 0;
        float xt[4][8];
#pragma unroll
        for (int tap = 0; tap < 4; ++tap) unpack8(s_x[stream][ts + tap][lane16], xt[tap]);
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float4 wa = *reinterpret_cast<const float4 *>(wsm + (e * 16 + lane16) * 4);
            const float4 wb = *reinterpret_cast<const float4 *>(wsm + ((e + 1) * 16 + lane16) * 4);
            const float wea[4] = {wa.x, wa.y, wa.z, wa.w}, web[4] = {wb.x, wb.y, wb.z, wb.w};
            const float xea[4] = {xt[0][e], xt[1][e], xt[2][e], xt[3][e]};
            const float xeb[4] = {xt[0][e + 1], xt[1][e + 1], xt[2][e + 1], xt[3][e + 1]};
            conv4_bf16_fast2(wea, xea, web, xeb, x[e], x[e + 1]);
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        // the row this stream stores: the normalised K or the conv'd V, rounded to bf16
        uint4 row;
        if (stream == 0) {
            const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = x[e] * inv * s_gk[e * 16 + lane16];
            row = pack8(y);
        } else {
            row = pack8(x);
        }
        // E4M3 cache: one power-of-two scale per row (the half-warp's 128 values)
        uint2 codes = make_uint2(0, 0);
        float row_scale = 1.f;
        if (f8) {
            float r8[8];
            unpack8(row, r8);
            float am = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(r8[e]));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 8));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            const int k = e4m3_row_exponent(am);
            row_scale = pow2f(k);
            codes = e4m3_encode8(r8, pow2f(-k));
        }
        const int sm = __shfl_sync(0xffffffffu, sm_mine, ((half & 1) << 4) + u);
        if (!valid) continue;
        if (sm < 0 || (long long)sm >= slot_limit) {
            if (lane16 == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
            continue;
        }
        const size_t drow = ((size_t)(sm / kBlock) * p.Hkv + hk) * kBlock + (sm % kBlock);
        const size_t dst = drow * kHeadDim + c0;
        void *cache = stream == 0 ? p.k_cache : p.v_cache;
        if (!f8) {
            *reinterpret_cast<uint4 *>(static_cast<inkattn_bf16 *>(cache) + dst) = row;
        } else {
            *reinterpret_cast<uint2 *>(static_cast<unsigned char *>(cache) + dst) = codes;
            if (lane16 == 0) (stream == 0 ? p.k_scale : p.v_scale)[drow] = row_scale;
        }
    }

    // new conv state = the last 3 rows of [carried rows ; new rows], for this head's channels
    if (tile != 0) return;
    uint4 nv = make_uint4(0, 0, 0, 0);
    int task = tid;                              // 2 streams x 3 rows x 16 chunks
    const bool active = task < 2 * 3 * 16;
    const int sstream = task / 48, r = (task / 16) % 3, chunk = task % 16;
    const size_t ch = (size_t)hk * kHeadDim + chunk * 8;
    inkattn_bf16 *st = sstream == 0 ? p.conv_state_k : p.conv_state_v;
    if (active) {
        const int idx = q_len + r;
        if (idx < 3) {
            nv = *reinterpret_cast<const uint4 *>(st + ((size_t)slot * 3 + idx) * C + ch);
        } else {
            const inkattn_bf16 *src = sstream == 0 ? p.k : p.v;
            nv = __ldg(reinterpret_cast<const uint4 *>(src + ((size_t)start + idx - 3) * C + ch));
        }
    }
    __syncthreads();   // every read of the old state (the staged rows and the rows above) is done
    if (active) *reinterpret_cast<uint4 *>(st + ((size_t)slot * 3 + r) * C + ch) = nv;
}

cudaError_t launch_prologue(const inkattn_prologue_params &p, cudaStream_t stream) {
    const int tiles = p.max_seqlen_q > 0 ? (p.max_seqlen_q + kPrologueTokens - 1) / kPrologueTokens : 1;
    // larger K/V groups amortise their fixed cost on large grids; smaller ones keep the
    // K/V work spread out on short ones
    const int kv_tiles = ((long long)tiles * p.B >= 2048) ? 4 : 2;
    const int groups = (tiles + kv_tiles - 1) / kv_tiles;
    dim3 grid(groups * (kv_tiles + 1), p.B, p.Hkv);
    return launch_dependent(k_prologue, grid, dim3(kPrologueThreads), 0, stream, 1, p, kv_tiles);
}

}  // namespace inkattn
