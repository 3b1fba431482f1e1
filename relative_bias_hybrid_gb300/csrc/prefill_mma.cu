// prefill_mma.cu -- relative-position-bias GQA prefill over the paged cache on the
// mma.sync tensor-core path.
//
// [SGLang と Miles が Inkling を初日からサポート, §相対位置バイアス付き Attention]: every logit
// gets the learned, query-conditioned bias r_i . P_h[:, i-j] for 0 <= i-j < rel_extent
// (zero beyond), future keys are masked; sliding-window and full layers are mixed, and
// full layers scale the logits with a length-dependent factor.
// [vLLM hỗ trợ TML Inkling ..., §FA4 với sheared bias]: the relative term complicates the
// memory access pattern of the attention pipeline; the bias is applied as a sheared band.
//
// One CTA per (128-query tile of one sequence, query head h).  8 compute warps own 16
// query rows each; a producer warp loads the Q tile once and streams 64-key cache blocks
// (K and V, two 64x64 TMA boxes each, 128-byte swizzle) through a ring of stages.
// QK^T and PV are mma.sync m16n8k16 (bf16 in, fp32 accumulate); the softmax is online
// in the log2 domain.
//
// The sheared bias: for a warp whose rows start at position pw and a block starting at
// key j0, every distance i-j lies in [pw-j0-63, pw-j0+15], an 80-wide window.  If that
// window reaches below rel_extent, the warp computes R[a][c] = r_{pw+a} . P_h[:, dlo+c]
// (dlo = pw-j0-63) for its 16 rows and 80 distances on the tensor cores, writes it to
// its own shared-memory table, and reads the bias of element (a, key b) at column
// a + 63 - b: each row reads its own shifted window (the shear).  Blocks outside the
// band skip all of this.
#include "common.cuh"
#include "internal.h"

namespace inkattn {

constexpr int kPmStages = 4;
constexpr int kPmStageBytes = 4 * 8192;          // K lo, K hi, V lo, V hi
constexpr int kPmWarps = 8;                      // compute warps
constexpr int kPmThreads = (kPmWarps + 1) * 32;
constexpr int kPmRWidth = 80;
constexpr int kPmQOff = kPmStages * kPmStageBytes;          // 2 x 16 KB Q boxes
constexpr int kPmROff = kPmQOff + 2 * 16384;
constexpr int kPmBarOff = kPmROff + kPmWarps * 16 * kPmRWidth * 4;
constexpr int kPmSmem = kPmBarOff + (2 * kPmStages + 1) * 8 + 16;

struct PrefillArgs {
    inkattn_attn_params p;
    float c_qk_base;        // softmax_scale * log2(e)
    int n_tiles_max;        // gridDim.x
};

__global__ void __launch_bounds__(kPmThreads, 1)
k_prefill_mma(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
              const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const inkattn_attn_params &p = a.p;
    const int tile = a.n_tiles_max - 1 - (int)blockIdx.x;   // longest tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = p.Hq / p.Hkv, hk = h / g;

    const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1];
    const int T = p.seqlen_k[b];
    const int q_len = end - start;
    if (start < 0 || end < start || end > p.N_tok || q_len > p.max_seqlen_q || T < q_len ||
        T > p.max_seqlen_k) {
        if (threadIdx.x == 0 && tile == 0 && h == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const int row0 = tile * kPrefillMmaRows;         // first query row of the tile (in the sequence)
    if (row0 >= q_len) return;
    const int pos0 = T - q_len;                      // position of the sequence's first new token
    const int p_lo = pos0 + row0;
    const int p_hi = pos0 + min(q_len, row0 + kPrefillMmaRows) - 1;   // last valid row position
    int k_lo = 0;
    if (p.window > 0) k_lo = max(0, p_lo - p.window + 1);
    const int blk_lo = k_lo / kBlock, blk_hi = p_hi / kBlock;         // inclusive
    const int n_blk = blk_hi - blk_lo + 1;

    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar_full = s_base + kPmBarOff;
    const uint32_t bar_empty = bar_full + kPmStages * 8;
    const uint32_t bar_q = bar_empty + kPmStages * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPmBarOff + (2 * kPmStages + 1) * 8);
    if ((s_base & 1023u) != 0u) {      // the 128-byte-swizzled TMA boxes need 1024-byte alignment
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPmStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kPmWarps);
        }
        mbar_init(bar_q, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const float lam = (p.log_scale_base > 1.f) ? fmaxf(1.f, logf((float)T) / logf(p.log_scale_base)) : 1.f;
    const float c_qk = lam * a.c_qk_base;
    const float c_b = lam * kLog2e;
    const bool has_bias = p.rel_extent > 0;

    if (warp == kPmWarps) {
        // ============================ producer ============================
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            mbar_arrive_expect_tx(bar_q, 2 * 16384);
            tma_load_3d(s_base + kPmQOff, &qmap, 0, h, start + row0, bar_q);
            tma_load_3d(s_base + kPmQOff + 16384, &qmap, 64, h, start + row0, bar_q);
            for (int it = 0; it < n_blk; ++it) {
                const int st = it % kPmStages;
                if (it >= kPmStages &&
                    !mbar_wait(bar_empty + 8 * st, ((it / kPmStages) - 1) & 1, p.dev_status, abort_flag))
                    break;
                const int lb = blk_lo + it;
                int blk = lb < p.max_blocks_per_seq ? p.block_table[(size_t)b * p.max_blocks_per_seq + lb] : -1;
                if (blk < 0 || blk >= p.num_blocks) {
                    set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                    blk = 0;
                }
                const int row = (blk * p.Hkv + hk) * kBlock;
                const uint32_t dst = s_base + st * kPmStageBytes;
                const uint32_t fb = bar_full + 8 * st;
                mbar_arrive_expect_tx(fb, kPmStageBytes);
                tma_load_2d(dst, &kmap, 0, row, fb);
                tma_load_2d(dst + 8192, &kmap, 64, row, fb);
                tma_load_2d(dst + 16384, &vmap, 0, row, fb);
                tma_load_2d(dst + 24576, &vmap, 64, row, fb);
            }
            // nothing may still be landing in shared memory when the CTA exits
            mbar_wait(bar_q, 0, p.dev_status, abort_flag);
            for (int it = max(0, n_blk - kPmStages); it < n_blk; ++it)
                mbar_wait(bar_full + 8 * (it % kPmStages), (it / kPmStages) & 1, p.dev_status, abort_flag);
        }
        return;
    }

    // ============================ compute warps ============================
    const int gq = lane >> 2, tq = lane & 3;
    const int pw = p_lo + warp * 16;                    // position of this warp's row 0
    const int row_pos[2] = {pw + gq, pw + gq + 8};
    bool ok = mbar_wait(bar_q, 0, p.dev_status, abort_flag);

    // Q fragments are re-read per k-step from the two swizzled Q boxes (ldmatrix) and the
    // relative-feature fragments only in band blocks, to leave registers for O.
    const int q_row = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int q_cadd = (lane >> 4) << 3;
    float *r_tab = reinterpret_cast<float *>(smem + kPmROff) + warp * 16 * kPmRWidth;
    const float *Ph = has_bias ? p.P + (size_t)h * p.d_r * p.rel_extent : nullptr;

    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    for (int it = 0; it < n_blk; ++it) {
        const int st = it % kPmStages;
        if (ok && !mbar_wait(bar_full + 8 * st, (it / kPmStages) & 1, p.dev_status, abort_flag)) ok = false;
        if (!ok) break;                 // compute warps share no barrier inside the loop
        const uint32_t kbase = s_base + st * kPmStageBytes;
        const uint32_t vbase = kbase + 16384;
        const int j0 = (blk_lo + it) * kBlock;

        // skip blocks that no row of this warp can see
        const bool any_vis = (j0 <= pw + 15) && (p.window == 0 || (pw - (j0 + kBlock - 1)) < p.window);
        if (any_vis) {
            // ---- S = Q K^T (16 x 64)
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t box = kbase + (ks >> 2) * 8192;
                uint32_t qf[4];
                ldmatrix_x4(qf, s_base + kPmQOff + (ks >> 2) * 16384 + sw128_offset(q_row, (ks & 3) * 16 + q_cadd));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int col = (ks & 3) * 16 + (((lane >> 3) & 1) << 3);
                    uint32_t kb[4];
                    ldmatrix_x4(kb, box + sw128_offset(key, col));
                    mma_16816(s[2 * np], qf, kb[0], kb[1]);
                    mma_16816(s[2 * np + 1], qf, kb[2], kb[3]);
                }
            }
            // ---- sheared relative bias for band blocks
            const int dlo = pw - j0 - (kBlock - 1);
            const bool band = has_bias && dlo < p.rel_extent;
            if (band) {
                uint32_t rf[4][4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int rr = row0 + warp * 16 + gq + ((e & 1) << 3);   // row in the sequence
                        const int col = kk * 16 + 2 * tq + ((e >> 1) << 3);
                        rf[kk][e] = (kk * 16 < p.d_r && rr < q_len)
                            ? __ldg(reinterpret_cast<const uint32_t *>(
                                  p.r + ((size_t)(start + rr) * p.Hq + h) * p.d_r + col))
                            : 0u;
                    }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < kPmRWidth / 8; ++nt) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    const int dl = dlo + nt * 8 + gq;
                    const bool dv = dl >= 0 && dl < p.rel_extent;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (kk * 16 >= p.d_r) continue;
                        const int e0 = kk * 16 + 2 * tq;
                        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
                        if (dv) {
                            p0 = __ldg(Ph + (size_t)e0 * p.rel_extent + dl);
                            p1 = __ldg(Ph + (size_t)(e0 + 1) * p.rel_extent + dl);
                            p2 = __ldg(Ph + (size_t)(e0 + 8) * p.rel_extent + dl);
                            p3 = __ldg(Ph + (size_t)(e0 + 9) * p.rel_extent + dl);
                        }
                        mma_16816(acc, rf[kk], pack_bf16(p0, p1), pack_bf16(p2, p3));
                    }
                    const int c = nt * 8 + 2 * tq;
                    *reinterpret_cast<float2 *>(r_tab + gq * kPmRWidth + c) = make_float2(acc[0], acc[1]);
                    *reinterpret_cast<float2 *>(r_tab + (gq + 8) * kPmRWidth + c) = make_float2(acc[2], acc[3]);
                }
                __syncwarp();
            }
            // ---- scale, bias, mask, online softmax
            float mnew[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int i = row_pos[hr];
                const int a_row = gq + 8 * hr;
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kb_ = n * 8 + 2 * tq + e;
                        const int dist = i - (j0 + kb_);
                        float v = s[n][2 * hr + e] * c_qk;
                        if (band && dist < p.rel_extent && dist >= 0)
                            v = fmaf(r_tab[a_row * kPmRWidth + a_row + (kBlock - 1) - kb_], c_b, v);
                        const bool vis = dist >= 0 && (p.window == 0 || dist < p.window);
                        v = vis ? v : -INFINITY;
                        s[n][2 * hr + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mnew[hr] = fmaxf(m_run[hr], mx);
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float ref = mnew[hr] == -INFINITY ? 0.f : mnew[hr];
                const float corr = fast_exp2(m_run[hr] - ref);
                m_run[hr] = mnew[hr];
                float ls = 0.f;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const float e0 = fast_exp2(s[n][2 * hr] - ref);
                    const float e1 = fast_exp2(s[n][2 * hr + 1] - ref);
                    s[n][2 * hr] = e0;
                    s[n][2 * hr + 1] = e1;
                    ls += e0 + e1;
                }
                l_run[hr] = l_run[hr] * corr + ls;
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o[n][2 * hr] *= corr;
                    o[n][2 * hr + 1] *= corr;
                }
            }
            // ---- O += P V; keys past the sequence end contribute exact zeros
            const bool tail = j0 + kBlock > T;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t pf[4];
                pf[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
                pf[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
                pf[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pf[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
                const int krow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    const int dcol = np * 16 + ((lane >> 4) << 3);
                    uint32_t vb[4];
                    ldmatrix_x4_trans(vb, vbase + (dcol >> 6) * 8192 + sw128_offset(krow, dcol & 63));
                    if (tail) {
                        const int jb = j0 + kk * 16 + 2 * tq;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int jj = jb + ((e & 1) << 3);
                            uint32_t m = 0u;
                            if (jj < T) m |= 0x0000FFFFu;
                            if (jj + 1 < T) m |= 0xFFFF0000u;
                            vb[e] &= m;
                        }
                    }
                    mma_16816(o[2 * np], pf, vb[0], vb[1]);
                    mma_16816(o[2 * np + 1], pf, vb[2], vb[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // ---- epilogue: normalise and write the valid rows
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }
    if (!ok) return;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int rr = row0 + warp * 16 + gq + 8 * hr;
        if (rr >= q_len) continue;
        const size_t qrow = (size_t)(start + rr) * p.Hq + h;
        const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
        if (p.out_dtype == INKATTN_DTYPE_F32) {
            float *dst = static_cast<float *>(p.out) + qrow * kHeadDim;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
                    make_float2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
        } else {
            inkattn_bf16 *dst = static_cast<inkattn_bf16 *>(p.out) + qrow * kHeadDim;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * tq) =
                    pack_bf16(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
        }
        if (p.lse && tq == 0) {
            const float ref = m_run[hr] == -INFINITY ? 0.f : m_run[hr];
            p.lse[qrow] = l_run[hr] > 0.f ? (ref + log2f(l_run[hr])) * 0.6931471805599453f : -INFINITY;
        }
    }
}

cudaError_t launch_prefill_mma(const inkattn_attn_params &p, const AttnScalars &s,
                               const CUtensorMap &qmap, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, cudaStream_t stream) {
    PrefillArgs a;
    a.p = p;
    a.c_qk_base = s.scale * kLog2e;
    a.n_tiles_max = (p.max_seqlen_q + kPrefillMmaRows - 1) / kPrefillMmaRows;
    cudaError_t err = cudaFuncSetAttribute(k_prefill_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, kPmSmem);
    if (err != cudaSuccess) return err;
    dim3 grid(a.n_tiles_max, p.Hq, p.B);
    k_prefill_mma<<<grid, kPmThreads, kPmSmem, stream>>>(a, qmap, kmap, vmap);
    return cudaGetLastError();
}

}  // namespace inkattn
