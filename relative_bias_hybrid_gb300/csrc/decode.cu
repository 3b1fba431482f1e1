// decode.cu -- split-KV decode over the paged cache with the relative-position bias,
// and the split combine.
//
// [vLLM TML Inkling サポート, §低レイテンシコレクティブとカーネル "FA4 Kernel"] and
// [vLLM hỗ trợ TML Inkling ..., §FA4 với sheared bias]: the attention kernel splits the
// KV length (num_splits picked from batch size, TP size and KV length); the partial
// results are merged afterwards.
// [SGLang と Miles が Inkling を初日からサポート, §相対位置バイアス付き Attention]: the logit is
// the scaled dot product plus the bias r_i . P_h[:, i-j] for 0 <= i-j < rel_extent.
//
// One CTA per (split, KV head hk, sequence b).  Its rows are every (token t, query head
// h = hk*g + hh) pair of the sequence, packed as row = t*g + hh (72 rows for 9 MTP-verify
// tokens x 8 heads), so all query heads that share a KV head read each K/V block once.
// Rows are cut into 16-row tiles; each tile has two compute warps that take the two
// 32-key halves of every 64-key cache block and merge their softmax states at the end.
// A producer warp streams the blocks of the split with TMA (two 64x64 boxes for K and
// two for V, 128-byte swizzle) into a ring of shared-memory stages.
// QK^T and PV run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// For cache blocks within rel_extent of the queries, one warp per query head computes
// its relative rows R[t][delta] = r_t . P_h[:, delta] for the block's 80 distances with
// the tensor cores as well and shares them through shared memory.
#include "common.cuh"
#include "internal.h"

namespace inkattn {

constexpr int kDecStages = 4;
constexpr int kDecStageBytes = 4 * 8192;     // K lo, K hi, V lo, V hi boxes
constexpr int kDecQStride = kHeadDim * 2 + 16; // padded bf16 row (bytes), conflict-free ldmatrix
constexpr int kDecRWidth = 80;               // distances covered per block: 64 + 16

struct DecodeArgs {
    inkattn_attn_params p;
    float c_qk;          // lambda * softmax_scale * log2(e) applied to q.k  (per call: lambda is per sequence -> computed in kernel)
    int S;               // number of splits
    int mt;              // 16-row tiles
    int ql;              // max_seqlen_q (rows of the R table per head)
    float *ws_o;
    float *ws_lse;
};

struct DecodeSmem {
    int q_off, r_off, bar_off, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int mt, int ql, int g) {
    DecodeSmem L;
    int off = kDecStages * kDecStageBytes;                  // stage ring (1024-aligned at 0)
    const int merge = mt * (16 * kHeadDim * 4 + 2 * 16 * 4);
    if (merge > off) off = merge;                           // merge buffers reuse the ring
    L.q_off = off;
    off += mt * 16 * kDecQStride;
    L.r_off = off;
    off += g * ql * kDecRWidth * 4;
    off = (off + 15) & ~15;
    L.bar_off = off;
    off += 2 * kDecStages * 8 + 16;
    L.total = off;
    return L;
}

template <int MT>
__global__ void __launch_bounds__((2 * MT + 1) * 32, 1)
k_decode(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
         const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const inkattn_attn_params &p = a.p;
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int n_compute = 2 * MT;
    const int g = p.Hq / p.Hkv;
    const DecodeSmem L = decode_smem_layout(MT, a.ql, g);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar_full = s_base + L.bar_off;
    const uint32_t bar_empty = bar_full + kDecStages * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.bar_off + 2 * kDecStages * 8);

    // ---- sequence geometry (uniform over the CTA)
    const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1];
    const int T = p.seqlen_k[b];
    const int q_len = end - start;
    if (start < 0 || end < start || end > p.N_tok || q_len > a.ql || T < q_len ||
        T > p.max_seqlen_k || q_len * g > 16 * MT) {
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    if (q_len == 0) return;
    const int pos0 = T - q_len;                       // position of token 0
    int blk_first = 0;
    if (p.window > 0) blk_first = max(0, pos0 - p.window + 1) / kBlock;
    const int blk_end = (T + kBlock - 1) / kBlock;    // exclusive
    const int nblk = blk_end - blk_first;
    const int per = (nblk + a.S - 1) / a.S;
    const int my_lo = blk_first + split * per;
    const int my_hi = min(blk_end, my_lo + per);
    const int my_n = max(0, my_hi - my_lo);

    if ((s_base & 1023u) != 0u) {      // the 128-byte-swizzled TMA boxes need 1024-byte alignment
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, n_compute);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // ---- Q tile -> shared memory (rows t*g+hh), zero padding rows
    {
        const int rows = MT * 16;
        for (int idx = threadIdx.x; idx < rows * 16; idx += blockDim.x) {
            const int row = idx >> 4, chunk = idx & 15;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row < q_len * g) {
                const int t = row / g, hh = row - t * g;
                v = __ldg(reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)(start + t) * p.Hq + hk * g + hh) * kHeadDim + chunk * 8));
            }
            *reinterpret_cast<uint4 *>(smem + L.q_off + row * kDecQStride + chunk * 16) = v;
        }
    }
    __syncthreads();

    const float lam = (p.log_scale_base > 1.f) ? fmaxf(1.f, logf((float)T) / logf(p.log_scale_base)) : 1.f;
    const float c_qk = lam * a.c_qk;                 // applied to q.k (log2 domain)
    const float c_b = lam * kLog2e;                  // applied to the bias
    const bool has_bias = p.rel_extent > 0;

    if (warp == n_compute) {
        // ======================= producer =======================
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            for (int it = 0; it < my_n; ++it) {
                const int st = it % kDecStages;
                if (it >= kDecStages) {
                    if (!mbar_wait(bar_empty + 8 * st, ((it / kDecStages) - 1) & 1, p.dev_status, abort_flag))
                        break;
                }
                const int lb = my_lo + it;
                int blk = (lb < p.max_blocks_per_seq) ? p.block_table[(size_t)b * p.max_blocks_per_seq + lb] : -1;
                if (blk < 0 || blk >= p.num_blocks) {
                    set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                    blk = 0;
                }
                const int row = (blk * p.Hkv + hk) * kBlock;
                const uint32_t dst = s_base + st * kDecStageBytes;
                const uint32_t fb = bar_full + 8 * st;
                mbar_arrive_expect_tx(fb, kDecStageBytes);
                tma_load_2d(dst, &kmap, 0, row, fb);
                tma_load_2d(dst + 8192, &kmap, 64, row, fb);
                tma_load_2d(dst + 16384, &vmap, 0, row, fb);
                tma_load_2d(dst + 24576, &vmap, 64, row, fb);
            }
        }
        // wait for every issued stage to land before the CTA may exit
        __syncwarp();
        if (lane == 0) {
            for (int it = max(0, my_n - kDecStages); it < my_n; ++it)
                mbar_wait(bar_full + 8 * (it % kDecStages), (it / kDecStages) & 1, p.dev_status, abort_flag);
        }
    } else {
        // ======================= compute warps =======================
        const int mtile = warp >> 1, kh = warp & 1;
        const int gq = lane >> 2, tq = lane & 3;
        // Q fragments are re-read from shared memory per k-step (ldmatrix) to keep
        // the register budget for the output accumulators.
        const uint32_t q_addr = s_base + L.q_off +
            (mtile * 16 + (lane & 7) + (((lane >> 3) & 1) << 3)) * kDecQStride + ((lane >> 4) << 4);
        // row metadata for the two rows this thread holds (gq and gq+8)
        int row_t[2], row_hh[2], row_pos[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int rho = mtile * 16 + gq + hr * 8;
            if (rho < q_len * g) {
                row_t[hr] = rho / g;
                row_hh[hr] = rho - row_t[hr] * g;
                row_pos[hr] = pos0 + row_t[hr];
            } else {
                row_t[hr] = 0; row_hh[hr] = 0; row_pos[hr] = -1;   // padding row: sees nothing
            }
        }
        float* r_tab = reinterpret_cast<float *>(smem + L.r_off);

        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        bool ok = true;

        // A warp whose wait gave up keeps iterating without computing, so that every
        // compute warp still reaches each named barrier the same number of times.
        for (int it = 0; it < my_n; ++it) {
            const int st = it % kDecStages;
            if (ok && !mbar_wait(bar_full + 8 * st, (it / kDecStages) & 1, p.dev_status, abort_flag))
                ok = false;
            const uint32_t kbase = s_base + st * kDecStageBytes;
            const uint32_t vbase = kbase + 16384;
            const int j0 = (my_lo + it) * kBlock;

            // ---- S = Q K^T for this warp's 32 keys
            float s[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
            if (ok) {
    #pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t box = kbase + (ks >> 2) * 8192;
                    uint32_t qf[4];
                    ldmatrix_x4(qf, q_addr + ks * 32);
    #pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        const int key = kh * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                        const int col = (ks & 3) * 16 + (((lane >> 3) & 1) << 3);
                        uint32_t kb[4];
                        ldmatrix_x4(kb, box + sw128_offset(key, col));
                        mma_16816(s[2 * np], qf, kb[0], kb[1]);
                        mma_16816(s[2 * np + 1], qf, kb[2], kb[3]);
                    }
                }
            }

            // ---- relative bias for blocks within rel_extent of the queries
            const bool band = has_bias && (pos0 - (j0 + kBlock - 1) < p.rel_extent);
            const int dlo = pos0 - j0 - (kBlock - 1);   // distance at table column 0
            if (band) {
                named_bar_sync(1, n_compute * 32);      // previous block's table reads done
                for (int hh = warp; hh < g; hh += n_compute) {
                    const int h = hk * g + hh;
                    const float *Ph = p.P + (size_t)h * p.rel_extent * p.d_r;
                    const inkattn_bf16 *rh = p.r + ((size_t)start * p.Hq + h) * p.d_r;
                    uint32_t rf[4][4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int t = gq + ((e & 1) << 3);
                            const int col = kk * 16 + 2 * tq + ((e >> 1) << 3);
                            rf[kk][e] = (kk * 16 < p.d_r && t < q_len)
                                ? __ldg(reinterpret_cast<const uint32_t *>(rh + (size_t)t * p.Hq * p.d_r + col))
                                : 0u;
                        }
#pragma unroll
                    for (int nt = 0; nt < kDecRWidth / 8; ++nt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        const int dl = dlo + nt * 8 + gq;
                        const bool dv = dl >= 0 && dl < p.rel_extent;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (kk * 16 >= p.d_r) continue;
                            const int e0 = kk * 16 + 2 * tq;
                            float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
                            if (dv) {
                                const float2 lo = __ldg(reinterpret_cast<const float2 *>(Ph + (size_t)dl * p.d_r + e0));
                                const float2 hi = __ldg(reinterpret_cast<const float2 *>(Ph + (size_t)dl * p.d_r + e0 + 8));
                                p0 = lo.x; p1 = lo.y; p2 = hi.x; p3 = hi.y;
                            }
                            mma_16816(acc, rf[kk], pack_bf16(p0, p1), pack_bf16(p2, p3));
                        }
                        const int c = nt * 8 + 2 * tq;
                        if (gq < q_len) {
                            float *dst = r_tab + ((size_t)hh * a.ql + gq) * kDecRWidth + c;
                            dst[0] = acc[0]; dst[1] = acc[1];
                        }
                        if (gq + 8 < q_len) {
                            float *dst = r_tab + ((size_t)hh * a.ql + gq + 8) * kDecRWidth + c;
                            dst[0] = acc[2]; dst[1] = acc[3];
                        }
                    }
                }
                named_bar_sync(1, n_compute * 32);      // table complete
            }

            if (!ok) continue;
            // ---- scale, bias, mask, online softmax
            float mt_new[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float mx = -INFINITY;
                const int i = row_pos[hr];
#pragma unroll
                for (int n = 0; n < 4; ++n) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = j0 + kh * 32 + n * 8 + 2 * tq + e;
                        float v = s[n][2 * hr + e] * c_qk;
                        const int dist = i - j;
                        if (band && dist >= 0 && dist < p.rel_extent)
                            v = fmaf(r_tab[((size_t)row_hh[hr] * a.ql + row_t[hr]) * kDecRWidth +
                                           (dist - dlo)], c_b, v);
                        const bool vis = dist >= 0 && (p.window == 0 || dist < p.window);
                        v = vis ? v : -INFINITY;
                        s[n][2 * hr + e] = v;
                        mx = fmaxf(mx, v);
                    }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mt_new[hr] = fmaxf(m_run[hr], mx);
            }
            uint32_t pf[2][4];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float ref = mt_new[hr] == -INFINITY ? 0.f : mt_new[hr];
                const float corr = fast_exp2(m_run[hr] - ref);
                m_run[hr] = mt_new[hr];
                float ls = 0.f;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
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
            // P as A fragments: k-step kk covers keys kh*32 + kk*16 .. +15
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                pf[kk][0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
                pf[kk][1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
                pf[kk][2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pf[kk][3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            }

            // ---- O += P V (keys past the sequence end contribute exact zeros)
            const bool tail = j0 + kBlock > T;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int krow = kh * 32 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    const int dcol = np * 16 + ((lane >> 4) << 3);
                    uint32_t vb[4];
                    ldmatrix_x4_trans(vb, vbase + (dcol >> 6) * 8192 + sw128_offset(krow, dcol & 63));
                    if (tail) {
                        const int kbase_j = j0 + kh * 32 + kk * 16 + 2 * tq;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int jj = kbase_j + ((e & 1) << 3);
                            uint32_t m = 0u;
                            if (jj < T) m |= 0x0000FFFFu;
                            if (jj + 1 < T) m |= 0xFFFF0000u;
                            vb[e] &= m;
                        }
                    }
                    mma_16816(o[2 * np], pf[kk], vb[0], vb[1]);
                    mma_16816(o[2 * np + 1], pf[kk], vb[2], vb[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        }

        // ---- merge the two key halves of this row tile, then write
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
            l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
        }
        // all stages are consumed before the ring is reused for the merge
        named_bar_sync(2, n_compute * 32);
        float *mb = reinterpret_cast<float *>(smem) + mtile * (16 * kHeadDim + 32);
        if (kh == 1) {
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float *dst = mb + (gq + 8 * hr) * kHeadDim + n * 8 + 2 * tq;
                    dst[0] = o[n][2 * hr];
                    dst[1] = o[n][2 * hr + 1];
                }
            if (tq == 0) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    mb[16 * kHeadDim + gq + 8 * hr] = m_run[hr];
                    mb[16 * kHeadDim + 16 + gq + 8 * hr] = l_run[hr];
                }
            }
        }
        named_bar_sync(3 + mtile, 64);
        if (kh == 0 && ok) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int rho = mtile * 16 + gq + 8 * hr;
                const float m1 = mb[16 * kHeadDim + gq + 8 * hr];
                const float l1 = mb[16 * kHeadDim + 16 + gq + 8 * hr];
                const float m0 = m_run[hr];
                const float mm = fmaxf(m0, m1);
                const float ref = mm == -INFINITY ? 0.f : mm;
                const float w0 = fast_exp2(m0 - ref), w1 = fast_exp2(m1 - ref);
                const float l = l_run[hr] * w0 + l1 * w1;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                if (rho >= q_len * g) continue;
                const int t = rho / g, hh = rho - t * g;
                const size_t qrow = (size_t)(start + t) * p.Hq + hk * g + hh;
                const float lse_nat = l > 0.f ? (ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
                if (a.S == 1) {
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int c = n * 8 + 2 * tq;
                        const float *src = mb + (gq + 8 * hr) * kHeadDim + c;
                        const float v0 = (o[n][2 * hr] * w0 + src[0] * w1) * inv;
                        const float v1 = (o[n][2 * hr + 1] * w0 + src[1] * w1) * inv;
                        if (p.out_dtype == INKATTN_DTYPE_F32)
                            *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + qrow * kHeadDim + c) =
                                make_float2(v0, v1);
                        else
                            *reinterpret_cast<uint32_t *>(static_cast<inkattn_bf16 *>(p.out) + qrow * kHeadDim + c) =
                                pack_bf16(v0, v1);
                    }
                    if (p.lse && tq == 0) p.lse[qrow] = lse_nat;
                } else {
                    float *dst = a.ws_o + (qrow * a.S + split) * kHeadDim;
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int c = n * 8 + 2 * tq;
                        const float *src = mb + (gq + 8 * hr) * kHeadDim + c;
                        float2 v;
                        v.x = (o[n][2 * hr] * w0 + src[0] * w1) * inv;
                        v.y = (o[n][2 * hr + 1] * w0 + src[1] * w1) * inv;
                        *reinterpret_cast<float2 *>(dst + c) = v;
                    }
                    if (tq == 0) a.ws_lse[qrow * a.S + split] = lse_nat;
                }
            }
        }
    }
}

// One warp per (token, query head): lse = ln sum_s exp(lse_s), out = sum_s exp(lse_s - lse) o_s.
__global__ void __launch_bounds__(256)
k_combine(const inkattn_attn_params p, int S, const float *__restrict__ ws_o,
          const float *__restrict__ ws_lse) {
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

cudaError_t launch_decode(const inkattn_attn_params &p, const AttnScalars &sc, int num_splits,
                          float *ws_o, float *ws_lse, const CUtensorMap &kmap,
                          const CUtensorMap &vmap, cudaStream_t stream) {
    DecodeArgs a;
    a.p = p;
    a.c_qk = sc.scale * kLog2e;
    a.S = num_splits;
    a.ql = p.max_seqlen_q;
    a.mt = (p.max_seqlen_q * sc.group + 15) / 16;
    a.ws_o = ws_o;
    a.ws_lse = ws_lse;
    const DecodeSmem L = decode_smem_layout(a.mt, a.ql, sc.group);
    dim3 grid(num_splits, p.Hkv, p.B);
    switch (a.mt) {
#define INKATTN_DECODE_CASE(M)                                                                   \
    case M: {                                                                                    \
        cudaError_t err = cudaFuncSetAttribute(k_decode<M>,                                      \
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                               L.total);                                         \
        if (err != cudaSuccess) return err;                                                      \
        k_decode<M><<<grid, (2 * M + 1) * 32, L.total, stream>>>(a, kmap, vmap);                 \
        return cudaGetLastError();                                                               \
    }
        INKATTN_DECODE_CASE(1) INKATTN_DECODE_CASE(2) INKATTN_DECODE_CASE(3)
        INKATTN_DECODE_CASE(4) INKATTN_DECODE_CASE(5) INKATTN_DECODE_CASE(6)
        INKATTN_DECODE_CASE(7) INKATTN_DECODE_CASE(8)
#undef INKATTN_DECODE_CASE
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const inkattn_attn_params &p, int num_splits, const float *ws_o,
                           const float *ws_lse, cudaStream_t stream) {
    const long long rows = (long long)p.N_tok * p.Hq;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    k_combine<<<blocks, 256, 0, stream>>>(p, num_splits, ws_o, ws_lse);
    return cudaGetLastError();
}

int decode_smem_bytes(int max_seqlen_q, int group) {
    const int mt = (max_seqlen_q * group + 15) / 16;
    return decode_smem_layout(mt, max_seqlen_q, group).total;
}

}  // namespace inkattn
