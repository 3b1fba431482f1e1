// prefill_tc.cu -- relative-position-bias GQA prefill on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), sm_103a.
//
// [SGLang と Miles が Inkling を初日からサポート, §相対位置バイアス付き Attention]: every logit
// gets the learned, query-conditioned bias r_i . P_h[:, i-j] for 0 <= i-j < rel_extent and
// nothing beyond; future keys are masked; sliding-window and full layers are mixed; full
// layers scale the logits by a length-dependent factor.
// [same page, §Relative Attention と FA4 経路] and [vLLM hỗ trợ TML Inkling ..., §FA4 với
// sheared bias]: a warp-specialized attention kernel that applies the relative term as a
// sheared bias band.
//
// One CTA per (128-query tile of one sequence, query head).  Roles:
//   warp 0      producer: TMA loads of the Q tile and of 128-key K/V tiles (two 64-key
//               cache blocks, two 64-column boxes each, 128-byte swizzle) into a 3-slot
//               ring; the relative-projection windows (128 distances of P_h) for the band.
//   warp 1      MMA issuer (one lane): S = Q K^T (operands in shared memory), O += P V
//               (P read from TMEM), R = r P_h (tf32, both operands K-major) for the band.
//   warps 2-9   softmax: two warpgroups; row i (TMEM lane i) is shared by one thread of
//               each, which own its key columns [0, 64) and [64, 128).
// TMEM (512 columns): O [0,128) | S0 [128,256) | S1 [256,384) | R [384,512).  P (bf16)
// overwrites the first 64 columns of its S buffer.  S is double-buffered so Q K^T of the
// next tile runs while the softmax works on this one.
//
// Key tiles are walked nearest-first (from the diagonal outwards).  With D_n the offset
// i0 - j0 of tile n (i0 = the tile's first query position, j0 = the key tile's first key),
// row a of tile n needs distances D_n + a - b for its 128 keys b: a window that shifts with
// the row (the shear).  The windows of consecutive tiles abut, so the band is covered by
// chunks C_n = [D_n + 1, D_n + 128] of 128 distances, one new chunk per tile (plus
// C_{-1} = [D_0 - 127, D_0] before the first).  For each chunk the MMA warp computes
// R[a][x] = r_a . P_h[:, D_n + 1 + x] (M=128, N=128, K=d_r) into TMEM.  Row a owns one
// row of a 128-entry fp16 buffer indexed by key column; it resolves the shear as it moves
// its values there: value x is the bias of column a - 1 - x in tile n when x < a (moved
// before tile n reads its bias) and of column a + 127 - x in tile n + 1 when x >= a (moved
// after).  Each tile then reads its bias row with sequential 16-byte loads.  Tiles farther
// than rel_extent skip all of this.
//
// The softmax runs in the log2 domain and keeps a stale row maximum unless the new one
// exceeds it by more than 8 (P stays below 2^8); only then is O rescaled in TMEM.  Column
// pairs go through paired fp32 instructions (fma/add .f32x2); three pairs in eight take a
// polynomial exp2 on the FMA pipe and the rest the special-function unit: 16 exp2 per clock
// per SM would alone take about as long as the MMAs of a tile, while the polynomial costs
// issue slots the softmax warps share.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace inkattn {

namespace {

constexpr int kRows = 128;                 // query rows per CTA (MMA M)
constexpr int kKeys = 128;                 // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kSlots = 3;                  // K/V ring slots
constexpr int kSlotBytes = 32768;          // one K or V tile: [d half][128 keys][128 B]
constexpr int kThreads = 320;            // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int kStageStride = 136;          // halves per row of the bias buffer
constexpr int kMaxDr = 32;                 // d_r (the relative features fill one 128-byte row)
constexpr int kPwinBytes = 128 * 128;      // [128 distances][32 fp32] (K-major)

constexpr int kOffQ = 0;
constexpr int kOffKV = 32768;
constexpr int kOffPwin = kOffKV + kSlots * kSlotBytes;
constexpr int kOffRfeat = kOffPwin + 2 * kPwinBytes;
constexpr int kOffStage = kOffRfeat + 16384;
constexpr int kOffXchg = kOffStage + kRows * kStageStride * 2;   // row maxima / sums of the two halves
constexpr int kOffBar = kOffXchg + 3 * 2 * kRows * 4;

enum Bar {
    B_Q = 0, B_KV_FULL = 1, B_KV_EMPTY = 4, B_S_FULL = 7, B_P_FULL = 9, B_PV_DONE = 11,
    B_R_FULL = 13, B_R_EMPTY = 14, B_PW_FULL = 15, B_PW_EMPTY = 17, B_RFEAT = 19, B_DRAIN = 20,
    B_PAIR = 21, B_COUNT = 25
};
constexpr int kSmem = kOffBar + B_COUNT * 8 + 16;

constexpr uint32_t kTmemO = 0, kTmemS0 = 128, kTmemR = 384;

struct TcArgs {
    inkattn_attn_params p;
    float scale;            // softmax scale
    int n_qtiles_max;       // gridDim.y
    long long kv_rows;      // rows of the cache tensor maps (OOB row = this)
};

__device__ __forceinline__ uint32_t sw128_chunk(int row, int chunk) {
    return (uint32_t)(row * 128 + (((chunk ^ row) & 7) << 4));
}

}  // namespace

template <int kCluster>
__global__ void __launch_bounds__(kThreads, 1)
k_prefill_tc(const TcArgs A, const __grid_constant__ CUtensorMap qmap,
             const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
             const __grid_constant__ CUtensorMap pmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const inkattn_attn_params &p = A.p;
    const int h = blockIdx.x, b = blockIdx.z;
    const int qt = A.n_qtiles_max - 1 - (int)blockIdx.y;     // longest tiles first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = p.Hq / p.Hkv, hk = h / g;
    // with kCluster = 2 the CTAs of heads 2i and 2i + 1 (same KV head) form a cluster; each
    // loads one 64-key half of every K/V tile and multicasts it to both
    const uint32_t crank = kCluster > 1 ? cluster_ctarank() : 0u;
    constexpr uint16_t kPeers = (uint16_t)((1u << kCluster) - 1u);

    // ---- sequence and tile geometry (uniform over the CTA)
    const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1];
    const int T = p.seqlen_k[b];
    const int q_len = end - start;
    if (start < 0 || end < start || end > p.N_tok || q_len > p.max_seqlen_q || T < q_len ||
        T > p.max_seqlen_k) {
        if (threadIdx.x == 0 && qt == 0 && h == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const int row0 = qt * kRows;
    if (row0 >= q_len) return;
    const int pos0 = T - q_len;
    const int p_lo = pos0 + row0;                                  // position of row 0
    const int p_hi = pos0 + min(q_len, row0 + kRows) - 1;          // last valid row
    const int k_lo = p.window > 0 ? max(0, p_lo - p.window + 1) : 0;
    const int t_hi = p_hi / kKeys, t_lo = k_lo / kKeys;
    const int N = t_hi - t_lo + 1;                                 // key tiles
    const bool has_bias = p.rel_extent > 0;
    int n_band = 0;
    if (has_bias) {
        // tile n is in the band iff its smallest distance D_n - 127 is below rel_extent
        const long long lim = (long long)p.rel_extent + 127 - (p_lo - (long long)kKeys * t_hi);
        const long long nb = (lim + kKeys - 1) / kKeys;
        n_band = lim <= 0 ? 0 : (nb < N ? (int)nb : N);
    }
    const int d_r = p.d_r;

    const uint32_t s_base = smem_u32(smem);
    if ((s_base & 1023u) != 0u) {
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    auto bar = [&](int i) { return s_base + kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + B_COUNT * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + B_COUNT * 8 + 4);
    // every lane waits; the outcome is made uniform over the warp, because the warps that
    // act on it next issue warp-collective (.sync.aligned) tcgen05 instructions
    auto wwait = [&](uint32_t addr, uint32_t parity) -> bool {
        const bool r = mbar_wait(addr, parity, p.dev_status, abort_flag);
        return __all_sync(0xffffffffu, r);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), kCluster);         // released by every CTA's MMAs
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 256);
            mbar_init(bar(B_PW_FULL + s), 1);
            mbar_init(bar(B_PW_EMPTY + s), 1);
            mbar_init(bar(B_PV_DONE + s), 1);
        }
        mbar_init(bar(B_R_FULL), 1);
        mbar_init(bar(B_R_EMPTY), 256);
        mbar_init(bar(B_RFEAT), 256);
        mbar_init(bar(B_DRAIN), 1);
        for (int q = 0; q < 4; ++q) mbar_init(bar(B_PAIR + q), 64);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if constexpr (kCluster > 1) cluster_sync();          // peers' barriers exist before any multicast
    const uint32_t tmem = *tmem_slot;

    const float lam = (p.log_scale_base > 1.f) ? fmaxf(1.f, logf((float)T) / logf(p.log_scale_base)) : 1.f;
    const float c_qk = lam * A.scale * kLog2e;       // S (with the bias folded in) -> log2 logit
    const float inv_scale = 1.f / A.scale;           // bias in S units

    if (warp == 0) {
        // ================================ producer ================================
        bool ok = true;
        const uint32_t q_dst = s_base + kOffQ;
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            if (n_band > 0) tma_prefetch_desc(&pmap);
            mbar_arrive_expect_tx(bar(B_Q), 2 * 16384);
            tma_load_3d(q_dst, &qmap, 0, h, start + row0, bar(B_Q));
            tma_load_3d(q_dst + 16384, &qmap, 64, h, start + row0, bar(B_Q));
        }
        // relative-projection window of chunk rho-1 (rho = 0 is C_{-1}): P_h rows of the 128
        // distances from D_{rho-1} + 1, one TMA box [128][d_r] fp32 that lands K-major with
        // the 128-byte swizzle, as the tf32 MMA reads it; distances outside [0, rel_extent)
        // are out of the tensor and arrive as zeros
        auto load_pwin = [&](int rho) -> bool {
            const int slot = rho & 1;
            if (rho >= 2 && !wwait(bar(B_PW_EMPTY + slot), ((rho >> 1) - 1) & 1))
                return false;
            if (lane == 0) {
                const int x0 = p_lo - kKeys * (t_hi - (rho - 1)) + 1;
                mbar_arrive_expect_tx(bar(B_PW_FULL + slot), kPwinBytes);
                tma_load_3d(s_base + kOffPwin + slot * kPwinBytes, &pmap, 0, x0, h, bar(B_PW_FULL + slot));
            }
            __syncwarp();
            return true;
        };
        int kv_loads = 0;                       // K/V tiles issued, in the MMA warp's order
        auto load_kv = [&](int n, int isv) -> bool {
            const int L = kv_loads++, slot = L % kSlots;
            if (L >= kSlots && !wwait(bar(B_KV_EMPTY + slot), ((L / kSlots) - 1) & 1))
                return false;
            if (lane == 0) {
                const int t = t_hi - n;
                const uint32_t dst = s_base + kOffKV + slot * kSlotBytes;
                const uint32_t fb = bar(B_KV_FULL + slot);
                mbar_arrive_expect_tx(fb, kSlotBytes);       // both halves land in every CTA
                const void *map = isv ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
#pragma unroll
                for (int hh = 0; hh < 3 - kCluster; ++hh) {
                    const int half = kCluster > 1 ? (int)crank : hh;
                    const int lb = 2 * t + half;                 // logical cache block
                    long long row = A.kv_rows;                   // past the tensor: TMA fills zeros
                    if ((long long)lb * kBlock < T) {
                        const int blk = lb < p.max_blocks_per_seq
                            ? p.block_table[(size_t)b * p.max_blocks_per_seq + lb] : -1;
                        if (blk >= 0 && blk < p.num_blocks) row = ((long long)blk * p.Hkv + hk) * kBlock;
                        else set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                    }
                    if constexpr (kCluster > 1) {
                        tma_load_2d_mc(dst + half * 8192, map, 0, (int)row, fb, kPeers);
                        tma_load_2d_mc(dst + 16384 + half * 8192, map, 64, (int)row, fb, kPeers);
                    } else {
                        tma_load_2d(dst + half * 8192, map, 0, (int)row, fb);
                        tma_load_2d(dst + 16384 + half * 8192, map, 64, (int)row, fb);
                    }
                }
            }
            __syncwarp();
            return true;
        };
        // the MMA warp consumes K_0, [W_1], then per tile n >= 1: K_n, [W_{n+1}], V_{n-1},
        // and finally V_{N-1} (W = relative-projection window); loading in that order lets
        // K_{n+1} reuse the slot of V_{n-2} instead of waiting for V_{n-1} to be consumed
        if (n_band > 0) ok = load_pwin(0);
        if (ok) ok = load_kv(0, 0);
        if (ok && 0 < n_band) ok = load_pwin(1);
        for (int n = 1; n < N && ok; ++n) {
            ok = load_kv(n, 0);
            if (ok && n < n_band) ok = load_pwin(n + 1);
            if (ok) ok = load_kv(n - 1, 1);
        }
        if (ok) ok = load_kv(N - 1, 1);
        // nothing may still be landing in shared memory when the CTA tears down
        if (lane == 0) {
            mbar_wait(bar(B_Q), 0, p.dev_status, abort_flag);
            for (int L = max(0, kv_loads - kSlots); L < kv_loads; ++L)
                mbar_wait(bar(B_KV_FULL + L % kSlots), (L / kSlots) & 1, p.dev_status, abort_flag);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        const uint32_t id_qk = tc::idesc(128, 128, tc::kFmtBF16, 0, 0);
        const uint32_t id_pv = tc::idesc(128, 128, tc::kFmtBF16, 0, 1);
        const uint32_t id_r = tc::idesc(128, 128, tc::kFmtTF32, 0, 0);
        // Base descriptors, built once; the per-k-step ones differ only in the start
        // address field (bits 0-13, 16-byte units), which never carries out of its 14 bits
        // since shared-memory addresses stay below 256 KB.
        const uint64_t dq = tc::sdesc_sw128(s_base + kOffQ, 16, 1024);
        uint64_t dk[kSlots], dv[kSlots];
#pragma unroll
        for (int sl = 0; sl < kSlots; ++sl) {
            dk[sl] = tc::sdesc_sw128(s_base + kOffKV + sl * kSlotBytes, 16, 1024);
            dv[sl] = tc::sdesc_sw128(s_base + kOffKV + sl * kSlotBytes, 16384, 1024);
        }
        const uint64_t dr = tc::sdesc_sw128(s_base + kOffRfeat, 16, 1024);
        const uint64_t dw0 = tc::sdesc_sw128(s_base + kOffPwin, 16, 1024);
        bool ok = wwait(bar(B_Q), 0);
        if (ok && n_band > 0) ok = wwait(bar(B_RFEAT), 0);

        auto issue_r = [&](int rho) -> bool {
            if (rho >= 1 && !wwait(bar(B_R_EMPTY), (rho - 1) & 1)) return false;
            const int slot = rho & 1;
            if (!wwait(bar(B_PW_FULL + slot), (rho >> 1) & 1)) return false;
            tc::fence_after();
            if (lane == 0) {
                const uint64_t dw = dw0 + (uint64_t)(slot * kPwinBytes >> 4);
                for (int kk = 0; kk < d_r / 8; ++kk)
                    tc::mma_tf32_ss(tmem + kTmemR, dr + (uint64_t)(kk * 2), dw + (uint64_t)(kk * 2), id_r, kk > 0);
                tc::commit(bar(B_R_FULL));
                tc::commit(bar(B_PW_EMPTY + slot));
            }
            __syncwarp();
            return true;
        };
        int kv_used = 0;                         // K/V tiles consumed, same order as loaded
        auto next_tile = [&](int &slot, bool &last) -> bool {
            const int L = kv_used++;
            slot = L % kSlots;
            last = L + kSlots >= 2 * N;          // no later load reuses the slot
            return wwait(bar(B_KV_FULL + slot), (L / kSlots) & 1);
        };
        // lane 0: the slot may be refilled once the MMAs issued so far have read it; a slot
        // with no later load is not released, so no arrival reaches a peer that has finished
        auto release = [&](int slot, bool last) {
            if (last) return;
            if constexpr (kCluster > 1) tc::commit_mc(bar(B_KV_EMPTY + slot), kPeers);
            else tc::commit(bar(B_KV_EMPTY + slot));
        };
        auto issue_pv = [&](int m) -> bool {
            if (!wwait(bar(B_P_FULL + (m & 1)), (m >> 1) & 1)) return false;
            int slot;
            bool last;
            if (!next_tile(slot, last)) return false;
            // keys at or past the sequence end inside a loaded block: zero their V rows so
            // that P = 0 there contributes exact zeros whatever the cache slots hold
            const int j0 = (t_hi - m) * kKeys;
            const int nvalid = min(kKeys, T - j0);
            const int nload = min(kKeys, (int)(((long long)((T + kBlock - 1) / kBlock)) * kBlock - j0));
            if (nvalid < nload) {
                unsigned char *vp = smem + kOffKV + slot * kSlotBytes;
                const int rows = nload - nvalid;
                for (int idx = lane; idx < rows * 16; idx += 32) {
                    const int key = nvalid + idx / 16, dh = (idx >> 3) & 1, ch = idx & 7;
                    *reinterpret_cast<uint4 *>(vp + dh * 16384 + (key >> 6) * 8192 + (key & 63) * 128 + ch * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc::fence_after();
            if (lane == 0) {
                const uint32_t ps = tmem + kTmemS0 + (uint32_t)(m & 1) * 128;
                const uint64_t db = dv[slot];
                tc::mma_bf16_ts(tmem + kTmemO, ps, db, id_pv, m > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < 8; ++kk)
                    tc::mma_bf16_ts(tmem + kTmemO, ps + kk * 8, db + (uint64_t)(kk * 128), id_pv, 1u);
                tc::commit(bar(B_PV_DONE + (m & 1)));
                release(slot, last);
            }
            __syncwarp();
            return true;
        };

        if (ok && n_band > 0) ok = issue_r(0);
        for (int n = 0; n < N && ok; ++n) {
            int slot;
            bool last;
            ok = next_tile(slot, last);
            if (!ok) break;
            tc::fence_after();
            if (lane == 0) {
                const uint32_t sd = tmem + kTmemS0 + (uint32_t)(n & 1) * 128;
                const uint64_t db = dk[slot];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    tc::mma_bf16_ss(sd, dq + off, db + off, id_qk, kk > 0 ? 1u : 0u);
                }
                tc::commit(bar(B_S_FULL + (n & 1)));
                release(slot, last);
            }
            __syncwarp();
            if (n < n_band) ok = issue_r(n + 1);
            if (ok && n >= 1) ok = issue_pv(n - 1);
        }
        if (ok) ok = issue_pv(N - 1);
        // every MMA of this CTA has completed before TMEM is released
        if (lane == 0) tc::commit(bar(B_DRAIN));
        __syncwarp();
        (void)wwait(bar(B_DRAIN), 0);
    } else {
        // ================================ softmax ================================
        // Two warpgroups share the 128 rows: warps 2-5 (half 0) and 6-9 (half 1) read the
        // same TMEM lane quarters; thread (half w, row a) owns key columns [64 w, 64 w + 64)
        // of row a.  The two threads of a row exchange row maxima (and, at the end, row
        // sums) through shared memory with a 64-thread named barrier per lane quarter.
        const int quad = warp & 3;
        const int hw = (warp - 2) >> 2;                       // column half
        const int a = quad * 32 + lane;                       // query row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int row = row0 + a;                             // row within the sequence
        const int i_pos = p_lo + a;
        const int cb = 64 * hw;                               // first key column of this thread
        __half *stage = reinterpret_cast<__half *>(smem + kOffStage) + a * kStageStride;
        float *xchg = reinterpret_cast<float *>(smem + kOffXchg);   // [2 tiles][2 halves][128 rows]
        // the two threads of each row meet on an mbarrier (a bounded wait, unlike bar.sync)
        int pair_phase = 0;
        auto pair_sync = [&]() -> bool {
            mbar_arrive(bar(B_PAIR + quad));
            return wwait(bar(B_PAIR + quad), (pair_phase++) & 1);
        };
        bool ok = true;

        if (n_band > 0) {
            // this row's relative features as fp32, K-major with the 128-byte swizzle; each
            // half writes 4 of the 8 16-byte chunks
            if (row < q_len) {
                const inkattn_bf16 *src = p.r + ((size_t)(start + row) * p.Hq + h) * d_r;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int cc = 2 * hw + c;                // 8-element group of the features
                    float4 f0 = make_float4(0.f, 0.f, 0.f, 0.f), f1 = f0;
                    if (cc * 8 < d_r) {
                        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src + cc * 8));
                        f0 = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
                        f1 = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
                    }
                    *reinterpret_cast<float4 *>(smem + kOffRfeat + sw128_chunk(a, 2 * cc)) = f0;
                    *reinterpret_cast<float4 *>(smem + kOffRfeat + sw128_chunk(a, 2 * cc + 1)) = f1;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<float4 *>(smem + kOffRfeat + sw128_chunk(a, 4 * hw + c)) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_RFEAT));
        }

        // Move this thread's half (positions [cb, cb + 64)) of the chunk in TMEM R (times
        // inv_scale) into the row's bias buffer, indexed by key column: value x of chunk C_n
        // is the bias of key column a - 1 - x in tile n (x < a, first part) and of key
        // column a + 127 - x in tile n + 1 (x >= a).
        auto drain = [&](bool first_part) {
            __half *base = stage + (first_part ? a - 1 : a + 127) - cb;
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tc::ld32(tmem + kTmemR + lane_off + cb + c * 32, r);
                tc::wait_ld();
                const int lim = a - cb - 32 * c;              // e < lim  <=>  x < a
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if ((e < lim) == first_part)
                        base[-(32 * c + e)] = __float2half_rn(__uint_as_float(r[e]) * inv_scale);
            }
        };

        float m_run = -INFINITY, l_run = 0.f;
        int r_round = 0;
        // P V of tile m signals PV_DONE[m & 1], phase m >> 1.  The MMA warp issues Q K^T of
        // tile m + 2 after P V of tile m, so once this thread has seen S of tile m + 2 the
        // phase before tile m's (tile m - 2) is complete: a parity wait is then unambiguous
        // without observing every phase, and the softmax waits only when it rescales O.
        auto wait_pv = [&](int m) -> bool { return wwait(bar(B_PV_DONE + (m & 1)), (m >> 1) & 1); };
        for (int n = 0; n < N; ++n) {
            if (!(ok = wwait(bar(B_S_FULL + (n & 1)), (n >> 1) & 1))) break;
            tc::fence_after();
            const uint32_t sbuf = tmem + kTmemS0 + (uint32_t)(n & 1) * 128 + lane_off;
            float s[64];
            {
                uint32_t *su = reinterpret_cast<uint32_t *>(s);
                tc::ld32(sbuf + cb, *reinterpret_cast<uint32_t(*)[32]>(su));
                tc::ld32(sbuf + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
                tc::wait_ld();
            }
            if (n < n_band) {
                if (n == 0) {
                    if (!(ok = wwait(bar(B_R_FULL), r_round & 1))) break;
                    tc::fence_after();
                    drain(false);                                 // C_{-1}: positions >= a
                    tc::fence_before();
                    mbar_arrive(bar(B_R_EMPTY));
                    ++r_round;
                }
                if (!(ok = wwait(bar(B_R_FULL), r_round & 1))) break;
                tc::fence_after();
                drain(true);                                      // C_n: positions < a
                if (!(ok = pair_sync())) break;                   // both halves moved
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(stage + cb + 8 * c8);
                    const __half2 *hp = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = fadd2(make_float2(s[8 * c8 + 2 * e], s[8 * c8 + 2 * e + 1]),
                                               __half22float2(hp[e]));
                        s[8 * c8 + 2 * e] = f.x;
                        s[8 * c8 + 2 * e + 1] = f.y;
                    }
                }
                if (!(ok = pair_sync())) break;                   // both halves read tile n
                drain(false);                                     // C_n: positions >= a (tile n+1)
                tc::fence_before();
                mbar_arrive(bar(B_R_EMPTY));
                ++r_round;
            }
            // mask and row maximum over this thread's 64 columns (unscaled; the scale is > 0)
            const int j0 = (t_hi - n) * kKeys;
            int b_lo, span;                                       // visible: (unsigned)(b - b_lo) <= span
            {
                const int jv_lo = p.window > 0 ? i_pos - p.window + 1 : 0;
                const int jv_hi = min(i_pos, T - 1);
                b_lo = jv_hi >= jv_lo ? jv_lo - j0 - cb : (1 << 20);
                span = jv_hi >= jv_lo ? jv_hi - jv_lo : 0;
            }
            const bool need_mask = (j0 + kKeys - 1 > p_lo) || (j0 + kKeys - 1 >= T) ||
                                   (p.window > 0 && p_lo + kRows - 1 - j0 >= p.window);
            if (need_mask) {
#pragma unroll
                for (int bb = 0; bb < 64; ++bb)
                    s[bb] = ((unsigned)(bb - b_lo) <= (unsigned)span) ? s[bb] : -INFINITY;
            }
            // four chains of three-input maxima over 16 columns each
            float m4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float m = fmax3(s[16 * c], s[16 * c + 1], s[16 * c + 2]);
#pragma unroll
                for (int e = 3; e < 15; e += 2) m = fmax3(m, s[16 * c + e], s[16 * c + e + 1]);
                m4[c] = fmaxf(m, s[16 * c + 15]);
            }
            float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
            float *xc = xchg + (n & 1) * 256;
            xc[hw * 128 + a] = mx;
            if (!(ok = pair_sync())) break;                       // also: both halves hold S
            mx = fmaxf(mx, xc[(1 - hw) * 128 + a]);
            mx = mx == -INFINITY ? -INFINITY : mx * c_qk;        // log2 units
            // lazy rescale: keep the running maximum unless it is exceeded by more than 8
            const bool need = mx > m_run + 8.f;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? fmaxf(m_run, mx) : m_run;
                // 0 when only m_run is -inf; 1 when the row has seen no visible key at all
                const float corr = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
                if (n > 0) {
                    if (!(ok = wait_pv(n - 1))) break;            // O holds P V of tiles < n
                    tc::fence_after();
                    uint32_t o[32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        tc::ld32(tmem + kTmemO + lane_off + cb + c * 32, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                        tc::st32(tmem + kTmemO + lane_off + cb + c * 32, o);
                    }
                    tc::wait_st();
                }
                l_run *= corr;
                m_run = m_new;
            }
            const float ref = m_run == -INFINITY ? 0.f : m_run;
            const float2 cq = make_float2(c_qk, c_qk), nref = make_float2(-ref, -ref);
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                // column pairs, logits to log2 units relative to the running maximum; three
                // pairs in eight take the polynomial exp2, the rest the special-function unit
                const float2 x = ffma2(make_float2(s[2 * e], s[2 * e + 1]), cq, nref);
                const int k8 = e & 7;
                const float2 y = (k8 == 1 || k8 == 4 || k8 == 6)
                    ? soft_exp2x2(x) : make_float2(fast_exp2(x.x), fast_exp2(x.y));
                l4[e & 3] = fadd2(l4[e & 3], y);
                pk[e] = pack_bf16(y.x, y.y);
            }
            // P for keys [64 w, 64 w + 64) -> packed columns [32 w, 32 w + 32) of the buffer
            tc::st32(sbuf + 32 * hw, pk);
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l_run += l2.x + l2.y;
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bar(B_P_FULL + (n & 1)));
        }
        // epilogue: the row sum of both halves, then O / l for this thread's 64 columns
        float *xl = xchg + 512;
        xl[hw * 128 + a] = l_run;
        if (ok) ok = pair_sync();
        const float l_tot = l_run + xl[(1 - hw) * 128 + a];
        if (ok) ok = wait_pv(N - 1);
        if (ok) {
            tc::fence_after();
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const bool valid = row < q_len;
            const size_t qrow = (size_t)(start + row) * p.Hq + h;
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tc::ld32(tmem + kTmemO + lane_off + cb + c * 32, o);
                tc::wait_ld();
                if (!valid) continue;
                const int col = cb + c * 32;
                if (p.out_dtype == INKATTN_DTYPE_F32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + qrow * kHeadDim + col);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                             __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<inkattn_bf16 *>(p.out) + qrow * kHeadDim + col);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(
                            pack_bf16(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                            pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                            pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                            pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
                }
            }
            if (valid && p.lse && hw == 0) {
                const float ref = m_run == -INFINITY ? 0.f : m_run;
                p.lse[qrow] = l_tot > 0.f ? (ref + log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
    // a CTA leaves only when its peer no longer writes into its shared memory
    if constexpr (kCluster > 1) cluster_sync();
}

cudaError_t launch_prefill_tc(const inkattn_attn_params &p, const AttnScalars &s, const CUtensorMap &qmap,
                              const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &pmap,
                              cudaStream_t stream) {
    TcArgs a;
    a.p = p;
    a.scale = s.scale;
    a.n_qtiles_max = (p.max_seqlen_q + kRows - 1) / kRows;
    a.kv_rows = (long long)p.num_blocks * p.Hkv * kBlock;
    dim3 grid(p.Hq, a.n_qtiles_max, p.B);
    // head pairs (2i, 2i + 1) share a KV head when the group size is even
    const bool pair = (p.Hq / p.Hkv) % 2 == 0;
    if (!pair) {
        cudaError_t err = cudaFuncSetAttribute(k_prefill_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (err != cudaSuccess) return err;
        k_prefill_tc<1><<<grid, kThreads, kSmem, stream>>>(a, qmap, kmap, vmap, pmap);
        return cudaGetLastError();
    }
    cudaError_t err = cudaFuncSetAttribute(k_prefill_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_prefill_tc<2>, a, qmap, kmap, vmap, pmap);
}

}  // namespace inkattn
