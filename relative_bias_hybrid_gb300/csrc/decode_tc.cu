// decode_tc.cu -- split-KV decode on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// sm_103a, with the relative-position bias.
//
// [vLLM TML Inkling サポート, §低レイテンシコレクティブとカーネル "FA4 Kernel"] and
// [vLLM hỗ trợ TML Inkling ..., §FA4 với sheared bias]: the attention kernel splits the KV
// length (num_splits picked from batch size, TP size and KV length); the partial results are
// merged afterwards (k_combine in decode.cu).
// [SGLang と Miles が Inkling を初日からサポート, §相対位置バイアス付き Attention]: the logit is
// the scaled dot product plus the bias r_i . P_h[:, i-j] for 0 <= i-j < rel_extent.
//
// One CTA per (split, KV head hk, sequence b).  Its MMA rows are the (token t, query head
// h = hk*g + hh) pairs of the sequence, row = t*g + hh (72 rows for 9 MTP-verify tokens x 8
// heads, padded to 128), so every K/V tile is read once for all the query heads that share
// it.  The Q tile arrives as one 3D TMA box {64 dims, g heads, ql tokens} per half of the
// head dimension, which lands exactly in that row order.  Roles, as in the prefill kernel:
//   warp 0      producer: TMA loads of 128-key K/V tiles (two 64-key cache blocks) of this
//               split's key range into a 4-slot ring, in the order the MMAs consume them
//               (every tile comes from HBM: the ring's depth sets the bytes in flight).
//   warp 1      MMA issuer (the whole warp, one elected lane issuing): S = Q K^T into a
//               double-buffered S in TMEM, O += P V with P (bf16) read from TMEM.
//   warps 2-9   softmax: two warpgroups; row a (TMEM lane a) is shared by one thread of each,
//               which own its key columns [0, 64) and [64, 128).
// TMEM: O [0,128) | S0 [128,256) | S1 [256,384).
//
// Relative bias: only tiles within rel_extent of the queries carry it (the last ones of the
// sequence).  For such a tile the softmax warps first build, per query head, the table
// R[t][x] = r_t . P_h[:, dlo + x] over the tile's 128 + ql distances with mma.sync (one warp
// per head; fp16 operands, fp32 accumulation), then each thread adds its row's 64 entries.
// fp16 keeps 11 significant bits of P (bf16 would keep 8) and represents the bf16 r exactly;
// r is first scaled, per token, by a power of two that keeps it inside fp16's range (exact,
// undone on the fp32 results).  P must lie inside fp16's range (|P| < 65504); a table entry
// that comes out infinite or undefined is flagged as INKATTN_ERR_DEVICE_BOUNDS.  The table holds 16-bit fixed point with one
// step per (head, token) row and round of 72 distances, sigma = (largest |entry| of that
// part of the row) / 32000; the staged bias is within sigma / 2 of the fp32 value.
// Normalisation: O accumulates P V with P rounded to bf16, and each tile's largest P (its
// row maximum's) is the dominant term whose bf16 rounding matters; that rounding error is
// added to the row's normaliser, while the LSE uses the sum of the fp32 P.
//
// The softmax runs in the log2 domain with the lazy rescale of the prefill kernel (O is
// rescaled only when the running maximum grows by more than 8).  The epilogue writes O / l
// and the natural-log LSE: straight to `out` with one split, else to the split workspace.
#include "common.cuh"
#include "fp8.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace inkattn {

namespace {

constexpr int kRows = 128;                 // MMA M: (token, query head) rows, padded
constexpr int kKeys = 128;                 // keys per tile (two cache blocks)
constexpr int kSlotBytes = 32768;          // one MMA operand tile: [d half][128 keys][128 B]
constexpr int kTabW = 144;                 // distances per table row: 128 keys + up to 16 tokens
constexpr int kTabRows = kDecodeMaxRows;   // g * ql <= 128
constexpr int kF8TileBytes = kKeys * kHeadDim;           // one E4M3 tile: [128 keys][128 B]
constexpr int kF8SlotBytes = kF8TileBytes + kKeys * 4;   // + its 128 row scales

// Two variants.  kF8 = false (bf16 cache): TMA loads K/V tiles straight into the MMAs'
// 4-slot ring.  kF8 = true (E4M3 cache): TMA loads E4M3 tiles and their row scales into a
// 3-slot ring, and six converter warps (2-7) convert Q to f16 in place, then expand each
// tile (code * scale, exactly) to f16 in a 3-slot MMA ring; P is packed as f16, so the MMAs
// run kind::f16 on f16 operands.  Warps: 0 TMA, 1 MMA, [2, 8) converters (E4M3
// only), then 8 softmax warps.
template <bool kF8>
struct Dec {
    static constexpr int kThreads = kF8 ? 512 : 320;
    static constexpr int kWarpSm = kF8 ? 8 : 2;              // first softmax warp
    static constexpr int kConvThreads = kF8 ? 192 : 0;       // converter warps 2-7
    static constexpr int kSlots = kF8 ? 3 : 4;               // MMA operand ring
    static constexpr int kF8Slots = kF8 ? 3 : 0;             // E4M3 ring
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = 32768;
    static constexpr int kOffF8 = kOffKV + kSlots * kSlotBytes;
    static constexpr int kOffTab = kOffF8 + kF8Slots * kF8SlotBytes;   // 16-bit fixed point [g][ql][kTabW]
    static constexpr int kOffXchg = kOffTab + kTabRows * kTabW * 2;     // row maxima / sums
    static constexpr int kOffTsig = kOffXchg + 3 * 2 * kRows * 4;       // fp32 steps [g][ql][2 rounds]
    static constexpr int kOffBar = kOffTsig + kTabRows * 2 * 4;
    // mbarrier indices, laid out from the slot counts
    static constexpr int B_Q = 0;
    static constexpr int B_KV_FULL = 1;
    static constexpr int B_KV_EMPTY = B_KV_FULL + kSlots;
    static constexpr int B_S_FULL = B_KV_EMPTY + kSlots;
    static constexpr int B_P_FULL = B_S_FULL + 2;
    static constexpr int B_PV_DONE = B_P_FULL + 2;
    static constexpr int B_TAB_FULL = B_PV_DONE + 2;
    static constexpr int B_TAB_FREE = B_TAB_FULL + 1;
    static constexpr int B_DRAIN = B_TAB_FREE + 1;
    static constexpr int B_QF = B_DRAIN + 1;                 // E4M3: Q converted to f16
    static constexpr int B_F8_FULL = B_QF + 1;
    static constexpr int B_F8_EMPTY = B_F8_FULL + kF8Slots;
    static constexpr int B_COUNT = B_F8_EMPTY + kF8Slots;
    static constexpr int kSmem = kOffBar + B_COUNT * 8 + 16;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kOffKV % 1024 == 0 && kOffF8 % 1024 == 0 && kF8SlotBytes % 128 == 0, "alignment of the rings");
    static_assert(kThreads == 32 * (kWarpSm + 8), "eight softmax warps last");
};

constexpr uint32_t kTmemO = 0, kTmemS0 = 128;
constexpr int kBarPair = 8;                // named barriers 8-11: the softmax row pairs, per lane quarter

struct DecTcArgs {
    inkattn_attn_params p;
    float scale;            // softmax scale
    int S;                  // number of splits
    int band_split;         // S == 2 cut at the band's start; the grid is (Hkv, B, 2)
    int ql;                 // rows of the Q box per head (max_seqlen_q)
    float *ws_o;
    float *ws_lse;
    long long kv_rows;      // rows of the cache tensor maps (OOB row = this)
    uint64_t wait_ns;       // limit of every bounded wait
    int withhold;           // failure-path test: the softmax withholds its first P arrival
};

}  // namespace

template <bool kF8>
__global__ void __launch_bounds__(Dec<kF8>::kThreads, 1)
k_decode_tc(const DecTcArgs A, const __grid_constant__ CUtensorMap qmap,
            const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    grid_dep_wait();                                   // q and the cache: written by the prologue
    using C = Dec<kF8>;
    const inkattn_attn_params &p = A.p;
    // band split: the CTAs of split 0 (the keys before the band) come first in the grid, so
    // that the short split-1 CTAs run on the SMs the streaming ones leave free
    const int split = A.band_split ? (int)blockIdx.z : (int)blockIdx.x;
    const int hk = A.band_split ? (int)blockIdx.x : (int)blockIdx.y;
    const int b = A.band_split ? (int)blockIdx.y : (int)blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = p.Hq / p.Hkv;

    // ---- sequence geometry and this split's key range (uniform over the CTA)
    const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1];
    const int T = p.seqlen_k[b];
    const int q_len = end - start;
    if (start < 0 || end < start || end > p.N_tok || q_len > A.ql || T < q_len ||
        T > p.max_seqlen_k || q_len * g > kRows) {
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    if (q_len == 0) return;
    const int n_rows = q_len * g;
    const int pos0 = T - q_len;                       // position of token 0
    int blk_first = 0;
    if (p.window > 0) blk_first = max(0, pos0 - p.window + 1) / kBlock;
    const int blk_end = (T + kBlock - 1) / kBlock;    // exclusive
    const int nblk = blk_end - blk_first;
    int my_lo, my_hi;
    if (A.band_split) {
        // two parts: the keys before the band, in whole 128-key tiles, and the rest (the keys
        // within rel_extent of the first query, whose tiles build bias tables)
        const int band_key_lo = max(0, pos0 - p.rel_extent + 1);
        const int cut = blk_first + ((max(blk_first, min(blk_end, band_key_lo / kBlock)) - blk_first) & ~1);
        my_lo = split == 0 ? blk_first : cut;
        my_hi = split == 0 ? cut : blk_end;
    } else {
        const int per = (nblk + A.S - 1) / A.S;
        my_lo = blk_first + split * per;
        my_hi = min(blk_end, my_lo + per);
    }
    const int my_n = max(0, my_hi - my_lo);
    const int N = (my_n + 1) / 2;                     // 128-key tiles
    const int kr_lo = my_lo * kBlock, kr_hi = my_hi * kBlock;
    const int g_shift = (g & (g - 1)) == 0 ? __ffs(g) - 1 : -1;

    if (N == 0) {
        // an empty split: its partial result is empty (O = 0, LSE = -inf)
        for (int idx = threadIdx.x; idx < n_rows * (kHeadDim / 4); idx += C::kThreads) {
            const int row = idx / (kHeadDim / 4), c4 = idx - row * (kHeadDim / 4);
            const int t = g_shift >= 0 ? row >> g_shift : row / g, hh = row - t * g;
            const size_t qrow = (size_t)(start + t) * p.Hq + hk * g + hh;
            *reinterpret_cast<float4 *>(A.ws_o + (qrow * A.S + split) * kHeadDim + c4 * 4) =
                make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 == 0) A.ws_lse[qrow * A.S + split] = -INFINITY;
        }
        return;
    }

    const uint32_t s_base = smem_u32(smem);
    if ((s_base & 1023u) != 0u) {
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    auto bar = [&](int i) { return s_base + C::kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + C::B_COUNT * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffBar + C::B_COUNT * 8 + 4);
    auto wwait = [&](uint32_t addr, uint32_t parity) -> bool {
        const bool r = mbar_wait(addr, parity, p.dev_status, abort_flag, A.wait_ns);
        return __all_sync(0xffffffffu, r);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_Q), 1);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(bar(C::B_KV_FULL + s), kF8 ? C::kConvThreads : 1);   // tile converters, or the TMA
            mbar_init(bar(C::B_KV_EMPTY + s), 1);
        }
        if constexpr (kF8) {
            mbar_init(bar(C::B_QF), 192);
            for (int s = 0; s < C::kF8Slots; ++s) {
                mbar_init(bar(C::B_F8_FULL + s), 1);
                mbar_init(bar(C::B_F8_EMPTY + s), C::kConvThreads);
            }
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_S_FULL + s), 1);
            mbar_init(bar(C::B_P_FULL + s), 256);
            mbar_init(bar(C::B_PV_DONE + s), 1);
        }
        mbar_init(bar(C::B_TAB_FULL), 256);
        mbar_init(bar(C::B_TAB_FREE), 256);
        mbar_init(bar(C::B_DRAIN), 1);
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
    const uint32_t tmem = *tmem_slot;

    const float lam = (p.log_scale_base > 1.f) ? fmaxf(1.f, logf((float)T) / logf(p.log_scale_base)) : 1.f;
    const float c_qk = lam * A.scale * kLog2e;       // S (with the bias folded in) -> log2 logit
    const float inv_scale = 1.f / A.scale;           // bias in S units

    // E4M3 variant (512 threads, 128 registers each at launch): the warpgroups of the TMA,
    // MMA and converter warps give registers to the two softmax warpgroups (80 + 176).
    if (warp == 0) {
        // ================================ producer ================================
        if constexpr (kF8) tc::reg_dealloc<80>();
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            const uint32_t qbytes = (uint32_t)(2 * 64 * 2 * g * A.ql);
            mbar_arrive_expect_tx(bar(C::B_Q), qbytes);
            tma_load_3d(s_base + C::kOffQ, &qmap, 0, hk * g, start, bar(C::B_Q));
            tma_load_3d(s_base + C::kOffQ + 16384, &qmap, 64, hk * g, start, bar(C::B_Q));
        }
        // the ring the TMA fills: the MMAs' own (bf16 cache) or the E4M3 one
        constexpr int kRing = kF8 ? C::kF8Slots : C::kSlots;
        constexpr int kRingFull = kF8 ? C::B_F8_FULL : C::B_KV_FULL;
        constexpr int kRingEmpty = kF8 ? C::B_F8_EMPTY : C::B_KV_EMPTY;
        int kv_loads = 0;
        auto load_kv = [&](int n, int isv) -> bool {
            const int L = kv_loads++, slot = L % kRing;
            // the tile's block-table entries are read before the wait for the slot, so that
            // their round trip to memory overlaps it instead of delaying the copy
            int blk[2];                                      // -2: past this split's range
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int lb = my_lo + 2 * n + half;         // logical cache block
                blk[half] = lb >= my_hi ? -2
                          : lb < p.max_blocks_per_seq ? __ldg(p.block_table + (size_t)b * p.max_blocks_per_seq + lb)
                          : -1;
            }
            if (L >= kRing && !wwait(bar(kRingEmpty + slot), ((L / kRing) - 1) & 1)) {
                --kv_loads;                                  // not issued
                return false;
            }
            const void *map = isv ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
            long long row[2];
            bool have[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                row[half] = A.kv_rows;                       // past the tensor: TMA fills zeros
                have[half] = blk[half] >= 0 && blk[half] < p.num_blocks;
                if (have[half]) row[half] = ((long long)blk[half] * p.Hkv + hk) * kBlock;
            }
            if constexpr (!kF8) {
                if (lane == 0) {
                    const uint32_t dst = s_base + C::kOffKV + slot * kSlotBytes;
                    const uint32_t fb = bar(C::B_KV_FULL + slot);
                    mbar_arrive_expect_tx(fb, kSlotBytes);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        if (blk[half] != -2 && !have[half]) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                        tma_load_2d(dst + half * 8192, map, 0, (int)row[half], fb);
                        tma_load_2d(dst + 16384 + half * 8192, map, 64, (int)row[half], fb);
                    }
                }
            } else {
                // codes [128 keys][128 B], then the 128 row scales; a half without a loaded
                // block reads as zero codes (TMA fill) with zero scales (written here)
                unsigned char *slot_p = smem + C::kOffF8 + slot * kF8SlotBytes;
                float *sc = reinterpret_cast<float *>(slot_p + kF8TileBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    if (!have[half]) {
                        sc[half * 64 + lane] = 0.f;
                        sc[half * 64 + 32 + lane] = 0.f;
                    }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t dst = smem_u32(slot_p);
                    const uint32_t fb = bar(C::B_F8_FULL + slot);
                    mbar_arrive_expect_tx(fb, kF8TileBytes + 256u * (uint32_t)(have[0] + have[1]));
                    const float *scales = isv ? p.v_scale : p.k_scale;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        if (blk[half] != -2 && !have[half]) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                        tma_load_2d(dst + half * 8192, map, 0, (int)row[half], fb);
                        if (have[half]) bulk_load(dst + kF8TileBytes + half * 256, scales + row[half], 256u, fb);
                    }
                }
            }
            __syncwarp();
            return true;
        };
        // consumption order of the MMA warp: K_0, then per tile n >= 1: K_n, V_{n-1}; then V_{N-1}
        ok = load_kv(0, 0);
        for (int n = 1; n < N && ok; ++n) {
            ok = load_kv(n, 0);
            if (ok) ok = load_kv(n - 1, 1);
        }
        if (ok) ok = load_kv(N - 1, 1);
        // nothing may still be landing in shared memory when the CTA tears down, also when a
        // role gave up: the copies issued and not yet consumed are the last kRing
        if (lane == 0) {
            mbar_drain(bar(C::B_Q), 0, p.dev_status, A.wait_ns);
            for (int L = max(0, kv_loads - kRing); L < kv_loads; ++L)
                mbar_drain(bar(kRingFull + L % kRing), (L / kRing) & 1, p.dev_status, A.wait_ns);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        if constexpr (kF8) tc::reg_dealloc<80>();
        constexpr uint32_t kFmt = kF8 ? tc::kFmtF16 : tc::kFmtBF16;   // both operands alike
        const uint32_t id_qk = tc::idesc(128, 128, kFmt, 0, 0);
        const uint32_t id_pv = tc::idesc(128, 128, kFmt, 0, 1);
        // the whole warp runs this loop with the same values in every lane (the MMAs and
        // commits are warp-collective); per-slot descriptors differ only in the start address
        // field, which stays below its 14 bits (shared memory < 256 KB)
        const uint64_t dq = tc::sdesc_sw128(s_base + C::kOffQ, 16, 1024);
        const uint64_t dk0 = tc::sdesc_sw128(s_base + C::kOffKV, 16, 1024);
        const uint64_t dv0 = tc::sdesc_sw128(s_base + C::kOffKV, 16384, 1024);
        auto slot_off = [](int slot) { return (uint64_t)(slot * (kSlotBytes >> 4)); };
        bool ok = wwait(bar(kF8 ? C::B_QF : C::B_Q), 0);      // (E4M3: Q once converted to f16)
        int kv_used = 0;
        auto next_tile = [&](int &slot, bool &last) -> bool {
            const int L = kv_used++;
            slot = L % C::kSlots;
            last = L + C::kSlots >= 2 * N;
            return wwait(bar(C::B_KV_FULL + slot), (L / C::kSlots) & 1);
        };
        auto issue_pv = [&](int m) -> bool {
            if (!wwait(bar(C::B_P_FULL + (m & 1)), (m >> 1) & 1)) return false;
            int slot;
            bool last;
            if (!next_tile(slot, last)) return false;
            // keys at or past the sequence end inside a loaded block: zero their V rows so
            // that P = 0 there contributes exact zeros whatever the cache slots hold
            const int j0 = kr_lo + m * kKeys;
            const int nvalid = max(0, min(kKeys, T - j0));
            const int nload = min(kKeys, (my_hi - my_lo - 2 * m) * kBlock);
            if (nvalid < nload) {
                unsigned char *vp = smem + C::kOffKV + slot * kSlotBytes;
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
            tc::mma_bf16_ts_k128_commit<false>(tmem + kTmemO, tmem + kTmemS0 + (uint32_t)(m & 1) * 128,
                                               dv0 + slot_off(slot), id_pv, m > 0 ? 1u : 0u, bar(C::B_PV_DONE + (m & 1)),
                                               bar(C::B_KV_EMPTY + slot), last ? 0u : 1u);
            __syncwarp();
            return true;
        };
        for (int n = 0; n < N && ok; ++n) {
            int slot;
            bool last;
            ok = next_tile(slot, last);
            if (!ok) break;
            tc::fence_after();
            tc::mma_bf16_ss_k128_commit<false>(tmem + kTmemS0 + (uint32_t)(n & 1) * 128, dq, dk0 + slot_off(slot),
                                               id_qk, 0u, bar(C::B_S_FULL + (n & 1)), bar(C::B_KV_EMPTY + slot),
                                               last ? 0u : 1u);
            __syncwarp();
            if (n >= 1) ok = issue_pv(n - 1);
        }
        if (ok) ok = issue_pv(N - 1);
        // every MMA of this CTA has completed before TMEM is released (also after a role gave up)
        tc::commit(bar(C::B_DRAIN));
        __syncwarp();
        (void)mbar_drain(bar(C::B_DRAIN), 0, p.dev_status, A.wait_ns);
        __syncwarp();
    } else if (kF8 && warp < C::kWarpSm) {
        // ================================ converters (E4M3 cache) ================================
        if constexpr (kF8) tc::reg_dealloc<80>();
        // warps 2-7 convert Q, then the K/V tiles
        const int ct = threadIdx.x - 64;                      // 0 .. 191
        bool ok = wwait(bar(C::B_Q), 0);
        if (ok) {
            uint4 *qw = reinterpret_cast<uint4 *>(smem + C::kOffQ);
            for (int i = ct; i < 32768 / 16; i += 192) {
                const uint4 w = qw[i];
                qw[i] = make_uint4(pack_f16(bf16_lo(w.x), bf16_hi(w.x)), pack_f16(bf16_lo(w.y), bf16_hi(w.y)),
                                   pack_f16(bf16_lo(w.z), bf16_hi(w.z)), pack_f16(bf16_lo(w.w), bf16_hi(w.w)));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(C::B_QF));
        }
        for (int L = 0; L < 2 * N && ok; ++L) {
            const int n = L == 0 ? 0 : L == 2 * N - 1 ? N - 1 : (L & 1) ? (L + 1) >> 1 : (L >> 1) - 1;
            const int s8 = L % C::kF8Slots, s16 = L % C::kSlots;
            if (!(ok = wwait(bar(C::B_F8_FULL + s8), (L / C::kF8Slots) & 1))) break;
            if (L >= C::kSlots && !(ok = wwait(bar(C::B_KV_EMPTY + s16), ((L / C::kSlots) - 1) & 1))) break;
            const unsigned char *src = smem + C::kOffF8 + s8 * kF8SlotBytes;
            const float *sc = reinterpret_cast<const float *>(src + kF8TileBytes);
            unsigned char *dst = smem + C::kOffKV + s16 * kSlotBytes;
            const int key_end = min(T, kr_hi) - (kr_lo + n * kKeys);
            bool bad = false;
            for (int it = ct; it < kKeys * 8; it += 192) {
                const int key = it >> 3, j16 = it & 7, sw = key & 7;
                const uint4 w = *reinterpret_cast<const uint4 *>(src + key * 128 + j16 * 16);
                float sv = key < key_end ? sc[key] : 0.f;
                const bool good = sv == 0.f || (sv >= 0x1p-24f && sv <= 128.f);
                bad |= !good;
                const __half2 s2 = __float2half2_rn(good ? sv : 0.f);
                const int base = (j16 >> 2) * 16384 + key * 128;
                *reinterpret_cast<uint4 *>(dst + base + ((((j16 & 3) * 2) ^ sw) << 4)) =
                    make_uint4(e4m3x2_to_f16x2_scaled(w.x, s2), e4m3x2_to_f16x2_scaled(w.x >> 16, s2),
                               e4m3x2_to_f16x2_scaled(w.y, s2), e4m3x2_to_f16x2_scaled(w.y >> 16, s2));
                *reinterpret_cast<uint4 *>(dst + base + ((((j16 & 3) * 2 + 1) ^ sw) << 4)) =
                    make_uint4(e4m3x2_to_f16x2_scaled(w.z, s2), e4m3x2_to_f16x2_scaled(w.z >> 16, s2),
                               e4m3x2_to_f16x2_scaled(w.w, s2), e4m3x2_to_f16x2_scaled(w.w >> 16, s2));
            }
            if (bad) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
            fence_proxy_async_smem();
            mbar_arrive(bar(C::B_F8_EMPTY + s8));
            mbar_arrive(bar(C::B_KV_FULL + s16));
        }
    } else {
        // ================================ softmax ================================
        if constexpr (kF8) tc::reg_alloc<176>();
        const int quad = warp & 3;
        const int sw = warp - C::kWarpSm;                     // softmax warp index 0..7
        const int hw = sw >> 2;                               // column half
        const int a = quad * 32 + lane;                       // MMA row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool valid_row = a < n_rows;
        const bool quad_live = quad * 32 < n_rows;            // uniform over the warp (and its pair)
        const int t = valid_row ? (g_shift >= 0 ? a >> g_shift : a / g) : 0;
        const int hh = a - t * g;
        const int i_pos = pos0 + t;
        const int cb = 64 * hw;
        unsigned short *tab = reinterpret_cast<unsigned short *>(smem + C::kOffTab);
        float *tsig = reinterpret_cast<float *>(smem + C::kOffTsig);
        float *xchg = reinterpret_cast<float *>(smem + C::kOffXchg);
        // The two threads of a row meet on a named barrier of the row's lane quarter (64
        // threads, one warp of each column half), as in the prefill kernel: every thread
        // makes exactly N + 1 meetings (warps whose rows are all padding skip their tiles'
        // meetings and make them up at the end, as a thread that left the loop early does).
        auto pair_meet = [&]() { asm volatile("bar.sync %0, 64;" :: "r"(kBarPair + quad) : "memory"); };
        int met = 0;
        const bool has_bias = p.rel_extent > 0;
        const int gq = lane >> 2, tq = lane & 3;              // mma.sync fragment coordinates
        int band_round = 0;
        bool ok = true;

        float m_run = -INFINITY, l_run = 0.f;   // l_run: sum of the fp32 P (for the LSE)
        float lc_run = 0.f;                      // bf16 rounding of each tile's largest P (normaliser)
        auto wait_pv = [&](int m) -> bool { return wwait(bar(C::B_PV_DONE + (m & 1)), (m >> 1) & 1); };
        for (int n = 0; n < N; ++n) {
            const int j0 = kr_lo + n * kKeys;
            const bool band = has_bias && (pos0 - (j0 + kKeys - 1) < p.rel_extent);
            const int dlo = pos0 - j0 - (kKeys - 1);          // distance at table column 0
            if (band) {
                // ---- relative rows of this tile, one query head per warp, into the table
                if (band_round > 0 && !(ok = wwait(bar(C::B_TAB_FREE), (band_round - 1) & 1))) break;
                for (int hq = sw; hq < g; hq += 8) {
                    const int h = hk * g + hq;
                    const float *Ph = p.P + (size_t)h * p.rel_extent * 32;
                    const inkattn_bf16 *rh = p.r + ((size_t)start * p.Hq + h) * 32;
                    // d_r = 32 (checked on the host): two k steps of 16.  A fragments: tokens gq
                    // (e even) and gq + 8 (e odd), each lane 8 of a token's 32 features; the four
                    // lanes of a token (tq = 0..3) hold all of them.
                    float rv[2][4][2];
                    float rm[2] = {0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tt = gq + ((e & 1) << 3);
                            const int col = kk * 16 + 2 * tq + ((e >> 1) << 3);
                            const uint32_t w2 = tt < q_len
                                ? __ldg(reinterpret_cast<const uint32_t *>(rh + (size_t)tt * 32 * p.Hq + col))
                                : 0u;
                            rv[kk][e][0] = bf16_lo(w2);
                            rv[kk][e][1] = bf16_hi(w2);
                            rm[e & 1] = fmaxf(rm[e & 1], fmaxf(fabsf(rv[kk][e][0]), fabsf(rv[kk][e][1])));
                        }
                    float rsc[2], rusc[2];                     // per token row: fp16 prescale and its inverse
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        rm[i] = fmaxf(rm[i], __shfl_xor_sync(0xffffffffu, rm[i], 1));
                        rm[i] = fmaxf(rm[i], __shfl_xor_sync(0xffffffffu, rm[i], 2));
                        rsc[i] = fp16_prescale(rm[i]);
                        rusc[i] = 1.f / rsc[i];
                    }
                    uint32_t rf[2][4];
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            rf[kk][e] = pack_f16(rv[kk][e][0] * rsc[e & 1], rv[kk][e][1] * rsc[e & 1]);
                    // the table in two rounds of nine groups of 8 distances: a round's P loads
                    // are all issued before its first MMA, so the table waits for two L2 round
                    // trips (the first also covers r above), not one per group; while K/V
                    // streams saturate the memory system a round trip costs thousands of cycles.
                    // Each round's results set the steps of its part of the rows and are stored.
                    constexpr int kGrp = 9;
                    static_assert(kTabW / 8 == 2 * kGrp, "two rounds");
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
                        float res[kGrp][4];
                        uint32_t pb[kGrp][2][2];
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            const int dl = dlo + (rd * kGrp + u) * 8 + gq;
                            const bool dv = dl >= 0 && dl < p.rel_extent;
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const int e0 = kk * 16 + 2 * tq;
                                const float2 lo = dv ? __ldg(reinterpret_cast<const float2 *>(Ph + (size_t)dl * 32 + e0))
                                                     : make_float2(0.f, 0.f);
                                const float2 hi = dv ? __ldg(reinterpret_cast<const float2 *>(Ph + (size_t)dl * 32 + e0 + 8))
                                                     : make_float2(0.f, 0.f);
                                pb[u][kk][0] = pack_f16(lo.x, lo.y);
                                pb[u][kk][1] = pack_f16(hi.x, hi.y);
                            }
                        }
                        bool finite = true;
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) mma_16816_f16(acc, rf[kk], pb[u][kk][0], pb[u][kk][1]);
                            res[u][0] = acc[0] * rusc[0];
                            res[u][1] = acc[1] * rusc[0];
                            res[u][2] = acc[2] * rusc[1];
                            res[u][3] = acc[3] * rusc[1];
                            finite = finite && isfinite(acc[0] + acc[1] + acc[2] + acc[3]);
                        }
                        // a P beyond fp16's range (|P| >= 65520) leaves an infinite or undefined entry
                        if (!finite) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                        // each token row's largest |entry| in this round (its four lanes hold all
                        // of its columns here)
                        float mx[2] = {0.f, 0.f};
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            mx[0] = fmaxf(mx[0], fmaxf(fabsf(res[u][0]), fabsf(res[u][1])));
                            mx[1] = fmaxf(mx[1], fmaxf(fabsf(res[u][2]), fabsf(res[u][3])));
                        }
                        float enc[2];
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
                            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
                            const float mm = fmaxf(mx[i], 1e-30f);
                            const int tt = gq + 8 * i;
                            // the step in S units (the table holds R / scale); entries encode to
                            // R * (32000 / max) in [-32000, 32000]
                            if (tq == 0 && tt < q_len) tsig[(hq * A.ql + tt) * 2 + rd] = mm * inv_scale * (1.f / 32000.f);
                            enc[i] = 32000.f / mm;
                        }
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            const int c = (rd * kGrp + u) * 8 + 2 * tq;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int tt = gq + 8 * i;
                                if (tt >= q_len) continue;
                                const float2 v = fix16_encode2(make_float2(res[u][2 * i], res[u][2 * i + 1]), enc[i]);
                                *reinterpret_cast<uint32_t *>(tab + ((size_t)hq * A.ql + tt) * kTabW + c) =
                                    (__float_as_uint(v.x) & 0xFFFFu) | (__float_as_uint(v.y) << 16);
                            }
                        }
                    }
                }
                mbar_arrive(bar(C::B_TAB_FULL));
                if (!(ok = wwait(bar(C::B_TAB_FULL), band_round & 1))) break;
            }

            if (!(ok = wwait(bar(C::B_S_FULL + (n & 1)), (n >> 1) & 1))) break;
            if (!quad_live) {
                // every row of this warp's lane quarter is padding: its P rows feed only O rows
                // that are never written, so the warp only keeps the barrier counts
                if (band) {
                    mbar_arrive(bar(C::B_TAB_FREE));
                    ++band_round;
                }
                tc::fence_before();
                if (!(A.withhold && n == 0)) mbar_arrive(bar(C::B_P_FULL + (n & 1)));
                continue;
            }
            tc::fence_after();
            const uint32_t sbuf = tmem + kTmemS0 + (uint32_t)(n & 1) * 128 + lane_off;
            float s[64];
            {
                uint32_t *su = reinterpret_cast<uint32_t *>(s);
                tc::ld32(sbuf + cb, *reinterpret_cast<uint32_t(*)[32]>(su));
                tc::ld32(sbuf + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
                tc::wait_ld();
            }
            if (band) {
                if (valid_row) {
                    // column b of the tile is at distance i - j = dlo + (t + 127 - b)
                    const int c0 = t + (kKeys - 1) - cb;             // table column of key column cb
                    const unsigned short *trow = tab + ((size_t)hh * A.ql + t) * kTabW + c0;
                    const float sg0 = tsig[(hh * A.ql + t) * 2], sg1 = tsig[(hh * A.ql + t) * 2 + 1];
#pragma unroll
                    for (int bb = 0; bb < 64; ++bb) {
                        const float q = __uint_as_float(0x4B000000u | (uint32_t)trow[-bb]) - 8421376.0f;
                        s[bb] = fmaf(q, c0 - bb < 72 ? sg0 : sg1, s[bb]);   // columns [0, 72): first round
                    }
                }
                mbar_arrive(bar(C::B_TAB_FREE));
                ++band_round;
            }
            // mask: key j visible iff it is in this split's range, j <= i and (SWA) i - j < window
            int b_lo, span;
            {
                int jv_lo = kr_lo, jv_hi = min(i_pos, kr_hi - 1);
                if (p.window > 0) jv_lo = max(jv_lo, i_pos - p.window + 1);
                const bool any = valid_row && jv_hi >= jv_lo;
                b_lo = any ? jv_lo - j0 - cb : (1 << 20);
                span = any ? jv_hi - jv_lo : 0;
            }
            const bool need_mask = !valid_row || (j0 + kKeys - 1 > pos0) || (j0 + kKeys > kr_hi) ||
                                   (p.window > 0 && pos0 + q_len - 1 - j0 >= p.window);
            if (need_mask) {
#pragma unroll
                for (int bb = 0; bb < 64; ++bb)
                    s[bb] = ((unsigned)(bb - b_lo) <= (unsigned)span) ? s[bb] : -INFINITY;
            }
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
            pair_meet();
            ++met;
            mx = fmaxf(mx, xc[(1 - hw) * 128 + a]);
            const float mx_raw = mx;                             // the row's largest logit of the tile (S units)
            mx = mx == -INFINITY ? -INFINITY : mx * c_qk;        // log2 units
            const bool need = mx > m_run + 8.f;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? fmaxf(m_run, mx) : m_run;
                const float corr = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
                if (n > 0) {
                    if (!(ok = wait_pv(n - 1))) break;
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
                lc_run *= corr;
                m_run = m_new;
            }
            const float ref = m_run == -INFINITY ? 0.f : m_run;
            const float2 cq = make_float2(c_qk, c_qk), nref = make_float2(-ref, -ref);
            if (hw == 0 && mx_raw != -INFINITY) {
                // the tile's largest P of this row, computed as its element is, and its bf16 rounding
                const float pm = fast_exp2(fmaf(mx_raw, c_qk, -ref));
                if constexpr (kF8) lc_run += __half2float(__float2half_rn(pm)) - pm;
                else lc_run += bf16_lo(pack_bf16(pm, 0.f)) - pm;
            }
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float2 x = ffma2(make_float2(s[2 * e], s[2 * e + 1]), cq, nref);
                const float2 y = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                l4[e & 3] = fadd2(l4[e & 3], y);
                pk[e] = kF8 ? pack_f16(y.x, y.y) : pack_bf16(y.x, y.y);
            }
            tc::st32(sbuf + 32 * hw, pk);
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l_run += l2.x + l2.y;
            tc::wait_st();
            tc::fence_before();
            if (!(A.withhold && n == 0)) mbar_arrive(bar(C::B_P_FULL + (n & 1)));
        }
        // epilogue: the row sum of both halves, then O / l for this thread's 64 columns
        // the column-half 0 thread of a row alone holds the correction (lc_run is 0 in the other)
        // and alone writes the LSE: it publishes l + lc, the other thread l
        for (; met < N; ++met) pair_meet();
        float *xl = xchg + 512;
        xl[hw * 128 + a] = l_run + lc_run;
        pair_meet();
        const float l_other = xl[(1 - hw) * 128 + a];
        const float l_tot = l_run + l_other;                  // the fp32 sum (read by half 0 only)
        const float l_norm = l_run + lc_run + l_other;        // normaliser of P V's bf16 P
        if (ok) ok = wait_pv(N - 1);
        if (ok) {
            tc::fence_after();
            const float inv = l_norm > 0.f ? 1.f / l_norm : 0.f;
            const size_t qrow = (size_t)(start + t) * p.Hq + hk * g + hh;
            const float ref = m_run == -INFINITY ? 0.f : m_run;
            const float lse_nat = l_tot > 0.f ? (ref + log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tc::ld32(tmem + kTmemO + lane_off + cb + c * 32, o);
                tc::wait_ld();
                if (!valid_row) continue;
                const int col = cb + c * 32;
                if (A.S > 1) {
                    float4 *dst = reinterpret_cast<float4 *>(A.ws_o + (qrow * A.S + split) * kHeadDim + col);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                             __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                } else if (p.out_dtype == INKATTN_DTYPE_F32) {
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
            if (valid_row && hw == 0) {
                if (A.S > 1) A.ws_lse[qrow * A.S + split] = lse_nat;
                else if (p.lse) p.lse[qrow] = lse_nat;
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

template <bool kF8>
cudaError_t launch_decode_variant(const DecTcArgs &a, dim3 grid, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                  const CUtensorMap &vmap, cudaStream_t stream) {
    using C = Dec<kF8>;
    if constexpr (kF8) {
        // the register split (2 warpgroups at 80 + 2 at 176 = 512 x 128) needs exactly 128
        // registers a thread at launch: with fewer, setmaxnreg.inc could never be satisfied
        static const cudaError_t regs_check = [] {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, k_decode_tc<true>) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
            return fa.numRegs == 128 ? cudaSuccess : cudaErrorInvalidConfiguration;
        }();
        if (regs_check != cudaSuccess) return regs_check;
    }
    cudaError_t err = cudaFuncSetAttribute(k_decode_tc<kF8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (err != cudaSuccess) return err;
    return launch_dependent(k_decode_tc<kF8>, grid, dim3(C::kThreads), C::kSmem, stream, 1, a, qmap, kmap, vmap);
}

cudaError_t launch_decode_tc(const inkattn_attn_params &p, const AttnScalars &s, int num_splits,
                             float *ws_o, float *ws_lse, const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, cudaStream_t stream) {
    DecTcArgs a;
    a.p = p;
    a.scale = s.scale;
    a.S = num_splits;
    a.band_split = num_splits == 2 && p.rel_extent > 0;
    a.ql = p.max_seqlen_q;
    a.ws_o = ws_o;
    a.ws_lse = ws_lse;
    a.kv_rows = (long long)p.num_blocks * p.Hkv * kBlock;
    a.wait_ns = kernel_debug().wait_ns;
    a.withhold = kernel_debug().withhold;
    const dim3 grid = a.band_split ? dim3(p.Hkv, p.B, 2) : dim3(num_splits, p.Hkv, p.B);
    return p.kv_dtype == INKATTN_KV_E4M3 ? launch_decode_variant<true>(a, grid, qmap, kmap, vmap, stream)
                                         : launch_decode_variant<false>(a, grid, qmap, kmap, vmap, stream);
}

}  // namespace inkattn
