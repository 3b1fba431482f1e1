// prefill_2q.cu -- GQA prefill without relative bias on tcgen05/TMEM, two query tiles per CTA.
//
// [SGLang と Miles が Inkling を初日からサポート, §Relative Attention と FA4 経路]: a
// warp-specialized attention kernel on Blackwell.  This kernel serves calls whose relative
// bias is off (rel_extent = 0) and has no sheared band to apply; prefill_tc.cu serves the
// others.
//
// One CTA per (pair of consecutive 128-query tiles A and B of one sequence, query head).
// The two tiles share every K/V tile, and their two softmax warpgroups take turns with the
// tensor pipe: while the softmax of A works on key tile n, the MMAs of B (P V of tile n - 1
// and Q K^T of tile n) run, and the other way round.  Roles:
//   warp 0      producer: TMA loads of Q_A, Q_B and of 128-key K/V tiles into a 3-slot ring,
//               in the order the MMAs first use them (K_0, V_0, K_1, V_1, ...).
//   warp 1      MMA issuer (the whole warp, one elected lane issuing).
//   warps 2-5   softmax of tile A, warps 6-9 softmax of tile B: one thread per query row,
//               all 128 key columns of the tile (no exchange between threads).
// TMEM (512 columns): O_A [0,128) | O_B [128,256) | S_A [256,384) | S_B [384,512).  P (bf16)
// overwrites the first 64 columns of its S; Q K^T of the next key tile follows P V of this
// one in the tensor pipe, so the overwrite is ordered.
//
// The softmax runs in the log2 domain with a lazy rescale (O is rescaled only when the row
// maximum grows by more than 8); column pairs use paired fp32 instructions, and every exp2
// goes through the special-function unit.  The bf16 rounding error of each tile's largest P
// (a row's dominant term once P V rounds P to bf16) is added to the row's normaliser; the
// LSE uses the sum of the fp32 P.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace inkattn {

namespace {

constexpr int kRows = 128;                 // query rows per tile (MMA M)
constexpr int kKeys = 128;                 // keys per tile
constexpr int kSlots = 3;                  // K/V ring slots
constexpr int kSlotBytes = 32768;
constexpr int kThreads = 320;

constexpr int kOffQ = 0;                   // Q_A, Q_B: 32 KB each
constexpr int kOffKV = 65536;
constexpr int kOffBar = kOffKV + kSlots * kSlotBytes;

// mbarrier indices, laid out from the slot count so that no two ranges overlap
enum Bar {
    B_Q = 0,
    B_KV_FULL = 1,
    B_KV_EMPTY = B_KV_FULL + kSlots,
    B_S_FULL = B_KV_EMPTY + kSlots,
    B_P_FULL = B_S_FULL + 2,
    B_PV_DONE = B_P_FULL + 2,
    B_DRAIN = B_PV_DONE + 2,
    B_COUNT = B_DRAIN + 1
};
constexpr int kSmem = kOffBar + B_COUNT * 8 + 16;
static_assert(kSmem <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
static_assert(kOffKV % 1024 == 0 && kOffBar % 8 == 0, "alignment of the regions");

constexpr uint32_t kTmemO = 0, kTmemS = 256;

struct Tc2Args {
    inkattn_attn_params p;
    float scale;
    int n_pairs_max;        // gridDim.y
    long long kv_rows;
    uint64_t wait_ns;       // limit of every bounded wait
    int withhold;           // failure-path test: tile A's softmax withholds its first P arrival
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
k_prefill_2q(const Tc2Args A, const __grid_constant__ CUtensorMap qmap,
             const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    grid_dep_wait();                                   // q and the cache: written by the prologue
    const inkattn_attn_params &p = A.p;
    const int h = blockIdx.x, b = blockIdx.z;
    const int pr = A.n_pairs_max - 1 - (int)blockIdx.y;     // longest pairs first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = p.Hq / p.Hkv, hk = h / g;

    const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1];
    const int T = p.seqlen_k[b];
    const int q_len = end - start;
    if (start < 0 || end < start || end > p.N_tok || q_len > p.max_seqlen_q || T < q_len ||
        T > p.max_seqlen_k) {
        if (threadIdx.x == 0 && pr == 0 && h == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    const int row0 = pr * 2 * kRows;                     // first row of tile A
    if (row0 >= q_len) return;
    const bool has_b = row0 + kRows < q_len;
    const int pos0 = T - q_len;
    // key-tile range of each query tile
    int tx_lo[2], tx_hi[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int lo = pos0 + row0 + x * kRows;
        const int hi = pos0 + min(q_len, row0 + (x + 1) * kRows) - 1;
        const int klo = p.window > 0 ? max(0, lo - p.window + 1) : 0;
        tx_hi[x] = hi / kKeys;
        tx_lo[x] = klo / kKeys;
    }
    if (!has_b) { tx_lo[1] = 1; tx_hi[1] = 0; }          // empty range
    const int t_top = has_b ? tx_hi[1] : tx_hi[0];
    const int t_bot = has_b ? min(tx_lo[0], tx_lo[1]) : tx_lo[0];
    const int N = t_top - t_bot + 1;                     // key tiles, nearest first
    auto in_x = [&](int x, int n) { const int t = t_top - n; return t >= tx_lo[x] && t <= tx_hi[x]; };

    const uint32_t s_base = smem_u32(smem);
    if ((s_base & 1023u) != 0u) {
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    auto bar = [&](int i) { return s_base + kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + B_COUNT * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + B_COUNT * 8 + 4);
    auto wwait = [&](uint32_t addr, uint32_t parity) -> bool {
        const bool r = mbar_wait(addr, parity, p.dev_status, abort_flag, A.wait_ns);
        return __all_sync(0xffffffffu, r);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_S_FULL + x), 1);
            mbar_init(bar(B_P_FULL + x), 128);
            mbar_init(bar(B_PV_DONE + x), 1);
        }
        mbar_init(bar(B_DRAIN), 1);
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
    const float c_qk = lam * A.scale * kLog2e;

    if (warp == 0) {
        // ================================ producer ================================
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            const int nq = has_b ? 2 : 1;
            mbar_arrive_expect_tx(bar(B_Q), nq * 2 * 16384);
            for (int x = 0; x < nq; ++x) {
                tma_load_3d(s_base + kOffQ + x * 32768, &qmap, 0, h, start + row0 + x * kRows, bar(B_Q));
                tma_load_3d(s_base + kOffQ + x * 32768 + 16384, &qmap, 64, h, start + row0 + x * kRows, bar(B_Q));
            }
        }
        int kv_loads = 0;
        auto load_kv = [&](int n, int isv) -> bool {
            const int L = kv_loads++, slot = L % kSlots;
            const int t = t_top - n;
            // the tile's block-table entries are read before the wait for the slot, so that
            // their round trip to memory overlaps it instead of delaying the copy
            int blk[2];                                      // -2: past the sequence end
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int lb = 2 * t + half;                 // logical cache block
                blk[half] = (long long)lb * kBlock >= T ? -2
                          : lb < p.max_blocks_per_seq ? __ldg(p.block_table + (size_t)b * p.max_blocks_per_seq + lb)
                          : -1;
            }
            if (L >= kSlots && !wwait(bar(B_KV_EMPTY + slot), ((L / kSlots) - 1) & 1)) {
                --kv_loads;                                  // not issued
                return false;
            }
            if (lane == 0) {
                const uint32_t dst = s_base + kOffKV + slot * kSlotBytes;
                const uint32_t fb = bar(B_KV_FULL + slot);
                mbar_arrive_expect_tx(fb, kSlotBytes);
                const void *map = isv ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    long long row = A.kv_rows;
                    if (blk[half] != -2) {
                        if (blk[half] >= 0 && blk[half] < p.num_blocks) row = ((long long)blk[half] * p.Hkv + hk) * kBlock;
                        else set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                    }
                    tma_load_2d(dst + half * 8192, map, 0, (int)row, fb);
                    tma_load_2d(dst + 16384 + half * 8192, map, 64, (int)row, fb);
                }
            }
            __syncwarp();
            return true;
        };
        for (int n = 0; n < N && ok; ++n) {
            ok = load_kv(n, 0);
            if (ok) ok = load_kv(n, 1);
        }
        // nothing may still be landing in shared memory when the CTA tears down, also when a
        // role gave up: the copies issued and not yet consumed are the last kSlots
        if (lane == 0) {
            mbar_drain(bar(B_Q), 0, p.dev_status, A.wait_ns);
            for (int L = max(0, kv_loads - kSlots); L < kv_loads; ++L)
                mbar_drain(bar(B_KV_FULL + L % kSlots), (L / kSlots) & 1, p.dev_status, A.wait_ns);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        const uint32_t id_qk = tc::idesc(128, 128, tc::kFmtBF16, 0, 0);
        const uint32_t id_pv = tc::idesc(128, 128, tc::kFmtBF16, 0, 1);
        // the whole warp runs this loop with the same values in every lane (the MMAs and
        // commits are warp-collective); per-tile and per-slot descriptors differ only in the
        // start address field, which stays below its 14 bits (shared memory < 256 KB)
        const uint64_t dq0 = tc::sdesc_sw128(s_base + kOffQ, 16, 1024);
        const uint64_t dk0 = tc::sdesc_sw128(s_base + kOffKV, 16, 1024);
        const uint64_t dv0 = tc::sdesc_sw128(s_base + kOffKV, 16384, 1024);
        auto slot_off = [](int slot) { return (uint64_t)(slot * (kSlotBytes >> 4)); };
        bool ok = wwait(bar(B_Q), 0);
        int kv_used = 0;
        auto acquire = [&](int &slot, bool &last) -> bool {
            const int L = kv_used++;
            slot = L % kSlots;
            last = L + kSlots >= 2 * N;
            return wwait(bar(B_KV_FULL + slot), (L / kSlots) & 1);
        };
        auto release = [&](int slot, bool last) {
            if (!last) tc::commit(bar(B_KV_EMPTY + slot));
        };
        auto qk = [&](int x, int slot) {
            tc::mma_bf16_ss_k128_commit<false>(tmem + kTmemS + x * 128, dq0 + (uint64_t)(x * (32768 >> 4)),
                                        dk0 + slot_off(slot), id_qk, 0u, bar(B_S_FULL + x));
            __syncwarp();
        };
        int kp[2] = {0, 0};                                   // P V issued per tile
        auto pv = [&](int x, int slot) -> bool {
            if (!wwait(bar(B_P_FULL + x), kp[x] & 1)) return false;
            tc::fence_after();
            tc::mma_bf16_ts_k128_commit<false>(tmem + kTmemO + x * 128, tmem + kTmemS + x * 128, dv0 + slot_off(slot),
                                        id_pv, kp[x] > 0 ? 1u : 0u, bar(B_PV_DONE + x));
            __syncwarp();
            ++kp[x];
            return true;
        };

        int kslot = 0, vslot = 0;
        bool klast = false, vlast = false;
        if (ok) ok = acquire(kslot, klast);                  // K_0
        if (ok) {
            tc::fence_after();
            if (in_x(0, 0)) qk(0, kslot);
            if (in_x(1, 0)) qk(1, kslot);
            release(kslot, klast);
        }
        for (int n = 0; n < N && ok; ++n) {
            if (!(ok = acquire(vslot, vlast))) break;        // V_n
            // keys at or past the sequence end inside a loaded block: zero their V rows
            {
                const int j0 = (t_top - n) * kKeys;
                const int nvalid = min(kKeys, T - j0);
                const int nload = min(kKeys, (int)(((long long)((T + kBlock - 1) / kBlock)) * kBlock - j0));
                if (nvalid < nload) {
                    unsigned char *vp = smem + kOffKV + vslot * kSlotBytes;
                    const int rows = nload - nvalid;
                    for (int idx = lane; idx < rows * 16; idx += 32) {
                        const int key = nvalid + idx / 16, dh = (idx >> 3) & 1, ch = idx & 7;
                        *reinterpret_cast<uint4 *>(vp + dh * 16384 + (key >> 6) * 8192 + (key & 63) * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }
            const bool more = n + 1 < N;
            bool next_ready = false;
            if (in_x(0, n)) {
                if (!(ok = pv(0, vslot))) break;
            }
            if (more) {
                if (!(ok = acquire(kslot, klast))) break;    // K_{n+1}
                tc::fence_after();
                next_ready = true;
                if (in_x(0, n + 1)) qk(0, kslot);
            }
            if (in_x(1, n)) {
                if (!(ok = pv(1, vslot))) break;
            }
            release(vslot, vlast);
            if (next_ready) {
                if (in_x(1, n + 1)) qk(1, kslot);
                release(kslot, klast);
            }
        }
        // every MMA of this CTA has completed before TMEM is released (also after a role gave up)
        tc::commit(bar(B_DRAIN));
        __syncwarp();
        (void)mbar_drain(bar(B_DRAIN), 0, p.dev_status, A.wait_ns);
        __syncwarp();
    } else {
        // ================================ softmax ================================
        const int x = (warp - 2) >> 2;                        // tile A or B
        const int quad = warp & 3;
        const int a = quad * 32 + lane;                       // row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int row = row0 + x * kRows + a;                 // row within the sequence
        const int i_pos = pos0 + row;
        const bool tile_valid = (x == 0) || has_b;
        const int t_lo_x = tx_lo[x], t_hi_x = tx_hi[x];
        const int p_lo_x = pos0 + row0 + x * kRows;
        const uint32_t sbuf = tmem + kTmemS + x * 128 + lane_off;
        const uint32_t obuf = tmem + kTmemO + x * 128 + lane_off;
        bool ok = true;
        float m_run = -INFINITY, l_run = 0.f;   // l_run: sum of the fp32 P (for the LSE)
        float lc_run = 0.f;                      // bf16 rounding of each tile's largest P (normaliser)
        int kx = 0;
        for (int n = 0; n < N && tile_valid; ++n) {
            const int t = t_top - n;
            if (t < t_lo_x || t > t_hi_x) continue;
            if (!(ok = wwait(bar(B_S_FULL + x), kx & 1))) break;
            tc::fence_after();
            const int j0 = t * kKeys;
            int b_lo, span;                                   // visible: (unsigned)(b - b_lo) <= span
            {
                const int jv_lo = p.window > 0 ? i_pos - p.window + 1 : 0;
                const int jv_hi = min(i_pos, T - 1);
                b_lo = jv_hi >= jv_lo ? jv_lo - j0 : (1 << 20);
                span = jv_hi >= jv_lo ? jv_hi - jv_lo : 0;
            }
            const bool need_mask = (j0 + kKeys - 1 > p_lo_x) || (j0 + kKeys - 1 >= T) ||
                                   (p.window > 0 && p_lo_x + kRows - 1 - j0 >= p.window);
            // pass 1: row maximum over the 128 columns, 64 at a time (two loads per wait)
            float mx = -INFINITY;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                float sc[64];
                tc::ld32(sbuf + 64 * c2, *reinterpret_cast<uint32_t(*)[32]>(sc));
                tc::ld32(sbuf + 64 * c2 + 32, *reinterpret_cast<uint32_t(*)[32]>(sc + 32));
                tc::wait_ld();
                if (need_mask) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        sc[e] = ((unsigned)(64 * c2 + e - b_lo) <= (unsigned)span) ? sc[e] : -INFINITY;
                }
                float m0 = fmax3(sc[0], sc[1], sc[2]), m1 = fmax3(sc[32], sc[33], sc[34]);
#pragma unroll
                for (int e = 3; e < 31; e += 2) {
                    m0 = fmax3(m0, sc[e], sc[e + 1]);
                    m1 = fmax3(m1, sc[32 + e], sc[32 + e + 1]);
                }
                mx = fmax3(mx, fmaxf(m0, sc[31]), fmaxf(m1, sc[63]));
            }
            const float mx_raw = mx;                          // the row's largest logit of the tile (S units)
            mx = mx == -INFINITY ? -INFINITY : mx * c_qk;     // log2 units
            const bool need = mx > m_run + 8.f;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? fmaxf(m_run, mx) : m_run;
                const float corr = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
                if (kx > 0) {
                    // S of this tile is complete, so every earlier MMA (P V of the previous
                    // tile included) has completed: O holds P V of the tiles before
                    if (!(ok = wwait(bar(B_PV_DONE + x), (kx - 1) & 1))) break;
                    tc::fence_after();
                    uint32_t o[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tc::ld32(obuf + c * 32, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                        tc::st32(obuf + c * 32, o);
                    }
                    tc::wait_st();
                }
                l_run *= corr;
                lc_run *= corr;
                m_run = m_new;
            }
            // pass 2: P = exp2(S * c - m) per 32 columns; P chunk c (bf16 pairs) goes to packed
            // columns [16 c, 16 c + 16), which only overlap S columns already read
            const float ref = m_run == -INFINITY ? 0.f : m_run;
            const float2 cq = make_float2(c_qk, c_qk), nref = make_float2(-ref, -ref);
            if (mx_raw != -INFINITY) {
                // the tile's largest P of this row, computed as its element is, and its bf16 rounding
                const float pm = fast_exp2(fmaf(mx_raw, c_qk, -ref));
                lc_run += bf16_lo(pack_bf16(pm, 0.f)) - pm;
            }
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            float scn[32];                                   // the next chunk, loading
            tc::ld32(sbuf, *reinterpret_cast<uint32_t(*)[32]>(scn));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                tc::wait_ld();
                float sc[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) sc[e] = scn[e];
                if (c < 3) tc::ld32(sbuf + 32 * (c + 1), *reinterpret_cast<uint32_t(*)[32]>(scn));
                if (need_mask) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        sc[e] = ((unsigned)(32 * c + e - b_lo) <= (unsigned)span) ? sc[e] : -INFINITY;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 xv = ffma2(make_float2(sc[2 * e], sc[2 * e + 1]), cq, nref);
                    const float2 y = make_float2(fast_exp2(xv.x), fast_exp2(xv.y));
                    l4[e & 3] = fadd2(l4[e & 3], y);
                    pk[e] = pack_bf16(y.x, y.y);
                }
                tc::st16(sbuf + 16 * c, pk);
            }
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l_run += l2.x + l2.y;
            tc::wait_st();
            tc::fence_before();
            if (!(A.withhold && x == 0 && kx == 0)) mbar_arrive(bar(B_P_FULL + x));
            ++kx;
        }
        // epilogue: O / l for this row
        if (ok && tile_valid && kx > 0) ok = wwait(bar(B_PV_DONE + x), (kx - 1) & 1);
        if (ok && tile_valid && kx > 0) {
            tc::fence_after();
            const float inv = (l_run + lc_run) > 0.f ? 1.f / (l_run + lc_run) : 0.f;
            const bool valid = row < q_len;
            const size_t qrow = (size_t)(start + row) * p.Hq + h;
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                tc::ld32(obuf + c * 32, o);
                tc::wait_ld();
                if (!valid) continue;
                const int col = c * 32;
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
            if (valid && p.lse) {
                const float ref = m_run == -INFINITY ? 0.f : m_run;
                p.lse[qrow] = l_run > 0.f ? (ref + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
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

cudaError_t launch_prefill_2q(const inkattn_attn_params &p, const AttnScalars &s, const CUtensorMap &qmap,
                              const CUtensorMap &kmap, const CUtensorMap &vmap, cudaStream_t stream) {
    Tc2Args a;
    a.p = p;
    a.scale = s.scale;
    const int n_qtiles = (p.max_seqlen_q + kRows - 1) / kRows;
    a.n_pairs_max = (n_qtiles + 1) / 2;
    a.kv_rows = (long long)p.num_blocks * p.Hkv * kBlock;
    a.wait_ns = kernel_debug().wait_ns;
    a.withhold = kernel_debug().withhold;
    cudaError_t err = cudaFuncSetAttribute(k_prefill_2q, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    dim3 grid(p.Hq, a.n_pairs_max, p.B);
    return launch_dependent(k_prefill_2q, grid, dim3(kThreads), kSmem, stream, 1, a, qmap, kmap, vmap);
}

}  // namespace inkattn
