// qkvr.cu -- the qkvr projections of the hidden states on the 5th-generation tensor cores
// (TMA + tcgen05/TMEM), with the attention prologue fused into the GEMM's epilogue.
//
// [vLLM TML Inkling サポート, §TML Inkling モデルアーキテクチャ] and [vLLM hỗ trợ TML Inkling
//  ..., the MoE item of the architecture list]: q, k, v and the relative features r come
//  from one bf16 linear layer ("qkvr linears") in front of the attention.
// [SGLang と Miles が Inkling を初日からサポート, §ShortConv 最適化：融合、グラフキャプチャ、
//  シャーディング]: the K/V conv, the Q/K RMSNorm and the cache write fused so that nothing
//  intermediate goes back to memory; here the projections themselves never do either.
// The prologue's arithmetic is that of prologue.cu: conv correctly rounded to bf16, RMSNorm
// in fp32 over the bf16 row, the same E4M3 row quantisation.
//
// GEMM: y[t][o] = sum_k x[t][k] w[o][k], fp32 accumulation in TMEM, each value rounded once
// to bf16.  Output features in the order [q heads | k | v | r heads].
//
// Tiles.  An M tile is 128 rows of x: the 125 tokens [t0, t0 + 125) of one sequence and the
// 3 tokens before them, whose projections are the conv's history (for a sequence's first
// tile the carried conv state takes their place).  Recomputing those 3 rows (2.4% of the
// MMAs) makes every tile independent: no tile waits for another's projections.  A work item
// is a pair of M tiles (consecutive in the list of all sequences' tiles) times a block of
// 256 output features, computed by the two CTAs of a cluster as one M = 256, N = 256 tile of
// pair MMAs (tcgen05 cta_group::2): each CTA holds its own 128 rows of x and one 128-row
// half of the weight block, and the even CTA issues MMAs that read both CTAs' shared
// memory and write each CTA's 128 rows of D to that CTA's TMEM.  Per SM and MMA step the
// tensor core thus reads 8 KB of operands from shared memory instead of the 12 KB of an
// M = 128, N = 256 MMA, and TMA writes 32 KB per stage instead of 48: shared-memory
// bandwidth, which bounds the single-CTA form near two thirds of the tensor rate, stays
// within reach.  Items go round-robin over a persistent grid of clusters, in groups of 8
// feature blocks with the M pairs fastest inside a group, so that the weight blocks of a
// group stay in L2 while the tiles stream past them.
//
// One CTA per SM, 10 warps:
//   warp 0      producer: TMA of the CTA's A and weight boxes into a 5-stage ring (32 KB a
//               stage; 4 stages ran 12% slower, 3 stages 30%)
//   warp 1      even CTA: MMA issuer (whole warp, one elected lane), M = 256, N = 256,
//               K = 16 steps into one of two TMEM accumulators (2 x 256 columns), so the
//               epilogue of one item overlaps the MMAs of the next (idle in the odd CTA)
//   warps 2-5   epilogue of the item's first 128 features, warps 6-9 of the second: each
//               128-feature block is one q head, one k or v head, or 128 features of r.
// Both CTAs' copies of a stage complete on the even CTA's barrier for it, which the MMA
// warp waits on; the pair MMAs' commits release the stage in both CTAs.  Waits for phases
// completed from the other CTA poll (a suspended waiter is not woken promptly by them).
// Epilogue of a block: each thread moves its TMEM lane (one tile row) to bf16 in a shared
// staging buffer (rows of 272 bytes: row-wise 16-byte and column-wise 2-byte accesses
// are both free of bank conflicts; one buffer, which the two groups use in turn, so that
// the ring can hold 5 stages) and releases the accumulator; a k/v block then runs the
// conv down each channel in place (thread = channel, oldest row first, a 3-value window in
// registers); finally each half-warp takes whole rows (16 lanes x 8 values): RMSNorm for q
// and k, the cache write for k and v, plain stores for q and r.  Rows 0-2 of a sequence's
// first tile are loaded from conv_state_*_in by their own threads; the three staging rows
// that form the new state go to conv_state_*_out before the conv overwrites them.
#include "common.cuh"
#include "conv4.cuh"
#include "fp8.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "cta_pair.cuh"

namespace inkattn {

namespace {

constexpr int kRowsM = 128;                       // MMA M: rows of an M tile
constexpr int kHalo = 3;                          // conv history rows (W - 1)
constexpr int kTileTok = kRowsM - kHalo;          // new tokens per M tile
static_assert(kTileTok == INKATTN_QKVR_TILE_TOKENS, "the tile size the header publishes");
constexpr int kCols = 256;                        // MMA N: output features of an item
constexpr int kKStep = 64;                        // K per ring stage (one 128-byte row)
constexpr int kStages = 5;
constexpr int kABytes = kRowsM * 128;             // 16 KB
constexpr int kBHalfBytes = 128 * 128;            // 16 KB, one CTA's half of the weight box
constexpr int kStageBytes = kABytes + kBHalfBytes;
constexpr int kThreads = 320;
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpEpi = 2;
constexpr int kRowStride = 272;                   // staging row: 256 bytes + 16
constexpr int kStagingBytes = kRowsM * kRowStride;
constexpr int kRaster = 8;                        // feature blocks per raster group
constexpr int kMaxSeqs = INKATTN_QKVR_MAX_SEQS;

constexpr int kOffRing = 0;
constexpr int kOffStaging = kOffRing + kStages * kStageBytes;
constexpr int kOffTiles = kOffStaging + kStagingBytes;            // int tile prefix [B + 1]
constexpr int kOffBar = kOffTiles + ((kMaxSeqs + 1) * 4 + 7) / 8 * 8;
enum Bar {
    B_FULL = 0,
    B_EMPTY = B_FULL + kStages,
    B_ACC_FULL = B_EMPTY + kStages,
    B_ACC_EMPTY = B_ACC_FULL + 2,
    B_DRAIN = B_ACC_EMPTY + 2,
    B_COUNT = B_DRAIN + 1
};
constexpr int kSmem = kOffBar + B_COUNT * 8 + 16;
static_assert(kSmem <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0 && kOffStaging % 16 == 0,
              "swizzled tiles start on 1024-byte boundaries");

struct QkvrArgs {
    inkattn_qkvr_params p;
    int n_cblocks;           // feature blocks: ceil(F / 256)
    uint64_t wait_ns;        // limit of every bounded wait
    int withhold;            // failure-path test: one epilogue warp of each odd CTA withholds
                             // its first accumulator release, so the MMA warp's wait runs out
};

// Named barriers of the epilogue warps: 1 and 2 for one group of 128 threads each, 3 and 4
// for both groups (256 threads).
constexpr int kBarBoth = 3, kBarHandoff = 4;
// bar.sync over n threads, reducing a predicate with AND
__device__ __forceinline__ bool named_all(int id, int n, bool v) {
    int r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
                 "selp.s32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((int)v), "r"(id), "r"(n) : "memory");
    return r != 0;
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void group_sync(int id) { named_sync(id, 128); }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
k_qkvr(const QkvrArgs A, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    grid_dep_wait();                                   // x and the states: written by the work before
    grid_dep_launch();
    const inkattn_qkvr_params &p = A.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const int cid = (int)blockIdx.x >> 1, nclusters = (int)gridDim.x >> 1;
    const uint32_t s_base = smem_u32(smem);
    if ((s_base & 1023u) != 0u) {                      // the same in both CTAs of a cluster
        if (threadIdx.x == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
        return;
    }
    auto bar = [&](int i) { return s_base + kOffBar + 8u * (uint32_t)i; };
    int *s_tiles = reinterpret_cast<int *>(smem + kOffTiles);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + B_COUNT * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + B_COUNT * 8 + 4);
    auto wwait = [&](uint32_t addr, uint32_t parity) -> bool {
        const bool r = mbar_wait(addr, parity, p.dev_status, abort_flag, A.wait_ns);
        return __all_sync(0xffffffffu, r);
    };
    // for phases completed from the other CTA (its commits, its remote arrivals)
    auto cwait = [&](uint32_t addr, uint32_t parity) -> bool {
        const bool r = mbar_wait_cluster(addr, parity, p.dev_status, abort_flag, A.wait_ns);
        return __all_sync(0xffffffffu, r);
    };
    const int C = p.Hkv * kHeadDim;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_FULL + s), 1);                   // (the even CTA's counts both CTAs' copies)
            mbar_init(bar(B_EMPTY + s), 1);                  // released by the pair's MMAs
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_ACC_FULL + s), 1);
            mbar_init(bar(B_ACC_EMPTY + s), 16);             // every epilogue warp of both CTAs
        }
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {                            // with the peer CTA's MMA warp
        tc::tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tc::tmem_relinquish_pair();
    }
    if (warp == kWarpEpi) {
        // tile prefix over the sequences: s_tiles[b] = M tiles of sequences 0 .. b-1
        int carry = 0;
        if (lane == 0) s_tiles[0] = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int tiles = 0;
            if (b < p.B) {
                const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1], slot = p.state_slot[b];
                if (start < 0 || end < start || end > p.N_tok || end - start > p.max_seqlen_q || slot < 0 ||
                    slot >= p.num_state_slots) {
                    set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                } else {
                    tiles = (end - start + kTileTok - 1) / kTileTok;
                }
            }
            int v = tiles;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += n;
            }
            if (b < p.B) s_tiles[b + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    if (warp >= kWarpEpi) {
        // a sequence with no new tokens passes its state from in to out
        const int et = threadIdx.x - kWarpEpi * 32, nthr = kThreads - kWarpEpi * 32;
        const bool ck = p.conv_state_k_out != p.conv_state_k_in, cv = p.conv_state_v_out != p.conv_state_v_in;
        if (ck || cv) {
            for (int b = (int)blockIdx.x; b < p.B; b += (int)gridDim.x) {
                const int start = p.cu_seqlens_q[b], end = p.cu_seqlens_q[b + 1], slot = p.state_slot[b];
                if (start < 0 || end != start || end > p.N_tok || slot < 0 || slot >= p.num_state_slots) continue;
                const size_t base = (size_t)slot * 3 * C;
                for (int i = et; i < 3 * C / 8; i += nthr) {
                    if (ck) reinterpret_cast<uint4 *>(p.conv_state_k_out + base)[i] =
                        reinterpret_cast<const uint4 *>(p.conv_state_k_in + base)[i];
                    if (cv) reinterpret_cast<uint4 *>(p.conv_state_v_out + base)[i] =
                        reinterpret_cast<const uint4 *>(p.conv_state_v_in + base)[i];
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    cluster_sync();                                    // the peer's barriers exist before any multicast
    const uint32_t tmem = *tmem_slot;

    const int m_total = s_tiles[p.B];
    const int m_pairs = (m_total + 1) >> 1;
    const int n_items = m_pairs * A.n_cblocks;
    const int nk = (p.d_model + kKStep - 1) / kKStep;
    // item -> (M tile of this CTA, feature block)
    auto item = [&](int w, int &mt, int &cb) {
        const int grp = w / (kRaster * m_pairs);
        const int rem = w - grp * kRaster * m_pairs;
        const int gsz = min(kRaster, A.n_cblocks - grp * kRaster);
        const int mp = rem / gsz;
        cb = grp * kRaster + (rem - mp * gsz);
        mt = 2 * mp + (int)crank;
    };
    // the sequence of M tile mt < m_total: s_tiles[b] <= mt < s_tiles[b + 1]
    auto seq_of = [&](int mt) {
        int lo = 0, hi = p.B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tiles[mid] <= mt) lo = mid;
            else hi = mid;
        }
        return lo;
    };

    if (warp == kWarpProducer) {
        // ================================ producer ================================
        int L = 0;                                    // stage loads issued
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&wmap);
        }
        for (int w = cid; w < n_items && ok; w += nclusters) {
            int mt, cb;
            item(w, mt, cb);
            int row0 = p.N_tok > 0 ? p.N_tok : 1;     // past the tensor: TMA fills zeros
            if (mt < m_total) {
                const int b = seq_of(mt);
                row0 = p.cu_seqlens_q[b] + (mt - s_tiles[b]) * kTileTok - kHalo;
            }
            const int wrow = cb * kCols + (int)crank * 128;   // this CTA's half of the block
            for (int k = 0; k < nk; ++k, ++L) {
                const int s = L % kStages;
                if (L >= kStages && !cwait(bar(B_EMPTY + s), ((L / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = s_base + kOffRing + (uint32_t)(s * kStageBytes);
                    if (crank == 0) {
                        const uint32_t fb = bar(B_FULL + s);
                        mbar_arrive_expect_tx(fb, 2 * kStageBytes);   // this CTA's copies and the peer's
                        tma_load_2d(dst, &xmap, k * kKStep, row0, fb);
                        tma_load_2d(dst + kABytes, &wmap, k * kKStep, wrow, fb);
                    } else {
                        const uint32_t fb = mapa_shared(bar(B_FULL + s), 0);
                        tma_load_2d_pair(dst, &xmap, k * kKStep, row0, fb);
                        tma_load_2d_pair(dst + kABytes, &wmap, k * kKStep, wrow, fb);
                    }
                }
                __syncwarp();
            }
        }
        // nothing may still be landing in shared memory when the pair tears down: the even
        // CTA waits for the last kStages stages of both CTAs (earlier ones were consumed
        // before their slot was reloaded), and the odd CTA leaves only after it (the
        // cluster barrier at the end)
        if (lane == 0 && crank == 0)
            for (int l = max(0, L - kStages); l < L; ++l)
                mbar_drain(bar(B_FULL + l % kStages), (l / kStages) & 1, p.dev_status, A.wait_ns);
    } else if (warp == kWarpMma && crank != 0) {
        // the odd CTA issues no MMAs
    } else if (warp == kWarpMma) {
        // ================================ even CTA: MMA issuer ================================
        const uint32_t id = tc::idesc(2 * kRowsM, kCols, tc::kFmtBF16, 0, 0);
        const uint64_t da0 = tc::sdesc_sw128(s_base + kOffRing, 16, 1024);
        const uint64_t db0 = tc::sdesc_sw128(s_base + kOffRing + kABytes, 16, 1024);
        // loads of this cluster in all; the last kStages are not released, so that no
        // arrival reaches a peer that has finished
        const int my_items = cid < n_items ? (n_items - cid + nclusters - 1) / nclusters : 0;
        const long long total = (long long)my_items * nk;
        long long L = 0;
        bool ok = true;
        int i = 0;
        for (int w = cid; w < n_items && ok; w += nclusters, ++i) {
            const int buf = i & 1;
            // both CTAs' epilogues are done with this accumulator
            if (i >= 2 && !cwait(bar(B_ACC_EMPTY + buf), ((i >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            tc::fence_after();
            for (int k = 0; k < nk; ++k, ++L) {
                const int s = (int)(L % kStages);
                const uint32_t par = (uint32_t)((L / kStages) & 1);
                if (!cwait(bar(B_FULL + s), par)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint64_t off = (uint64_t)(s * (kStageBytes >> 4));
                tc::mma_pair_bf16_ss_k64_commit(tmem + (uint32_t)(buf * kCols), da0 + off, db0 + off, id,
                                                k > 0 ? 1u : 0u, bar(B_EMPTY + s), L + kStages < total ? 1u : 0u,
                                                bar(B_ACC_FULL + buf), k == nk - 1 ? 1u : 0u);
                __syncwarp();
            }
        }
        // every MMA of the pair has completed before TMEM is released
        tc::commit_pair(bar(B_DRAIN));
        __syncwarp();
        (void)mbar_drain(bar(B_DRAIN), 0, p.dev_status, A.wait_ns);
        __syncwarp();
    } else {
        // ================================ epilogue ================================
        const int e = (warp - kWarpEpi) >> 2;                 // which 128 features of the item
        const int gt = (int)threadIdx.x - kWarpEpi * 32 - e * 128;   // thread within the group
        const int quarter = warp & 3;                         // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;                  // this thread's tile row
        const int gid = 1 + e;                                // named barrier of the group
        unsigned char *stg = smem + kOffStaging;              // one buffer, the groups take turns
        const int hw = gt >> 4, l16 = gt & 15, c0 = l16 * 8;  // row phase: half-warp hw, 8 values
        const int Qw = p.Hq * kHeadDim, F_kv = Qw + 2 * C, Rw = p.Hq * p.d_r;
        float gq[8], gk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            gq[j] = __ldg(p.q_norm_w + c0 + j);
            gk[j] = __ldg(p.k_norm_w + c0 + j);
        }
        const long long slot_limit = (long long)p.num_blocks * kBlock;
        const bool f8 = p.kv_dtype == INKATTN_KV_E4M3;
        int i = 0;
        for (int w = cid; w < n_items; w += nclusters, ++i) {
            int mt, cb;
            item(w, mt, cb);
            const int buf = i & 1;
            const int col0 = cb * kCols + e * 128;            // first feature of the block
            // 0 q, 1 k, 2 v, 3 r, 4 past the features
            const int type = col0 < Qw ? 0 : col0 < Qw + C ? 1 : col0 < F_kv ? 2 : col0 < F_kv + Rw ? 3 : 4;
            const bool live = mt < m_total && type < 4;
            int start = 0, q_len = 0, t0 = 0, nt = 0, slot = 0;
            if (live) {
                const int b = seq_of(mt);
                start = p.cu_seqlens_q[b];
                q_len = p.cu_seqlens_q[b + 1] - start;
                t0 = (mt - s_tiles[b]) * kTileTok;
                nt = min(kTileTok, q_len - t0);
                slot = p.state_slot[b];
            }
            const bool kv = live && (type == 1 || type == 2);
            const int hk = type == 1 ? (col0 - Qw) >> 7 : (col0 - Qw - C) >> 7;
            const inkattn_bf16 *st_in = type == 1 ? p.conv_state_k_in : p.conv_state_v_in;
            inkattn_bf16 *st_out = type == 1 ? p.conv_state_k_out : p.conv_state_v_out;

            // the accumulator is ready; both groups decide together whether to go on (a
            // named barrier must never wait for a group that has left), and the same barrier
            // finds the second group done with the staging rows of the previous item
            bool ok = mbar_wait_cluster(bar(B_ACC_FULL + buf), (uint32_t)((i >> 1) & 1), p.dev_status,
                                        abort_flag, A.wait_ns);
            if (!named_all(kBarBoth, 256, ok)) break;
            tc::fence_after();
            if (e == 1) named_sync(kBarHandoff, 256);         // the first group is done with them
            const bool release = !(A.withhold && i == 0 && crank == 1 && warp == kWarpEpi);
            if (!live) {
                __syncwarp();
                if (lane == 0 && release) mbar_remote_arrive(bar(B_ACC_EMPTY + buf), 0);
                if (e == 0) named_arrive(kBarHandoff, 256);
                continue;
            }

            // ---- TMEM lane `row` -> bf16 staging row (or the carried state, rows 0-2 of a
            // sequence's first tile)
            const bool from_state = kv && t0 == 0 && row < kHalo;
            const size_t st_base = (size_t)slot * 3 * C + (size_t)hk * kHeadDim;
            uint4 *srow = reinterpret_cast<uint4 *>(stg + row * kRowStride);
            const uint32_t taddr = tmem + (uint32_t)(buf * kCols + e * 128) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tc::ld32(taddr + (uint32_t)(c * 32), v);
                tc::wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 o;
                    o.x = pack_bf16(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1]));
                    o.y = pack_bf16(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3]));
                    o.z = pack_bf16(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5]));
                    o.w = pack_bf16(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7]));
                    const int chunk = c * 4 + q4;             // 16-byte chunk of the row
                    if (from_state)
                        o = *reinterpret_cast<const uint4 *>(st_in + st_base + (size_t)row * C + chunk * 8);
                    srow[chunk] = o;
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0 && release) mbar_remote_arrive(bar(B_ACC_EMPTY + buf), 0);   // the even CTA's MMA warp waits
            group_sync(gid);                                  // the staging rows are complete

            if (p.y_out != nullptr) {                         // the projections themselves
                const int F = F_kv + Rw;
                for (int tt = hw; tt < nt; tt += 8)
                    if (col0 + c0 < F)
                        *reinterpret_cast<uint4 *>(p.y_out + (size_t)(start + t0 + tt) * F + col0 + c0) =
                            *reinterpret_cast<const uint4 *>(stg + (kHalo + tt) * kRowStride + l16 * 16);
            }
            // the new state: rows q_len .. q_len + 2 of [carried rows ; new rows], the last
            // three of the staging rows of the sequence's last tile.  Written only now, when
            // every read of the old state (rows 0-2 of the first tile, perhaps this very tile)
            // is done, so that in and out may be one array when the sequence is one tile.
            const bool last_tile = kv && t0 + nt == q_len;
            if (last_tile && gt < kHalo * 16) {
                const int j = gt >> 4, chunk = gt & 15;
                *reinterpret_cast<uint4 *>(st_out + st_base + (size_t)j * C + chunk * 8) =
                    *reinterpret_cast<const uint4 *>(stg + (q_len - t0 + j) * kRowStride + chunk * 16);
            }
            if (kv && (p.y_out != nullptr || last_tile)) group_sync(gid);   // read before the conv

            if (kv) {
                // ---- conv down channel gt, in place, oldest row first
                const float *cw = (type == 1 ? p.conv_w_k : p.conv_w_v) + (size_t)(hk * kHeadDim + gt) * 4;
                const float wr[4] = {__ldg(cw), __ldg(cw + 1), __ldg(cw + 2), __ldg(cw + 3)};
                uint16_t *col = reinterpret_cast<uint16_t *>(stg) + gt;
                constexpr int kHalves = kRowStride / 2;
                float x0 = bf16_bits_to_float(col[0]);
                float x1 = bf16_bits_to_float(col[kHalves]);
                float x2 = bf16_bits_to_float(col[2 * kHalves]);
                for (int r = kHalo; r < kHalo + nt; ++r) {
                    const float x3 = bf16_bits_to_float(col[r * kHalves]);
                    const float xs[4] = {x0, x1, x2, x3};
                    const float y = conv4_bf16_fast(wr, xs);
                    col[r * kHalves] = (uint16_t)(__float_as_uint(y) >> 16);
                    x0 = x1;
                    x1 = x2;
                    x2 = x3;
                }
                group_sync(gid);
            }

            // ---- rows: half-warp hw takes tokens hw, hw + 8, ... of the tile (a trip count
            // uniform over the group, so every lane takes part in the shuffles)
            for (int u = 0; 8 * u < nt; ++u) {
                const int tt = hw + 8 * u;
                const bool valid = tt < nt;
                const int ts = valid ? tt : 0;
                const uint4 raw = *reinterpret_cast<const uint4 *>(stg + (kHalo + ts) * kRowStride + l16 * 16);
                const int tok = start + t0 + ts;
                if (type == 3) {
                    const int rc = col0 - F_kv + c0;          // feature within the r row
                    if (valid && rc < Rw) *reinterpret_cast<uint4 *>(p.r_out + (size_t)tok * Rw + rc) = raw;
                    continue;
                }
                float x[8];
                unpack8(raw, x);
                uint4 outrow = raw;
                if (type != 2) {
                    float ss = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
                    float y[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) y[j] = x[j] * inv * (type == 0 ? gq[j] : gk[j]);
                    outrow = pack8(y);
                }
                if (type == 0) {
                    if (valid)
                        *reinterpret_cast<uint4 *>(p.q_out + ((size_t)tok * p.Hq + (col0 >> 7)) * kHeadDim + c0) =
                            outrow;
                    continue;
                }
                // k or v: the paged cache row of this token
                uint2 codes = make_uint2(0, 0);
                float row_scale = 1.f;
                if (f8) {
                    float r8[8];
                    unpack8(outrow, r8);
                    float am = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(r8[j]));
                    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 8));
                    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
                    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
                    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
                    const int kx = e4m3_row_exponent(am);
                    row_scale = pow2f(kx);
                    codes = e4m3_encode8(r8, pow2f(-kx));
                }
                if (!valid) continue;
                const int sm = __ldg(p.slot_mapping + tok);
                if (sm < 0 || (long long)sm >= slot_limit) {
                    if (l16 == 0) set_status(p.dev_status, INKATTN_ERR_DEVICE_BOUNDS);
                    continue;
                }
                const size_t drow = ((size_t)(sm / kBlock) * p.Hkv + hk) * kBlock + (sm % kBlock);
                const size_t dst = drow * kHeadDim + c0;
                void *cache = type == 1 ? p.k_cache : p.v_cache;
                if (!f8) {
                    *reinterpret_cast<uint4 *>(static_cast<inkattn_bf16 *>(cache) + dst) = outrow;
                } else {
                    *reinterpret_cast<uint2 *>(static_cast<unsigned char *>(cache) + dst) = codes;
                    if (l16 == 0) (type == 1 ? p.k_scale : p.v_scale)[drow] = row_scale;
                }
            }
            if (e == 0) named_arrive(kBarHandoff, 256);       // the staging rows go to the second group
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == kWarpMma) {                            // with the peer CTA's MMA warp
        tc::fence_after();
        tc::tmem_dealloc_pair(tmem, 512);
    }
    cluster_sync();                  // a CTA leaves only when its peer no longer writes into it
}

cudaError_t launch_qkvr(const inkattn_qkvr_params &p, const CUtensorMap &xmap, const CUtensorMap &wmap,
                        int num_sms, cudaStream_t stream) {
    QkvrArgs a;
    a.p = p;
    const long long F = (long long)(p.Hq + 2 * p.Hkv) * kHeadDim + (long long)p.Hq * p.d_r;
    a.n_cblocks = (int)((F + kCols - 1) / kCols);
    a.wait_ns = kernel_debug().wait_ns;
    a.withhold = kernel_debug().withhold;
    cudaError_t err = cudaFuncSetAttribute(k_qkvr, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    // a persistent grid: as many clusters as are resident at once (one CTA per SM), and no
    // more than there can be items (at most N_tok / 125 + B M tiles)
    static const int max_clusters = [num_sms] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2 > 0 ? num_sms / 2 : 1), 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_qkvr, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        return n;
    }();
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const long long m_upper = (long long)p.N_tok / kTileTok + p.B;
    const long long items = ((m_upper + 1) / 2) * a.n_cblocks;
    const int clusters = (int)(items < max_clusters ? (items > 0 ? items : 1) : max_clusters);
    return launch_dependent(k_qkvr, dim3(2 * clusters), dim3(kThreads), kSmem, stream, 2, a, xmap, wmap);
}

}  // namespace inkattn
