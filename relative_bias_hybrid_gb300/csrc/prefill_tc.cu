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
// One CTA per (128-query tile of one sequence, query head), 16 warps in four warpgroups:
//   warp 0      MMA issuer (the whole warp, one elected lane issuing): S = Q K^T (operands
//               in shared memory), O += P V (P read from TMEM).
//   warp 1      producer: TMA loads of the Q tile and of 128-key K/V tiles (two 64-key
//               cache blocks, two 64-column boxes each, 128-byte swizzle) into a 3-slot ring.
//   warps 2-3   idle (they complete the first warpgroup's register hand-back).
//   warps 4-7   relative bias: the band's R chunks (below), issued by warp 4, and their move
//               from TMEM into the bias rows.
//   warps 8-15  softmax: two warpgroups; row i (TMEM lane i) is shared by one thread of
//               each, which own its key columns [0, 64) and [64, 128).
// The MMA and TMA warps have the lowest warp numbers: among warps ready to issue, the
// scheduler favours those, and every instruction on the MMA warp's path (barrier checks,
// commits, loop) is on the critical path of the tile pipeline, while the softmax warps
// beside it on each SM sub-partition always have independent work.
// Registers are moved between warpgroups at the start (setmaxnreg): the softmax threads,
// which keep 64 logits and their P live, get 176 each; the bias warps 104; TMA and MMA 56.
// TMEM (512 columns): O [0,128) | S0 [128,256) | S1 [256,384) | R [384,512).  P (bf16)
// overwrites the first 64 columns of its S buffer.  S is double-buffered so Q K^T of the
// next tile runs while the softmax works on this one.
//
// Key tiles are walked nearest-first (from the diagonal outwards).  With D_n the offset
// i0 - j0 of tile n (i0 = the tile's first query position, j0 = the key tile's first key),
// row a of tile n needs distances D_n + a - b for its 128 keys b: a window that shifts with
// the row (the shear).  The windows of consecutive tiles abut, so the band is covered by
// chunks C_n = [D_n, D_n + 127] of 128 distances, one new chunk per tile (plus
// C_{-1} = [D_0 - 128, D_0 - 1] before the first, which only reaches keys past the diagonal
// and is skipped when D_0 = 0).  For each chunk the bias warps compute
// R^T[x][a] = P_h[:, D_n + x] . r_a (M = 128 distances, N = 128 rows, K = d_r) into TMEM;
// value x of row a is the bias of key column a - x of tile n when x <= a and of column
// a + 128 - x of tile n + 1 when x > a.  The thread of TMEM lane x writes both into
// 128-entry 16-bit rows indexed by key column, one per tile, alternating between two
// buffers: tile n's row is complete once C_n is moved, and C_{n+1} can be computed as soon
// as C_n has left TMEM, so the chunks run ahead of the softmax, which reads its bias row
// with sequential 16-byte loads.  Tiles farther than rel_extent skip all of this.
// The bias MMA takes bf16 operands: r as given, and P_h (times 1/scale, so that R is in
// the units of S) split into high and low bf16 parts, two products accumulated in fp32.
// The bias rows hold 16-bit fixed point (offset binary) with one step per chunk:
// |R[a][delta]| <= |r_a| |P_h[delta]| (Cauchy-Schwarz), so with B_c = max_a |r_a| times the
// largest |P_h[delta]| of chunk c's window, sigma_c = B_c / 32000 bounds every value of
// chunk c with room for rounding.  Row a of tile n holds chunk n's values in columns b <= a
// and chunk n - 1's in columns b > a, so the softmax takes the step of each column from the
// side of the diagonal it is on.  The staged bias is within sigma / 2 of the fp32 value, 16
// bits below the bound; fp16 (11 significant bits) moved logits of |bias| ~ 15 by ~4e-3.
// Each warp publishes its part of B_c when it stores chunk c's window, before its arrival
// on the barrier that the chunk's MMA waits on, so B_c is complete before the chunk is.
//
// Normalisation: O accumulates P V with P rounded to bf16.  With the lazy rescale the
// largest P of a tile is rarely exactly a power of two, and when it dominates the row,
// dividing by the sum of the unrounded P leaves its bf16 rounding (up to 2^-9 of |o|) in the
// output.  So the rounding error of each tile's largest P is added to the row's normaliser
// (a few instructions per tile); the LSE uses the sum of the fp32 P.
//
// The softmax runs in the log2 domain and keeps a stale row maximum unless the new one
// exceeds it by more than 8 (P stays below 2^8); only then is O rescaled in TMEM.  Column
// pairs go through paired fp32 instructions (fma/add .f32x2) and every exp2 through the
// special-function unit: its 16 a clock per SM leave it below the tile period, while each
// extra instruction of the softmax warps takes an issue slot from the MMA warp beside them.
// (A polynomial exp2 on the FMA pipe for three pairs in eight was 5-6% slower.)
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace inkattn {

namespace {

constexpr int kRows = 128;                 // query rows per CTA (MMA M)
constexpr int kKeys = 128;                 // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kSlots = 3;                  // K/V ring slots
constexpr int kSlotBytes = 32768;          // one K or V tile: [d half][128 keys][128 B]
constexpr int kThreads = 512;            // warp 0 MMA, 1 TMA, 2-3 idle, 4-7 bias, 8-15 softmax
constexpr int kWarpMma = 0, kWarpProducer = 1, kWarpBias = 4, kWarpSoftmax = 8;
constexpr int kStageStride = 136;          // halves per row of the bias buffer
constexpr int kMaxDr = 32;                 // d_r (the relative features fill one 64-byte bf16 row)
constexpr int kWin64 = 128 * kMaxDr * 2;  // [128 rows][32 bf16], K-major 64-byte rows

constexpr int kOffQ = 0;
constexpr int kOffKV = 32768;
constexpr int kOffPwHi = kOffKV + kSlots * kSlotBytes;        // P window, bf16 high parts
constexpr int kOffPwLo = kOffPwHi + kWin64;                     // P window, bf16 low parts
constexpr int kOffRfeat = kOffPwLo + kWin64;                    // relative features (bf16)
constexpr int kOffStage = kOffRfeat + kWin64;                   // two bias buffers
constexpr int kStageBuf = kRows * kStageStride;                 // halves per bias buffer
constexpr int kOffXchg = kOffStage + 2 * kStageBuf * 2;         // row maxima / sums of the two halves
constexpr int kOffNorm = kOffXchg + 3 * 2 * kRows * 4;          // bias bounds and tile scales (below)
constexpr int kOffBar = kOffNorm + 64;
// kOffNorm: float wmax[2][4] (per window parity and bias warp: max |P_h row|^2 of the window,
// S units), float rmax[4] (per bias warp: max |r row|^2), float sigma[4] (the fixed-point
// step of chunk c in entry (c + 1) & 3, c >= -1)

// mbarrier indices, laid out from the slot count so that no two ranges overlap
enum Bar {
    B_Q = 0,
    B_KV_FULL = 1,
    B_KV_EMPTY = B_KV_FULL + kSlots,
    B_S_FULL = B_KV_EMPTY + kSlots,
    B_P_FULL = B_S_FULL + 2,
    B_PV_DONE = B_P_FULL + 2,
    B_R_FULL = B_PV_DONE + 2,
    B_R_EMPTY = B_R_FULL + 1,
    B_PW_READY = B_R_EMPTY + 1,
    B_DRAIN = B_PW_READY + 1,
    B_STAGE_FULL = B_DRAIN + 1,
    B_STAGE_EMPTY = B_STAGE_FULL + 2,
    B_BDRAIN = B_STAGE_EMPTY + 2,
    B_NORM = B_BDRAIN + 1,
    B_COUNT = B_NORM + 1
};
constexpr int kSmem = kOffBar + B_COUNT * 8 + 16;
static_assert(kSmem <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
static_assert(kOffBar % 8 == 0 && kOffKV % 1024 == 0 && kOffStage % 16 == 0, "alignment of the regions");

constexpr uint32_t kTmemO = 0, kTmemS0 = 128, kTmemR = 384;
constexpr int kBarPair = 8;                // named barriers 8-11: the softmax row pairs, per lane quarter

struct TcArgs {
    inkattn_attn_params p;
    float scale;            // softmax scale
    int n_qtiles_max;       // gridDim.y
    long long kv_rows;      // rows of the cache tensor maps (OOB row = this)
    uint64_t wait_ns;       // limit of every bounded wait
    int withhold;           // failure-path test: the softmax withholds its first P arrival
};

// byte offset of 16-byte chunk j of row r in a K-major tile of 64-byte rows with the 64-byte
// swizzle (address bits 4-5 XOR bits 7-8)
__device__ __forceinline__ uint32_t sw64_chunk(int r, int j) {
    return (uint32_t)(r * 64 + (((j ^ (r >> 1)) & 3) << 4));
}

}  // namespace

template <int kCluster>
__global__ void __launch_bounds__(kThreads, 1)
k_prefill_tc(const TcArgs A, const __grid_constant__ CUtensorMap qmap,
             const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    grid_dep_wait();                                   // q and the cache: written by the prologue
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
        const bool r = mbar_wait(addr, parity, p.dev_status, abort_flag, A.wait_ns);
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
            mbar_init(bar(B_STAGE_FULL + s), 128);
            mbar_init(bar(B_STAGE_EMPTY + s), 256);
            mbar_init(bar(B_PV_DONE + s), 1);
        }
        mbar_init(bar(B_R_FULL), 1);
        mbar_init(bar(B_R_EMPTY), 128);
        mbar_init(bar(B_PW_READY), 128);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_BDRAIN), 1);
        mbar_init(bar(B_NORM), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
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

    // Registers: the kernel is launched with 128 a thread (64 K in all).  Each warpgroup sets
    // its own budget first thing in its branch: the softmax threads keep 64 logits and their
    // P live (176), the bias warps a 32-column TMEM load and a P window in flight (104), TMA and
    // MMA little (56).
    if (warp < kWarpBias) {
      tc::reg_dealloc<56>();
      if (warp == kWarpProducer) {
        // ================================ producer ================================
        bool ok = true;
        const uint32_t q_dst = s_base + kOffQ;
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            mbar_arrive_expect_tx(bar(B_Q), 2 * 16384);
            tma_load_3d(q_dst, &qmap, 0, h, start + row0, bar(B_Q));
            tma_load_3d(q_dst + 16384, &qmap, 64, h, start + row0, bar(B_Q));
        }
        int kv_loads = 0;                       // K/V tiles issued, in the MMA warp's order
        auto load_kv = [&](int n, int isv) -> bool {
            const int L = kv_loads++, slot = L % kSlots;
            const int t = t_hi - n;
            // the tile's block-table entries are read before the wait for the slot, so that
            // their round trip to memory overlaps it instead of delaying the copy
            constexpr int kHalves = 3 - kCluster;
            int blk[kHalves];                                // -2: past the sequence end
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) {
                const int lb = 2 * t + (kCluster > 1 ? (int)crank : hh);   // logical cache block
                blk[hh] = (long long)lb * kBlock >= T ? -2
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
                mbar_arrive_expect_tx(fb, kSlotBytes);       // both halves land in every CTA
                const void *map = isv ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
#pragma unroll
                for (int hh = 0; hh < kHalves; ++hh) {
                    const int half = kCluster > 1 ? (int)crank : hh;
                    long long row = A.kv_rows;                   // past the tensor: TMA fills zeros
                    if (blk[hh] != -2) {
                        if (blk[hh] >= 0 && blk[hh] < p.num_blocks) row = ((long long)blk[hh] * p.Hkv + hk) * kBlock;
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
        // the MMA warp consumes K_0, then per tile n >= 1: K_n, V_{n-1}, and finally V_{N-1};
        // loading in that order lets K_{n+1} reuse the slot of V_{n-2} instead of waiting for
        // V_{n-1} to be consumed
        ok = load_kv(0, 0);
        for (int n = 1; n < N && ok; ++n) {
            ok = load_kv(n, 0);
            if (ok) ok = load_kv(n - 1, 1);
        }
        if (ok) ok = load_kv(N - 1, 1);
        // nothing may still be landing in shared memory when the CTA tears down, also when a
        // role gave up: every copy issued and not yet consumed is waited for (a slot is only
        // reloaded after its previous copy was consumed, so those are the last kSlots)
        if (lane == 0) {
            mbar_drain(bar(B_Q), 0, p.dev_status, A.wait_ns);
            for (int L = max(0, kv_loads - kSlots); L < kv_loads; ++L)
                mbar_drain(bar(B_KV_FULL + L % kSlots), (L / kSlots) & 1, p.dev_status, A.wait_ns);
        }
      } else if (warp == kWarpMma) {
        // ================================ MMA issuer ================================
        const uint32_t id_qk = tc::idesc(128, 128, tc::kFmtBF16, 0, 0);
        const uint32_t id_pv = tc::idesc(128, 128, tc::kFmtBF16, 0, 1);
        // Base descriptors, built once; the per-slot and per-k-step ones differ only in the
        // start address field (bits 0-13, 16-byte units), which never carries out of its 14
        // bits since shared-memory addresses stay below 256 KB.  The whole warp runs this
        // loop with the same values in every lane (the MMAs and commits are warp-collective).
        const uint64_t dq = tc::sdesc_sw128(s_base + kOffQ, 16, 1024);
        const uint64_t dk0 = tc::sdesc_sw128(s_base + kOffKV, 16, 1024);
        const uint64_t dv0 = tc::sdesc_sw128(s_base + kOffKV, 16384, 1024);
        auto slot_off = [](int slot) { return (uint64_t)(slot * (kSlotBytes >> 4)); };
        bool ok = wwait(bar(B_Q), 0);

        // K/V tiles consumed, in load order: slot and phase kept as counters (this warp's
        // instructions are on the critical path of every tile)
        int c_slot = 0, c_L = 0;
        uint32_t c_par = 0;
        const int first_last = 2 * N - kSlots;   // loads from here on are not reused
        auto next_tile = [&](int &slot, bool &last) -> bool {
            slot = c_slot;
            const uint32_t par = c_par;
            last = c_L++ >= first_last;
            if (++c_slot == kSlots) {
                c_slot = 0;
                c_par ^= 1u;
            }
            return wwait(bar(B_KV_FULL + slot), par);
        };
        // only the nearest key tile can hold keys at or past the sequence end inside a
        // loaded cache block (when T is not a multiple of the block size)
        const bool zero_tail = (T % kBlock) != 0 && t_hi == (T - 1) / kKeys;
        // A K/V slot may be refilled once the MMAs issued so far have read it: each MMA group
        // ends with that release (in every CTA of the cluster), except for a slot with no
        // later load, so that no arrival reaches a peer that has finished.
        auto issue_pv = [&](int m) -> bool {
            if (!wwait(bar(B_P_FULL + (m & 1)), (m >> 1) & 1)) return false;
            int slot;
            bool last;
            if (!next_tile(slot, last)) return false;
            // keys at or past the sequence end inside a loaded block: zero their V rows so
            // that P = 0 there contributes exact zeros whatever the cache slots hold
            if (m == 0 && zero_tail) {
                const int j0 = t_hi * kKeys;
                const int nvalid = T - j0;
                const int nload = min(kKeys, (int)(((long long)((T + kBlock - 1) / kBlock)) * kBlock - j0));
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
            tc::mma_bf16_ts_k128_commit<(kCluster > 1)>(
                tmem + kTmemO, tmem + kTmemS0 + (uint32_t)(m & 1) * 128, dv0 + slot_off(slot), id_pv,
                m > 0 ? 1u : 0u, bar(B_PV_DONE + (m & 1)), bar(B_KV_EMPTY + slot), last ? 0u : 1u, kPeers);
            __syncwarp();
            return true;
        };

        for (int n = 0; n < N && ok; ++n) {
            int slot;
            bool last;
            ok = next_tile(slot, last);
            if (!ok) break;
            tc::fence_after();
            tc::mma_bf16_ss_k128_commit<(kCluster > 1)>(
                tmem + kTmemS0 + (uint32_t)(n & 1) * 128, dq, dk0 + slot_off(slot), id_qk, 0u,
                bar(B_S_FULL + (n & 1)), bar(B_KV_EMPTY + slot), last ? 0u : 1u, kPeers);
            __syncwarp();
            if (n >= 1) ok = issue_pv(n - 1);
        }
        if (ok) ok = issue_pv(N - 1);
        // every MMA of this CTA has completed before TMEM is released (also after a role gave up)
        tc::commit(bar(B_DRAIN));
        __syncwarp();
        (void)mbar_drain(bar(B_DRAIN), 0, p.dev_status, A.wait_ns);
        __syncwarp();
      }
    } else if (warp < kWarpSoftmax) {
        // ============================== relative bias ==============================
        tc::reg_dealloc<104>();
        // R is computed transposed, R^T[x][a] = P_h[:, D + 1 + x] . r_a (M = 128 distances,
        // N = 128 rows), so this thread (TMEM lane x) holds position x of the chunk for every
        // row a, in column a.  Its value for row a goes to column a - x of tile n's bias row
        // when x <= a and to column a + 128 - x of tile n + 1's when x > a: for a fixed
        // thread both are one base address plus a per-row constant, so every value is one
        // store with an immediate offset, and the 32 lanes of a store write 32 consecutive
        // columns of one row.  Tiles alternate between two bias buffers, so a chunk is
        // moved out of TMEM as soon as it is computed and the next one can follow: the chunks
        // run a tile ahead of the softmax.
        //
        // The MMA takes bf16 operands: r exactly, and P_h split into a high and a low bf16
        // part (P = hi + lo to 16 significant bits), two products accumulated in fp32.
        const int w = warp - kWarpBias;                       // TMEM lane quarter
        const int x = 32 * w + lane;
        const uint32_t lane_off = (uint32_t)(w * 32) << 16;
        bool ok = true;
        float *wmax = reinterpret_cast<float *>(smem + kOffNorm);       // [2][4]
        float *rmax = wmax + 8;                                          // [4]
        float *sigma_s = wmax + 12;                                      // [4]
        if (n_band > 0) {
            // row x's relative features (bf16 as given), and the largest |r_a|^2 of each warp
            {
                const int row = row0 + x;
                uint4 u[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                              make_uint4(0, 0, 0, 0)};
                if (row < q_len) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.r + ((size_t)(start + row) * p.Hq + h) * d_r);
#pragma unroll
                    for (int j = 0; j < 4; ++j) u[j] = __ldg(src + j);
                }
                float n2 = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<uint4 *>(smem + kOffRfeat + sw64_chunk(x, j)) = u[j];
                    const uint32_t wd[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        n2 = fmaf(bf16_lo(wd[e]), bf16_lo(wd[e]), n2);
                        n2 = fmaf(bf16_hi(wd[e]), bf16_hi(wd[e]), n2);
                    }
                }
                // squares are >= 0, so their bit patterns order like the values
                const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(n2));
                if (lane == 0) rmax[w] = __uint_as_float(m);
            }
            // row x of the P window of chunk rho - 1 (rho = 0 is C_{-1}): distance
            // D_{rho-1} + x; distances outside [0, rel_extent) have no bias (zeros)
            const float *Ph = p.P + (size_t)h * p.rel_extent * d_r;
            auto load_p = [&](int rho, float4 (&v)[8]) {
                const long long d = (long long)p_lo - (long long)kKeys * (t_hi - (rho - 1)) + x;
                if (d >= 0 && d < p.rel_extent) {
                    const float4 *src = reinterpret_cast<const float4 *>(Ph + (size_t)d * d_r);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = __ldg(src + j);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            };
            // windows stored so far; window k publishes its per-warp max |P row|^2 in wmax[k & 1]
            // and completes phase k of B_NORM
            int n_win = 0;
            auto store_p = [&](const float4 (&v)[8]) {
                float2 a2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};   // |row|^2 in four independent chains
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float f[8] = {v[2 * j].x * inv_scale, v[2 * j].y * inv_scale, v[2 * j].z * inv_scale,
                                        v[2 * j].w * inv_scale, v[2 * j + 1].x * inv_scale, v[2 * j + 1].y * inv_scale,
                                        v[2 * j + 1].z * inv_scale, v[2 * j + 1].w * inv_scale};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hi[e] = pack_bf16(f[2 * e], f[2 * e + 1]);
                        lo[e] = pack_bf16(f[2 * e] - bf16_lo(hi[e]), f[2 * e + 1] - bf16_hi(hi[e]));
                        const float2 fe = make_float2(f[2 * e], f[2 * e + 1]);
                        a2[e] = ffma2(fe, fe, a2[e]);
                    }
                    *reinterpret_cast<uint4 *>(smem + kOffPwHi + sw64_chunk(x, j)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(smem + kOffPwLo + sw64_chunk(x, j)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                const float2 t2 = fadd2(fadd2(a2[0], a2[1]), fadd2(a2[2], a2[3]));
                const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(t2.x + t2.y));
                if (lane == 0) wmax[(n_win & 1) * 4 + w] = __uint_as_float(m);
                mbar_arrive(bar(B_NORM));
                ++n_win;
                fence_proxy_async_smem();
                mbar_arrive(bar(B_PW_READY));
            };
            // bound B_k = max_a |r_a| * max |P row| over window k (S units), once all four warps
            // have published it
            auto bound = [&](int k, float &out) -> bool {
                if (!wwait(bar(B_NORM), k & 1)) return false;
                const float *wm = wmax + (k & 1) * 4;
                const float pm = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
                const float rm = fmaxf(fmaxf(rmax[0], rmax[1]), fmaxf(rmax[2], rmax[3]));
                out = sqrtf(pm) * sqrtf(rm);
                return true;
            };
            // fixed-point step of chunk c (bounded by b_c; no value of a zero bound), published for
            // the softmax in sigma entry (c + 1) & 3; returns 1 / step
            auto set_step = [&](int c, float b) {
                const float sg = fmaxf(b, 1e-30f) * (1.f / 32000.f);
                if (x == 0) sigma_s[(c + 1) & 3] = sg;
                return 1.f / sg;
            };

            const uint32_t id_r = tc::idesc(128, 128, tc::kFmtBF16, 0, 0);
            const uint64_t dhi = tc::sdesc_sw64(s_base + kOffPwHi, 16, 512);
            const uint64_t dlo = tc::sdesc_sw64(s_base + kOffPwLo, 16, 512);
            const uint64_t dr = tc::sdesc_sw64(s_base + kOffRfeat, 16, 512);
            // the first bias warp issues the ci-th chunk once its window is in place and every
            // thread has moved the previous chunk out of TMEM; K = 32 in two steps of 16 (32 B)
            auto issue = [&](int ci) -> bool {
                if (w != 0) return true;
                if (ci >= 1 && !wwait(bar(B_R_EMPTY), (ci - 1) & 1)) return false;
                if (!wwait(bar(B_PW_READY), ci & 1)) return false;
                tc::fence_after();
                tc::mma_bf16_ss(tmem + kTmemR, dhi, dr, id_r, 0u);
                tc::mma_bf16_ss(tmem + kTmemR, dhi + 2, dr + 2, id_r, 1u);
                tc::mma_bf16_ss(tmem + kTmemR, dlo, dr, id_r, 1u);
                tc::mma_bf16_ss(tmem + kTmemR, dlo + 2, dr + 2, id_r, 1u);
                tc::commit(bar(B_R_FULL));
                __syncwarp();
                return true;
            };
            constexpr int kRowStep = kStageStride + 1;        // (row a, column a - x) -> next row
            unsigned short *const stage = reinterpret_cast<unsigned short *>(smem + kOffStage);
            // rows [32 j, 32 j + 32) of the chunk: the part for tile n (first) or for tile
            // n + 1 (second), into bias buffer buf, as fixed point with step 1 / inv_sig
            auto drain_block = [&](int j, bool first, int buf, float inv_sig) {
                uint32_t r[32];
                tc::ld32(tmem + kTmemR + lane_off + 32 * j, r);
                tc::wait_ld();
                unsigned short *base = stage + buf * kStageBuf + (first ? -x : 128 - x) + 32 * j * kRowStep;
                if (j != w) {                                  // every lane's x is on one side
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 v = fix16_encode2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), inv_sig);
                        base[e * kRowStep] = fix16_bits(v.x);
                        base[(e + 1) * kRowStep] = fix16_bits(v.y);
                    }
                } else {                                       // row 32 w + e vs x = 32 w + lane
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 v = fix16_encode2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), inv_sig);
                        if ((lane <= e) == first) base[e * kRowStep] = fix16_bits(v.x);
                        if ((lane <= e + 1) == first) base[(e + 1) * kRowStep] = fix16_bits(v.y);
                    }
                }
            };
            // C_{-1} gives tile 0 its columns past the diagonal (a + 1 .. 127), at distances
            // D_0 - 128 + x; when the tile sits on the diagonal (D_0 = 0) they are all future
            // keys, masked, and C_{-1} is skipped
            const bool need_prev = p_lo - kKeys * t_hi != 0;
            int ci = 0;                                        // chunks issued
            float4 pv[8];
            // window k of the chunks (k = c + 1 with C_{-1}, k = c without) is stored before its
            // chunk's MMA, so its bound is complete once the chunk is (see above)
            const int k_of_c0 = need_prev ? 1 : 0;
            float inv_c = 0.f;                                 // 1 / step of the chunk being moved
            if (need_prev) {
                load_p(0, pv);
                store_p(pv);                                   // window of C_{-1}
                if (ok) ok = issue(0);
                load_p(1, pv);                                 // window of C_0, in flight
                if (ok) ok = wwait(bar(B_R_FULL), 0);
                float b = 0.f;
                if (ok) ok = bound(0, b);
                if (ok) {
                    tc::fence_after();
                    store_p(pv);                               // the MMA has read window 0
                    inv_c = set_step(-1, b);
                    for (int j = 0; j <= w; ++j) drain_block(j, false, 0, inv_c);   // C_{-1}: tile 0, columns (a, 128)
                    tc::fence_before();
                    mbar_arrive(bar(B_R_EMPTY));
                }
                ci = 1;
            } else {
                load_p(1, pv);
                store_p(pv);                                   // window of C_0
            }
            for (int n = 0; n < n_band && ok; ++n, ++ci) {
                const int rho = n + 1;                         // chunk C_n
                const bool more = n + 1 < n_band;              // tile n + 1 is in the band
                if (!(ok = issue(ci))) break;
                if (more) load_p(rho + 1, pv);
                if (!(ok = wwait(bar(B_R_FULL), ci & 1))) break;
                tc::fence_after();
                float b = 0.f;
                if (!(ok = bound(n + k_of_c0, b))) break;      // complete: C_n's MMA has run
                inv_c = set_step(n, b);
                const int bn = n & 1;
                for (int j = w; j < 4; ++j) drain_block(j, true, bn, inv_c);    // tile n, columns [0, a]
                mbar_arrive(bar(B_STAGE_FULL + bn));          // tile n's bias is complete
                if (more) {
                    store_p(pv);                               // the MMA has read this window
                    // tile n + 1 shares its buffer with tile n - 1, whose reads must be done
                    if (n >= 1 && !(ok = wwait(bar(B_STAGE_EMPTY + (bn ^ 1)), ((n - 1) >> 1) & 1))) break;
                    for (int j = 0; j <= w; ++j) drain_block(j, false, bn ^ 1, inv_c);  // tile n + 1, columns (a, 128)
                }
                tc::fence_before();
                mbar_arrive(bar(B_R_EMPTY));
            }
            // the issuing thread's MMAs (and their barrier arrivals) end before teardown
            if (w == 0) {
                tc::commit(bar(B_BDRAIN));
                __syncwarp();
                (void)mbar_drain(bar(B_BDRAIN), 0, p.dev_status, A.wait_ns);
                __syncwarp();
            }
        }
    } else {
        // ================================ softmax ================================
        tc::reg_alloc<176>();
        // Two warpgroups share the 128 rows: warps 4-7 (half 0) and 8-11 (half 1) read the
        // same TMEM lane quarters; thread (half w, row a) owns key columns [64 w, 64 w + 64)
        // of row a.  The two threads of a row exchange row maxima (and, at the end, row
        // sums) through shared memory with a 64-thread named barrier per lane quarter.
        const int quad = warp & 3;
        const int hw = (warp - kWarpSoftmax) >> 2;            // column half
        const int a = quad * 32 + lane;                       // query row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int row = row0 + a;                             // row within the sequence
        const int i_pos = p_lo + a;
        const int cb = 64 * hw;                               // first key column of this thread
        const unsigned short *stage = reinterpret_cast<const unsigned short *>(smem + kOffStage) + a * kStageStride;
        const float *sigma_s = reinterpret_cast<const float *>(smem + kOffNorm) + 12;
        float *xchg = reinterpret_cast<float *>(smem + kOffXchg);   // [2 tiles][2 halves][128 rows]
        // The two threads of each row meet on a named barrier of the row's lane quarter (one
        // warp of each column half, 64 threads): a hardware barrier, quicker than an mbarrier
        // round trip on this path, but with no time limit.  So every thread meets its partner
        // exactly N + 1 times, once per key tile and once at the end: a thread that leaves
        // the tile loop early (a wait that ran out) still makes the meetings it skipped, and
        // its partner, whose next wait then gives up too (the abort flag), does the same.
        auto pair_meet = [&]() { asm volatile("bar.sync %0, 64;" :: "r"(kBarPair + quad) : "memory"); };
        int met = 0;                             // meetings made in the tile loop
        bool ok = true;

        float m_run = -INFINITY, l_run = 0.f;   // l_run: sum of the fp32 P (for the LSE)
        float lc_run = 0.f;                      // bf16 rounding of each tile's largest P (normaliser)
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
                const int bn = n & 1;
                if (!(ok = wwait(bar(B_STAGE_FULL + bn), (n >> 1) & 1))) break;
                const unsigned short *bias_row = stage + bn * kStageBuf;
                // columns b <= a hold chunk n's values, b > a chunk n - 1's
                const float sg_n = sigma_s[(n + 1) & 3], sg_p = sigma_s[n & 3];
                const int split = a - cb;                         // bb <= split: chunk n
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(bias_row + cb + 8 * c8);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int bb = 8 * c8 + 2 * e;
                        const float2 sg = make_float2(bb <= split ? sg_n : sg_p, bb + 1 <= split ? sg_n : sg_p);
                        const float2 f = ffma2(fix16_decode2(wd[e]), sg, make_float2(s[bb], s[bb + 1]));
                        s[bb] = f.x;
                        s[bb + 1] = f.y;
                    }
                }
                mbar_arrive(bar(B_STAGE_EMPTY + bn));
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
            pair_meet();                                          // also: both halves hold S
            ++met;
            mx = fmaxf(mx, xc[(1 - hw) * 128 + a]);
            const float mx_raw = mx;                             // the row's largest logit of the tile (S units)
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
                lc_run *= corr;
                m_run = m_new;
            }
            const float ref = m_run == -INFINITY ? 0.f : m_run;
            const float2 cq = make_float2(c_qk, c_qk), nref = make_float2(-ref, -ref);
            if (hw == 0 && mx_raw != -INFINITY) {
                // the tile's largest P of this row, computed as its element is, and its bf16 rounding
                const float pm = fast_exp2(fmaf(mx_raw, c_qk, -ref));
                lc_run += bf16_lo(pack_bf16(pm, 0.f)) - pm;
            }
            float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                // column pairs, logits to log2 units relative to the running maximum
                const float2 x = ffma2(make_float2(s[2 * e], s[2 * e + 1]), cq, nref);
                const float2 y = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                l4[e & 3] = fadd2(l4[e & 3], y);
                pk[e] = pack_bf16(y.x, y.y);
            }
            // P for keys [64 w, 64 w + 64) -> packed columns [32 w, 32 w + 32) of the buffer
            tc::st32(sbuf + 32 * hw, pk);
            const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
            l_run += l2.x + l2.y;
            tc::wait_st();
            tc::fence_before();
            if (!(A.withhold && n == 0)) mbar_arrive(bar(B_P_FULL + (n & 1)));
        }
        // epilogue: the row sum of both halves, then O / l for this thread's 64 columns
        // the column-half 0 thread of a row alone holds the correction (lc_run is 0 in the other)
        // and alone writes the LSE: it publishes l + lc, the other thread l
        float *xl = xchg + 512;
        for (; met < N; ++met) pair_meet();
        xl[hw * 128 + a] = l_run + lc_run;
        pair_meet();
        const float l_other = xl[(1 - hw) * 128 + a];
        const float l_tot = l_run + l_other;                  // the fp32 sum (read by half 0 only)
        const float l_norm = l_run + lc_run + l_other;        // normaliser of P V's bf16 P
        if (ok) ok = wait_pv(N - 1);
        if (ok) {
            tc::fence_after();
            const float inv = l_norm > 0.f ? 1.f / l_norm : 0.f;
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
    if (warp == kWarpMma) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
    // a CTA leaves only when its peer no longer writes into its shared memory
    if constexpr (kCluster > 1) cluster_sync();
}

cudaError_t launch_prefill_tc(const inkattn_attn_params &p, const AttnScalars &s, const CUtensorMap &qmap,
                              const CUtensorMap &kmap, const CUtensorMap &vmap, cudaStream_t stream) {
    // the warpgroups' register budgets (56 + 104 + 2 x 176 per thread of a warpgroup) add
    // up to the 64 K registers that 512 threads at 128 each are launched with
    // (checked once per process; the static's initialisation is thread-safe)
    static const cudaError_t regs_check = [] {
        cudaFuncAttributes fa1, fa2;
        if (cudaFuncGetAttributes(&fa1, k_prefill_tc<1>) != cudaSuccess ||
            cudaFuncGetAttributes(&fa2, k_prefill_tc<2>) != cudaSuccess)
            return cudaErrorInvalidDeviceFunction;
        return (fa1.numRegs == 128 && fa2.numRegs == 128) ? cudaSuccess : cudaErrorInvalidConfiguration;
    }();
    if (regs_check != cudaSuccess) return regs_check;
    TcArgs a;
    a.p = p;
    a.scale = s.scale;
    a.wait_ns = kernel_debug().wait_ns;
    a.withhold = kernel_debug().withhold;
    a.n_qtiles_max = (p.max_seqlen_q + kRows - 1) / kRows;
    a.kv_rows = (long long)p.num_blocks * p.Hkv * kBlock;
    dim3 grid(p.Hq, a.n_qtiles_max, p.B);
    // head pairs (2i, 2i + 1) share a KV head when the group size is even
    const bool pair = (p.Hq / p.Hkv) % 2 == 0;
    if (!pair) {
        cudaError_t err = cudaFuncSetAttribute(k_prefill_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (err != cudaSuccess) return err;
        return launch_dependent(k_prefill_tc<1>, grid, dim3(kThreads), kSmem, stream, 1, a, qmap, kmap, vmap);
    }
    cudaError_t err = cudaFuncSetAttribute(k_prefill_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    return launch_dependent(k_prefill_tc<2>, grid, dim3(kThreads), kSmem, stream, 2, a, qmap, kmap, vmap);
}

}  // namespace inkattn
