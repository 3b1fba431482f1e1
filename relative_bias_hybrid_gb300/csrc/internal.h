// internal.h -- launchers shared between the entry points (api.cu) and the kernel files.
// Each launcher assumes its params were validated by api.cu and returns the CUDA
// error of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/inkattn.h"

namespace inkattn {

constexpr int kHeadDim = 128;
constexpr int kBlock = 64;          // paged-cache block (tokens)

// Settings of the bounded device waits, read once per process.  In normal use every wait
// gives up after 1 s and nothing is withheld.  A test of the failure path sets the
// environment variables INKATTN_TEST_WAIT_LIMIT_US (a shorter limit, 100 us .. 10 s) and
// INKATTN_TEST_WITHHOLD_ARRIVAL=1 (the attention kernels' softmax withholds its first
// arrival on the barrier the MMA warp waits on before P V, and the qkvr kernel's odd CTAs
// their first accumulator release, so that wait runs out and the kernel winds down through
// its error path).
struct KernelDebug {
    uint64_t wait_ns;
    int withhold;
};
const KernelDebug &kernel_debug();

// Host checks shared by the entry points (api.cu).  validate_decode_call makes, in order,
// the checks inkattn_decode makes before it resolves the split count: the params, the
// decode shape, where q / k_cache / v_cache live, and the device (its SM count to *sms).
inkattn_status validate_decode_call(const inkattn_attn_params *p, int *sms);
int pick_splits(const inkattn_attn_params &p, int num_sms);
size_t decode_workspace_bytes(const inkattn_attn_params &p, int S);   // 0 when S <= 1

// Launches `kernel` as a programmatic dependent of the work before it on `stream` (see
// grid_dep_wait in common.cuh), optionally as clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Resolved per-call scalars of an attention call (host-computed).
struct AttnScalars {
    float scale;          // softmax scale (1/sqrt(128) by default)
    int group;            // Hq / Hkv
};

cudaError_t launch_prologue(const inkattn_prologue_params &p, cudaStream_t stream);
cudaError_t launch_output_conv(const inkattn_output_conv_params &p, cudaStream_t stream);
// The E4M3 cache blocks a prefill batch reads, expanded to bf16 copies (k_out, v_out:
// [B * max_blocks_per_seq][Hkv][64][128]) with their block table (table_out: [B][max_blocks_per_seq]).
cudaError_t launch_dequant_e4m3(const inkattn_attn_params &p, inkattn_bf16 *k_out, inkattn_bf16 *v_out,
                                int32_t *table_out, cudaStream_t stream);
// qkvr projections with the prologue in their epilogue; xmap / wmap from make_qkvr_maps
cudaError_t launch_qkvr(const inkattn_qkvr_params &p, const CUtensorMap &xmap, const CUtensorMap &wmap,
                        int num_sms, cudaStream_t stream);
// TMA descriptors of x as [max(N_tok, 1)][d_model] and w as [F][d_model] bf16, box 64
// columns x 128 rows, 128-byte swizzle.  Returns false on failure.
bool make_qkvr_maps(const inkattn_qkvr_params &p, CUtensorMap *xmap, CUtensorMap *wmap);

// Decode: S = num_splits (>= 1).  ws_o / ws_lse are unused when S == 1.
constexpr int kDecodeMaxRows = 128;     // max_seqlen_q * group
constexpr int kDecodeMaxSplits = 64;
constexpr int kDecodeCtasPerSm = 1;     // design occupancy used by the split heuristic
constexpr int kDecodeMinSplitBlocks = 8; // a split streams at least 8 cache blocks (512 keys)
// Fraction of the SMs whose decode CTAs together saturate HBM: one CTA streams K/V at about
// 40 B/clk (its MMAs take ~1600 cycles per 64 KB tile), HBM gives ~23 B/clk per SM.
constexpr double kDecodeHbmSmFrac = 0.6;
constexpr double kCombineCostBlocks = 600.0; // fixed cost of the combine launch (~3 us), in block loads
cudaError_t launch_combine(const inkattn_attn_params &p, int num_splits, const float *ws_o,
                           const float *ws_lse, cudaStream_t stream);

// tcgen05 prefill: 128 query rows per CTA, d_r = 32.
constexpr int kPrefillTcRows = 128;
cudaError_t launch_prefill_tc(const inkattn_attn_params &p, const AttnScalars &s, const CUtensorMap &qmap,
                              const CUtensorMap &kmap, const CUtensorMap &vmap, cudaStream_t stream);
// prefill without relative bias: two query tiles per CTA
cudaError_t launch_prefill_2q(const inkattn_attn_params &p, const AttnScalars &s, const CUtensorMap &qmap,
                              const CUtensorMap &kmap, const CUtensorMap &vmap, cudaStream_t stream);

// TMA descriptor for a paged cache viewed as [num_blocks*Hkv*64 rows][128] bf16,
// box 64 rows x 64 columns, 128-byte swizzle.  Returns false on failure.
bool make_cache_map(CUtensorMap *map, const void *base, long long rows);
// The same rows as E4M3 codes: [num_blocks*Hkv*64 rows][128] bytes, box 64 rows x 128 bytes,
// no swizzle (the decode's converter warps read it row by row).
bool make_cache_map_e4m3(CUtensorMap *map, const void *base, long long rows);
// TMA descriptor for q viewed as [N_tok][Hq][128] bf16, box {64, 1, box_rows}, 128-byte swizzle.
bool make_q_map(CUtensorMap *map, const void *base, int n_tok, int hq, int box_rows);
// Q as [N_tok][Hq][128] with a box of {64 dims, `group` heads, `tokens` tokens}: the rows of
// one KV head's query heads for consecutive tokens, in (token, head) order.
bool make_q_group_map(CUtensorMap *map, const void *base, int n_tok, int hq, int group, int tokens);
cudaError_t launch_decode_tc(const inkattn_attn_params &p, const AttnScalars &s, int num_splits,
                             float *ws_o, float *ws_lse, const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, cudaStream_t stream);

}  // namespace inkattn
