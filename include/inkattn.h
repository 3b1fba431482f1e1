/*
 * inkattn.h -- C ABI of libinkattn.so, the GB300 (sm_103a) attention hot path of
 * one Inkling decoder layer.
 *
 * Sources, cited by page title and section heading:
 *   [SG] "SGLang と Miles が Inkling を初日からサポート：975Bのマルチモーダル最先端モデルが公開"
 *        (winzheng.jp review page)
 *   [VJ] "vLLM TML Inkling サポート" (agentlenshq.com, Japanese)
 *   [VV] "vLLM hỗ trợ TML Inkling ngay khi ra mắt với hiệu năng tối ưu" (gpuhub.net)
 *
 * General conventions
 *   - Every pointer inside a params struct is a DEVICE pointer owned by the caller.
 *     The library allocates no device memory at run time: the split-KV partials of
 *     inkattn_decode live in a caller-provided workspace, those of
 *     inkattn_decode_noalloc in a fixed 64 MiB buffer that is part of the library image.
 *   - bf16 tensors are IEEE bfloat16 (inkattn_bf16 holds the raw 16-bit pattern);
 *     all arrays are dense and row-major in the layouts stated per field.
 *   - Every call is asynchronous on the caller's CUDA stream (passed as void*, a
 *     cudaStream_t; NULL = the legacy default stream), keeps no state between calls
 *     and is safe to call from several host threads.
 *   - Kernels are chained by programmatic dependent launch: each may become resident on
 *     the GPU while the kernel before it on the stream finishes, and reads no global
 *     memory before that kernel has completed, so stream order holds as for any launch.
 *     inkattn_prologue, inkattn_output_conv and inkattn_qkvr_prologue let the next kernel
 *     be scheduled once all their CTAs have started; the attention kernels do not.  Every call can be captured
 *     into a CUDA graph.
 *   - Host-side validation runs before any launch; on failure the call returns
 *     INKATTN_ERR_INVALID_ARG or INKATTN_ERR_UNSUPPORTED and launches nothing.
 *   - Alignment: bf16 arrays (activations, caches, conv states, outputs) must be 16-byte
 *     aligned; the fp32 conv weights and RMSNorm gains of inkattn_prologue and
 *     inkattn_qkvr_prologue, the index arrays, lse and dev_status 4-byte aligned; further
 *     rules are stated per entry point.  A pointer that breaks its rule is
 *     INKATTN_ERR_INVALID_ARG.
 *   - Index arrays are read only on the device.  Kernels bounds-check every index
 *     they read (cu_seqlens_q, seqlen_k, state_slot, slot_mapping, block_table);
 *     an out-of-range value skips the access and, when dev_status is non-NULL,
 *     writes INKATTN_ERR_DEVICE_BOUNDS there.  Bounded device waits that run out
 *     write INKATTN_ERR_DEVICE_TIMEOUT.  The first error written wins; the caller
 *     zeroes *dev_status before the call and reads it after synchronising.
 *   - head_dim must be 128 and block_size 64, else INKATTN_ERR_UNSUPPORTED.
 *   - Bounded device waits give up after 1 s.  For tests of that failure path only, two
 *     environment variables are read once per process: INKATTN_TEST_WAIT_LIMIT_US
 *     (100 .. 10000000: a shorter limit) and INKATTN_TEST_WITHHOLD_ARRIVAL=1 (the
 *     attention kernels' softmax withholds its first arrival before P V, and the qkvr
 *     kernel one release of an accumulator, so that the MMA warp's wait runs out).  Leave
 *     both unset in normal use.
 */
#ifndef INKATTN_H
#define INKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define INKATTN_ABI_VERSION 2

/* The library is built with hidden visibility; only these entry points are exported. */
#if defined(__GNUC__)
#define INKATTN_API __attribute__((visibility("default")))
#else
#define INKATTN_API
#endif

typedef uint16_t inkattn_bf16;

/* Element type of the attention output. */
#define INKATTN_DTYPE_BF16 0
#define INKATTN_DTYPE_F32 1

/* Element type of the paged KV cache (kv_dtype).
 * INKATTN_KV_BF16: k_cache and v_cache hold bf16 values.
 * INKATTN_KV_E4M3: they hold OCP FP8 E4M3 codes (1 byte per value, same
 *   [num_blocks][Hkv][64][128] layout), and k_scale / v_scale hold one fp32 scale per
 *   row ([num_blocks][Hkv][64]): the row's values are code * scale.  The prologue writes
 *   scale = 2^k, k the smallest integer >= -24 with 448 * 2^k >= the row's largest
 *   magnitude (1 for an all-zero row), and each code as the nearest E4M3 value to
 *   x / 2^k (ties to even), where x is the bf16 value the bf16 cache would hold; the
 *   dequantised value is exact.  [SG §Relative Attention と FA4 経路: MXFP8 on the FA4
 *   path; VJ §フューチャーロードマップ and VV: FP8 for the global-attention layers.]
 *   The decode reads such a cache, and inkattn_prefill_e4m3 (inkattn_prefill returns
 *   INKATTN_ERR_UNSUPPORTED for it).
 *   The decode expands each row to f16 (code * scale, exact for the prologue's scales
 *   down to 2^-15; below, values under 2^-24 flush) and requires every scale to lie in
 *   [2^-24, 2^7], which the prologue's scales do for rows whose magnitudes stay below
 *   57344; a scale outside that range is flagged as INKATTN_ERR_DEVICE_BOUNDS and its
 *   row read as zeros. */
#define INKATTN_KV_BF16 0
#define INKATTN_KV_E4M3 1

typedef enum inkattn_status {
    INKATTN_OK = 0,
    INKATTN_ERR_INVALID_ARG = 1,     /* bad pointer, size, or combination of sizes     */
    INKATTN_ERR_UNSUPPORTED = 2,     /* valid but not implemented (head_dim, block ...) */
    INKATTN_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed            */
    INKATTN_ERR_DEVICE_TIMEOUT = 4,  /* written to *dev_status by a bounded device wait */
    INKATTN_ERR_DEVICE_BOUNDS = 5    /* written to *dev_status by a device bounds check */
} inkattn_status;

/* Short English text for a status code (static storage, never NULL). */
INKATTN_API const char *inkattn_status_string(inkattn_status s);

/* INKATTN_ABI_VERSION of the built library. */
INKATTN_API int inkattn_abi_version(void);

/* ------------------------------------------------------------------------------
 * The attention prologue [SG §ShortConv 最適化：融合、グラフキャプチャ、シャーディング]:
 * K/V ShortConv + conv-state carry + Q/K RMSNorm + paged KV write, one kernel.
 *
 * Let C = Hkv*128, g = Hq/Hkv.  Sequence b owns new tokens
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]).  For each sequence and channel c, with xs =
 * the 3 carried rows (oldest first) followed by the new rows of k (resp. v):
 *   kc[t][c] = bf16( sum_{k=0..3} conv_w_k[c][k] * xs[t+k][c] )     (fp32 accumulate,
 *   vc[t][c] = bf16( same with v and conv_w_v )                      taps in order 0..3)
 * [SG §ShortConv：4カ所に現れる短距離因果畳み込み: W = 4, current token plus the 3 previous
 * positions of the same channel; conv_w[c][3] weighs the current token].
 * The state slot then holds the last 3 rows of xs [VV §Quản lý bộ nhớ đệm sconv].
 * Per (token, head) over the 128 values, in fp32, rounded to bf16:
 *   q_out = q  / sqrt(mean(q^2)  + eps) * q_norm_w
 *   kn    = kc / sqrt(mean(kc^2) + eps) * k_norm_w
 * [SG §Inkling のモデルアーキテクチャ: ShortConv on K and V before the Q/K normalisation].
 * Then, with slot = slot_mapping[t]: k_cache[slot/64][hk][slot%64][:] = kn,
 * v_cache[...] = vc (with kv_dtype = INKATTN_KV_E4M3: their E4M3 codes, and the row
 * scales to k_scale / v_scale[slot/64][hk][slot%64]).  V is not normalised and Q is not
 * convolved.
 * ------------------------------------------------------------------------------ */
typedef struct inkattn_prologue_params {
    size_t struct_size;        /* = sizeof(inkattn_prologue_params)                      */
    int32_t B;                 /* sequences in the batch, >= 1                           */
    int32_t N_tok;             /* new tokens = cu_seqlens_q[B], >= 0                     */
    int32_t max_seqlen_q;      /* >= every q_len[b]; sizes the grid                      */
    int32_t Hq, Hkv;           /* query / KV heads, Hq % Hkv == 0                        */
    int32_t head_dim;          /* 128                                                    */
    int32_t block_size;        /* paged-cache block, 64                                  */
    int32_t num_blocks;        /* cache capacity in blocks (bounds check)                */
    int32_t num_state_slots;   /* conv-state capacity in slots (bounds check)            */
    float eps;                 /* RMSNorm epsilon, >= 0                                  */
    const inkattn_bf16 *q;     /* [N_tok][Hq][128]                                       */
    const inkattn_bf16 *k;     /* [N_tok][C]  (K projection output, before the conv)     */
    const inkattn_bf16 *v;     /* [N_tok][C]                                             */
    const float *conv_w_k;     /* [C][4]                                                 */
    const float *conv_w_v;     /* [C][4]                                                 */
    const float *q_norm_w;     /* [128], shared by all query heads                       */
    const float *k_norm_w;     /* [128], shared by all KV heads                          */
    const int32_t *cu_seqlens_q;   /* [B+1], non-decreasing, cu[0] = 0                   */
    const int32_t *state_slot;     /* [B], distinct values in [0, num_state_slots)       */
    const int32_t *slot_mapping;   /* [N_tok], distinct values in [0, num_blocks*64)     */
    inkattn_bf16 *conv_state_k;    /* [num_state_slots][3][C], read then overwritten     */
    inkattn_bf16 *conv_state_v;    /* [num_state_slots][3][C]                            */
    inkattn_bf16 *q_out;           /* [N_tok][Hq][128]                                   */
    void *k_cache;                 /* [num_blocks][Hkv][64][128], bf16 or E4M3 (kv_dtype) */
    void *v_cache;                 /* [num_blocks][Hkv][64][128]                         */
    int32_t kv_dtype;              /* INKATTN_KV_BF16 (0) or INKATTN_KV_E4M3 (1)          */
    float *k_scale;                /* E4M3 only: [num_blocks][Hkv][64] row scales, 16-byte */
    float *v_scale;                /* aligned; written for the mapped slots (else NULL)   */
    int32_t *dev_status;           /* nullable, see the conventions above                */
} inkattn_prologue_params;

/* Runs the prologue.  Buffers may not alias except as stated (conv_state_* in/out). */
INKATTN_API inkattn_status inkattn_prologue(const inkattn_prologue_params *p, void *stream);

/* ------------------------------------------------------------------------------
 * Relative-position-bias GQA attention over the paged cache
 * [SG §相対位置バイアス付き Attention; VJ §TML Inkling モデルアーキテクチャ
 *  "Hybrid Attention", "Relative Attention"; VV §FA4 với sheared bias].
 *
 * Sequence b has q_len = cu_seqlens_q[b+1]-cu_seqlens_q[b] new tokens at positions
 * i = seqlen_k[b]-q_len+t; key j (0 <= j < seqlen_k[b]) sits at position j in block
 * block_table[b][j/64], offset j%64, head kv = h / (Hq/Hkv).  For query head h:
 *   s_ij = lambda_b * ( softmax_scale * q_i.k_j + bias_hij ),
 *   bias_hij = sum_{e<d_r} r[i][h][e] * P[h][i-j][e]  if 0 <= i-j < rel_extent, else 0,
 * visible keys: j <= i, and i-j < window when window > 0 (sliding-window layer),
 *   lambda_b = max(1, ln(seqlen_k[b]) / ln(log_scale_base)) when log_scale_base > 1
 *             (full layers' length-dependent logit scaling), else 1,
 *   out_i = sum_j softmax_j(s_ij) v_j,  lse_i = ln sum_j exp(s_ij)  (natural log).
 * softmax_scale <= 0 selects 1/sqrt(128).
 *
 * q, k_cache and v_cache are read by TMA through tensor maps and must be device memory of
 * the current device (cudaMalloc or a memory pool of that device); host memory, managed
 * memory and another GPU's memory are rejected with INKATTN_ERR_INVALID_ARG.  The prefill
 * kernel multicasts each K/V tile to the two CTAs of a head pair inside one cluster: the
 * tensor maps cover this GPU's memory alone.
 * The bias enters the logits as 16-bit fixed point in units of softmax_scale * q.k, so the
 * absolute error of a bias value is at most half a step.  Prefill takes one step per chunk
 * of 128 distances, max_a |r_a| * max_delta |P_h[delta]| / 32000 over the chunk's rows and
 * distances (by Cauchy-Schwarz no value of the chunk exceeds 32000 steps); decode takes one
 * per query row and table round, the largest magnitude in it / 32000.  The
 * decode tables are computed with fp16 operands: P's entries must lie inside fp16's range
 * (|P| < 65504), else the call reports INKATTN_ERR_DEVICE_BOUNDS.
 * ------------------------------------------------------------------------------ */
typedef struct inkattn_attn_params {
    size_t struct_size;        /* = sizeof(inkattn_attn_params)                          */
    int32_t B;                 /* sequences, >= 1                                        */
    int32_t N_tok;             /* query rows = cu_seqlens_q[B]                           */
    int32_t max_seqlen_q;      /* >= every q_len[b]                                      */
    int32_t max_seqlen_k;      /* >= every seqlen_k[b]                                   */
    int32_t Hq, Hkv;           /* Hq % Hkv == 0                                          */
    int32_t head_dim;          /* 128                                                    */
    int32_t block_size;        /* 64                                                     */
    int32_t num_blocks;        /* cache capacity in blocks (bounds check)                */
    int32_t max_blocks_per_seq;/* row length of block_table                              */
    int32_t d_r;               /* relative feature size: 32                              */
    int32_t rel_extent;        /* >= 0; 0 disables the bias                              */
    int32_t window;            /* 0 = full attention, else the sliding window (keys)     */
    int32_t out_dtype;         /* INKATTN_DTYPE_BF16 (0) or INKATTN_DTYPE_F32 (1) for out */
    float softmax_scale;       /* <= 0 -> 1/sqrt(128)                                    */
    float log_scale_base;      /* <= 1 -> no length-dependent scaling (8192 on full layers) */
    const inkattn_bf16 *q;     /* [N_tok][Hq][128], the normalised queries               */
    const inkattn_bf16 *r;     /* [N_tok][Hq][d_r], 16-byte aligned (nullable iff rel_extent == 0) */
    const float *P;            /* [Hq][rel_extent][d_r]: per query head, per distance,   */
                               /* the d_r projection weights; 16-byte aligned (nullable  */
                               /* iff rel_extent == 0)                                   */
    const void *k_cache;           /* [num_blocks][Hkv][64][128], bf16 or E4M3 (kv_dtype) */
    const void *v_cache;           /* [num_blocks][Hkv][64][128]                         */
    int32_t kv_dtype;              /* INKATTN_KV_BF16 (0) or INKATTN_KV_E4M3 (1)          */
    const float *k_scale;          /* E4M3 only: [num_blocks][Hkv][64] row scales, 16-byte */
    const float *v_scale;          /* aligned (else NULL)                                */
    const int32_t *cu_seqlens_q;   /* [B+1]                                              */
    const int32_t *seqlen_k;       /* [B], q_len[b] <= seqlen_k[b] <= max_seqlen_k       */
    const int32_t *block_table;    /* [B][max_blocks_per_seq]                            */
    void *out;                     /* [N_tok][Hq][128], bf16 or fp32 per out_dtype; the   */
                                   /* bf16 form is the fp32 result rounded once (RNE)     */
    float *lse;                    /* nullable, [N_tok][Hq]                              */
    int32_t *dev_status;           /* nullable                                           */
} inkattn_attn_params;

/* Prefill (any q_len) over a bf16 cache: writes out (and lse).  An E4M3 cache returns
 * INKATTN_ERR_UNSUPPORTED here; it takes inkattn_prefill_e4m3. */
INKATTN_API inkattn_status inkattn_prefill(const inkattn_attn_params *p, void *stream);

/* Prefill over an E4M3 cache (kv_dtype = INKATTN_KV_E4M3) [SG §Relative Attention と FA4
 * 経路; VJ §フューチャーロードマップ: FP8 for the global-attention layers].  The blocks the
 * batch reads, block_table[b][0 .. ceil(seqlen_k[b]/64)), are first expanded, code * scale
 * (exact in bf16), into a bf16 copy in the workspace with a block table of its own; then the
 * bf16 prefill runs on the copy, so the result is the bf16 prefill's over the dequantised
 * cache.  A row inside a sequence whose scale lies outside [2^-24, 2^7] (or a block id out
 * of range) is flagged INKATTN_ERR_DEVICE_BOUNDS and read as zeros, as in the decode.
 * workspace: device memory of the current device, 256-byte aligned, at least
 * inkattn_prefill_workspace_bytes(p) bytes (B * max_blocks_per_seq blocks of bf16 K and V
 * plus their table), else INKATTN_ERR_INVALID_ARG; a bf16 cache is INKATTN_ERR_INVALID_ARG
 * (it takes inkattn_prefill).  Two launches, chained like the others. */
INKATTN_API size_t inkattn_prefill_workspace_bytes(const inkattn_attn_params *p);   /* 0 if invalid or bf16 */
INKATTN_API inkattn_status inkattn_prefill_e4m3(const inkattn_attn_params *p, void *workspace,
                                                size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------------
 * Split-KV decode [VJ §低レイテンシコレクティブとカーネル "FA4 Kernel"; VV §FA4 với
 * sheared bias: num_splits is picked per configuration from batch size, TP size and
 * KV length].  Decode shapes: max_seqlen_q <= 16 and max_seqlen_q*(Hq/Hkv) <= 128
 * (e.g. 9 MTP-verify tokens x 8 query heads per KV head).  Same math as prefill.
 * ------------------------------------------------------------------------------ */

/* The split count the library would pick for these params on a GPU with num_sms
 * SMs (tensor-parallel size 1).  Host only; returns >= 1, or 0 for invalid params. */
INKATTN_API int inkattn_decode_num_splits(const inkattn_attn_params *p, int num_sms);

/* Bytes of workspace inkattn_decode needs for num_splits (0 = the heuristic on the
 * current device): N_tok*Hq*S*(128+1)*4 rounded up to 256, or 0 when S resolves to 1. */
INKATTN_API size_t inkattn_decode_workspace_bytes(const inkattn_attn_params *p, int num_splits);

/* Decode pass.  num_splits: 0 = heuristic, else 1..64.  The keys a sequence attends to
 * are divided into num_splits contiguous parts of near-equal size, except that with
 * num_splits = 2 and rel_extent > 0 the cut is at the start of the band (the keys
 * within rel_extent of the first query, moved down so that the part before it holds
 * whole 128-key tiles): the
 * streaming part and the band part then run in separate CTAs, the streaming ones
 * scheduled first.  With one split the result goes straight to out/lse; otherwise each
 * split's own softmax-normalised partial output and its lse go to the workspace, and
 * inkattn_combine must follow on the same stream with the same num_splits.
 * workspace: device memory of at least inkattn_decode_workspace_bytes bytes,
 * 256-byte aligned, owned by the caller, not read by the host. */
INKATTN_API inkattn_status inkattn_decode(const inkattn_attn_params *p, int num_splits,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Merges the per-split partials: lse = ln sum_s exp(lse_s), out = sum_s
 * exp(lse_s - lse) out_s.  A no-op when num_splits resolves to 1. */
INKATTN_API inkattn_status inkattn_combine(const inkattn_attn_params *p, int num_splits,
                               const void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------------
 * Decode without a caller-provided workspace.  The pages have no counterpart: this
 * is a library convenience.
 *
 * For callers that cannot allocate device memory where they decode: plugin hosts that
 * own all device memory and pass only inputs and outputs, and serving loops that must not
 * allocate on the hot path (an allocation can synchronise the device).  The call itself
 * still makes CUDA runtime calls (device and pointer queries, tensor-map encoding) and
 * launches kernels.
 *
 * Same computation and result as inkattn_decode followed by inkattn_combine with the
 * same split count, writing out/lse: with an explicit num_splits the results are
 * bit-identical to theirs.  The split partials go to a static device buffer of
 * INKATTN_DECODE_NOALLOC_MAX_BYTES inside the library instead of a workspace; the call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - num_splits = 0 takes the heuristic's split count and lowers it until the partials
 *     fit the buffer (down to 1, which needs none).
 *   - An explicit num_splits whose partials exceed the buffer, i.e. whose
 *     inkattn_decode_workspace_bytes(p, S) is above INKATTN_DECODE_NOALLOC_MAX_BYTES, is
 *     rejected with INKATTN_ERR_INVALID_ARG.
 *   - The buffer's device address belongs to a CUDA context; it is looked up with the
 *     caller's context current and cached per context (a new context, e.g. after
 *     cudaDeviceReset, looks it up again).  The first call in a context may load the
 *     library's device code: make it before any stream capture.
 *   - Every call on a device shares the one buffer and it keeps the last call's
 *     contents.  Each call writes every partial it reads, so nothing needs clearing,
 *     but calls whose GPU work overlaps (on different streams, or from several host
 *     threads without ordering) race on the buffer: serialise them.
 *   - Each GPU on which this part of the library is loaded holds the buffer until the
 *     process exits.
 * ------------------------------------------------------------------------------ */
#define INKATTN_DECODE_NOALLOC_MAX_BYTES (64u << 20)

INKATTN_API inkattn_status inkattn_decode_noalloc(const inkattn_attn_params *p, int num_splits,
                                                  void *stream);

/* ------------------------------------------------------------------------------
 * Attention-output ShortConv with the residual add and the RMSNorm, one kernel
 * [SG §ShortConv：4カ所に現れる短距離因果畳み込み (the third ShortConv position, after the
 * attention output); SG §ShortConv 最適化：融合、グラフキャプチャ、シャーディング (it sits on the
 * residual stream; in decode the residual add and the RMSNorm fold into the same
 * kernel); VV §TP sharding nhận biết sconv (order: o_proj output -> sconv -> residual
 * connection -> RMSNorm)].  On one GPU there is no all-reduce in front of it: the input is
 * the o_proj output itself.
 *
 * For each sequence b and hidden channel c, with xs = the 3 carried rows (oldest first)
 * followed by the new rows of y:
 *   conv[t][c] = bf16( sum_{k=0..3} conv_w[c][k] * xs[t+k][c] )   (correctly rounded)
 *   h[t][c]    = bf16( residual[t][c] + conv[t][c] )               (correctly rounded)
 *   out[t][c]  = bf16( h[t][c] / sqrt(mean_c'(h[t][c']^2) + eps) * norm_w[c] )
 * the mean over all D channels of the token.  The state slot then holds the last 3 rows
 * of xs.  conv and h are bit-exact; out is within 1 bf16 ulp of the fp64 value (its sum
 * of squares is taken in fp32).  An empty sequence keeps its state.
 * ------------------------------------------------------------------------------ */
typedef struct inkattn_output_conv_params {
    size_t struct_size;        /* = sizeof(inkattn_output_conv_params)                   */
    int32_t B;                 /* sequences, 1 .. 65535                                  */
    int32_t N_tok;             /* new tokens = cu_seqlens_q[B], >= 0                     */
    int32_t max_seqlen_q;      /* >= every q_len[b]; sizes the grid                      */
    int32_t D;                 /* hidden width: a multiple of 8, 8 .. 32768              */
    int32_t num_state_slots;   /* conv-state capacity in slots (bounds check)            */
    float eps;                 /* RMSNorm epsilon, >= 0                                  */
    const inkattn_bf16 *y;     /* [N_tok][D], the o_proj output                          */
    const float *conv_w;       /* [D][4], w[c][3] weighs the current token               */
    const float *norm_w;       /* [D]                                                    */
    const int32_t *cu_seqlens_q;   /* [B+1], non-decreasing, cu[0] = 0                   */
    const int32_t *state_slot;     /* [B], distinct values in [0, num_state_slots)       */
    inkattn_bf16 *conv_state;      /* [num_state_slots][3][D], read then overwritten     */
    const inkattn_bf16 *residual;  /* [N_tok][D], the residual stream before the add     */
    inkattn_bf16 *h_out;           /* [N_tok][D], the new residual stream; may equal residual */
    inkattn_bf16 *out;             /* [N_tok][D], its RMSNorm                            */
    int32_t *dev_status;           /* nullable, see the conventions above                */
} inkattn_output_conv_params;

/* Runs the attention-output conv.  y, conv_w, norm_w, conv_state, residual, h_out and out
 * must be 16-byte aligned.  out and h_out may not overlap y, and out may not overlap
 * residual or h_out (INKATTN_ERR_INVALID_ARG); h_out == residual (in place) is allowed,
 * a partial overlap of the two is not.  conv_state must not overlap the other arrays. */
INKATTN_API inkattn_status inkattn_output_conv(const inkattn_output_conv_params *p, void *stream);

/* ------------------------------------------------------------------------------
 * The qkvr projections with the attention prologue fused into their epilogue: one pass
 * from the hidden states to what inkattn_prologue writes, plus r
 * [VJ §TML Inkling モデルアーキテクチャ and VV, the MoE item of the architecture list: the
 * q, k, v and r projections ("qkvr linears") are one bf16 linear layer in front of the
 * attention; SG §ShortConv 最適化：融合、グラフキャプチャ、シャーディング: the prologue's work
 * fused so that nothing intermediate is written back].
 *
 * With F = Hq*128 + 2*Hkv*128 + Hq*d_r output features and the rows of w ordered
 * [q heads | k | v | r heads] (nn.Linear layout, [F][d_model]):
 *   y[t][o] = bf16( sum_k x[t][k] * w[o][k] )       (fp32 accumulation on the tensor cores)
 *   q = y[:, 0:Hq*128] as [N_tok][Hq][128],  k = the next Hkv*128 features,
 *   v = the next Hkv*128,  r = the last Hq*d_r as [N_tok][Hq][d_r] (written to r_out).
 * Then everything inkattn_prologue does, on q, k and v, with two differences: the conv
 * state is read from conv_state_*_in and the new state written to conv_state_*_out, and
 * a sequence with no new tokens copies its state from in to out.  The projections are
 * rounded once from the fp32 sum; against the exactly rounded sum that can differ by one
 * bf16 ulp where the sum lies within the fp32 accumulation error of a rounding midpoint.
 *
 * Work is cut into tiles of INKATTN_QKVR_TILE_TOKENS (125) new tokens of one sequence plus
 * the 3 before them (the conv's history, recomputed rather than exchanged), so a tile
 * never waits on another.  The new conv state is written by the tile holding a sequence's
 * last tokens while the sequence's first tile reads the old one; in and out may therefore
 * be the same array only when max_seqlen_q <= INKATTN_QKVR_TILE_TOKENS (every sequence in
 * one tile), else INKATTN_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------------ */
#define INKATTN_QKVR_TILE_TOKENS 125
#define INKATTN_QKVR_MAX_SEQS 1024

typedef struct inkattn_qkvr_params {
    size_t struct_size;        /* = sizeof(inkattn_qkvr_params)                          */
    int32_t B;                 /* sequences, 1 .. INKATTN_QKVR_MAX_SEQS                  */
    int32_t N_tok;             /* new tokens = cu_seqlens_q[B], >= 0                     */
    int32_t max_seqlen_q;      /* >= every q_len[b]                                      */
    int32_t Hq, Hkv;           /* query / KV heads, Hq % Hkv == 0                        */
    int32_t head_dim;          /* 128                                                    */
    int32_t d_r;               /* relative features per query head; Hq*d_r % 8 == 0      */
    int32_t d_model;           /* hidden width: a multiple of 8, >= 8                    */
    int32_t block_size;        /* paged-cache block, 64                                  */
    int32_t num_blocks;        /* cache capacity in blocks (bounds check)                */
    int32_t num_state_slots;   /* conv-state capacity in slots (bounds check)            */
    float eps;                 /* RMSNorm epsilon, >= 0                                  */
    const inkattn_bf16 *x;     /* [N_tok][d_model] hidden states; device memory of this GPU */
    const inkattn_bf16 *w;     /* [F][d_model]; device memory of this GPU                */
    const float *conv_w_k;     /* [C][4], C = Hkv*128; w[c][3] weighs the current token  */
    const float *conv_w_v;     /* [C][4]                                                 */
    const float *q_norm_w;     /* [128]                                                  */
    const float *k_norm_w;     /* [128]                                                  */
    const int32_t *cu_seqlens_q;   /* [B+1], non-decreasing, cu[0] = 0                   */
    const int32_t *state_slot;     /* [B], distinct values in [0, num_state_slots)       */
    const int32_t *slot_mapping;   /* [N_tok], distinct values in [0, num_blocks*64)     */
    const inkattn_bf16 *conv_state_k_in;  /* [num_state_slots][3][C]                     */
    const inkattn_bf16 *conv_state_v_in;  /* [num_state_slots][3][C]                     */
    inkattn_bf16 *conv_state_k_out;       /* [num_state_slots][3][C], rows of the        */
    inkattn_bf16 *conv_state_v_out;       /* sequences' slots written                    */
    inkattn_bf16 *q_out;           /* [N_tok][Hq][128], normalised                       */
    inkattn_bf16 *r_out;           /* [N_tok][Hq][d_r]                                   */
    inkattn_bf16 *y_out;           /* nullable: [N_tok][F], every projection as rounded  */
    void *k_cache;                 /* as in inkattn_prologue_params                      */
    void *v_cache;
    int32_t kv_dtype;              /* INKATTN_KV_BF16 or INKATTN_KV_E4M3                  */
    float *k_scale;                /* E4M3 only (else NULL), as in inkattn_prologue_params */
    float *v_scale;
    int32_t *dev_status;           /* nullable, see the conventions above                */
} inkattn_qkvr_params;

/* Runs the fused projections and prologue.  x and w are read by TMA (device memory of the
 * current device, 16-byte aligned; anything else is INKATTN_ERR_INVALID_ARG); q_out,
 * r_out, y_out, the caches and the states must be 16-byte aligned.  With y_out non-NULL the
 * projections (before conv and norm) are written there too, at the cost of their bytes.  No output may overlap an
 * input except conv_state_*_out == conv_state_*_in under the rule above. */
INKATTN_API inkattn_status inkattn_qkvr_prologue(const inkattn_qkvr_params *p, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* INKATTN_H */
