/*
 * oracle.c -- plain fp64 CPU oracle for the Inkling attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py may load this library.  The CUDA product path
 * never calls it, shares no code with it, and fails loudly when its own
 * extension is missing.
 *
 * Sources (cited by page title and section heading):
 *   [SG]  "SGLang と Miles が Inkling を初日からサポート：975Bのマルチモーダル最先端モデルが公開"
 *         (winzheng.jp review page)
 *   [VJ]  "vLLM TML Inkling サポート" (agentlenshq.com, Japanese)
 *   [VV]  "vLLM hỗ trợ TML Inkling ngay khi ra mắt với hiệu năng tối ưu" (gpuhub.net)
 *
 * What is computed, step by step (no blocking, fusion or reordering beyond
 * the definitions):
 *   1. ShortConv on the K and V streams [SG §ShortConv：4カ所に現れる短距離因果畳み込み;
 *      VJ §TML Inkling モデルアーキテクチャ "Short Convolution (Sconv)"]:
 *      per channel c, y[t] = sum_{k=0..3} w[c][k] * xs[t+k], where xs is the
 *      3 carried rows followed by the new rows of the sequence; w[c][3] weighs
 *      the current token and w[c][0] the token three back.  No bias, no
 *      activation.  The result is rounded to bf16 (round to nearest even).
 *   2. Conv-state carry [VV §"Quản lý bộ nhớ đệm sconv"]: the state holds the
 *      pre-conv inputs of the last W-1 = 3 tokens; the new state is the last 3
 *      rows of xs.
 *   3. Q/K RMSNorm [SG §ShortConv 最適化：融合、グラフキャプチャ、シャーディング,
 *      §Inkling のモデルアーキテクチャ]: per (token, head) over the 128 values,
 *      y = x / sqrt(mean(x^2) + eps) * g, rounded to bf16.  K is normalised
 *      after its conv (from the bf16-rounded conv output); V is not normalised;
 *      Q is not convolved.
 *   4. Paged KV write [SG §ShortConv 最適化]: k_cache/v_cache[blk][kv_head][off][:]
 *      with blk = slot / block_size, off = slot % block_size.
 *   5. Attention with relative-position bias [SG §相対位置バイアス付き Attention;
 *      VJ §TML Inkling モデルアーキテクチャ "Relative Attention", "Hybrid Attention"]:
 *      s_j = lambda * ( scale * q.k_j + [0 <= i-j < rel_extent] * sum_k r[i][h][k] P_h[k][i-j] )
 *      over keys j <= i (and i-j < window for sliding-window layers),
 *      o = softmax(s) . V, lse = log sum_j exp(s_j).
 *      lambda = max(1, ln T / ln base) on full layers that enable it (T = the
 *      sequence's key length), else 1; it scales the whole logit.
 *   6. Attention-output ShortConv on the residual stream [SG §ShortConv：4カ所に現れる
 *      短距離因果畳み込み (the third of the four positions: after the attention output);
 *      SG §ShortConv 最適化 (it sits on the residual stream, and in decode RMSNorm and the
 *      residual add are folded into the same kernel); VV §TP sharding nhận biết sconv
 *      (the unfused order: o_proj output -> sconv -> residual connection -> RMSNorm)]:
 *      per hidden channel c of the o_proj output y, the same W = 4 causal conv with its
 *      own carried state as in step 1, rounded to bf16; then
 *      h = bf16(residual + conv) (the new residual stream, the sum rounded once), and
 *      out = bf16(h / sqrt(mean_c(h^2) + eps) * g) over the D hidden channels of the
 *      token, from the bf16 h.
 *   7. FP8 KV cache [SG §Relative Attention と FA4 経路 (the FA4 path runs in MXFP8);
 *      VJ §フューチャーロードマップ and VV (FP8 for global attention, to relieve compute and
 *      the KV cache)]: a cache row (one token, one KV head, 128 values, after step 3's
 *      rounding to bf16) is stored as E4M3 codes with one power-of-two scale 2^k, k the
 *      smallest integer >= -24 with 448 * 2^k >= max|x| (k = 0 for an all-zero row); each
 *      code is x / 2^k rounded to the nearest E4M3 value, ties to even.  Reading the row
 *      back gives code * 2^k exactly; attention (step 5) runs on those values.
 *   8. The qkvr projections in front of the prologue [VJ §TML Inkling モデルアーキテクチャ and
 *      VV §"MoE" (the q, k, v and r linears are BF16 layers); SG §ShortConv：4カ所に現れる
 *      短距離因果畳み込み (the K and V ShortConvs follow the K and V projections)]: from the
 *      hidden states x [N][d_model] and one weight matrix w [Hq*d + 2*Hkv*d + Hq*d_r][d_model]
 *      (a row per output feature), y = x . w^T, each value rounded once to bf16; its columns
 *      are q, k, v and r in that order, and q, k, v then go through steps 1-4.  (The matrix
 *      product itself is library arithmetic on the Python side; this file only rounds.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_INDEX 2
#define ORACLE_ERR_NOMEM 3

static double bf16_bits_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to bf16 (1 implicit + 7 stored significand bits), ties to
 * even, directly from the fp64 value (no intermediate fp32 rounding). */
uint16_t oracle_f64_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(ax, &e);          /* ax in [2^(e-1), 2^e) */
    int ulp_exp = e - 8;          /* 8 significant bits */
    if (ulp_exp < -133) ulp_exp = -133; /* bf16 subnormal spacing */
    double q = ldexp(ax, -ulp_exp);      /* exact */
    double qr = nearbyint(q);            /* default mode: nearest, ties to even */
    double y = ldexp(qr, ulp_exp);
    if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)y;                  /* exact: y has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* lambda = max(1, ln T / ln base) for base > 1, else 1. */
double oracle_log_scale(double T, double base) {
    if (!(base > 1.0) || !(T > 0.0)) return 1.0;
    double l = log(T) / log(base);
    return l > 1.0 ? l : 1.0;
}

/*
 * The attention prologue: steps 1-4 above.
 *
 * Layouts (row-major, bf16 passed as raw uint16 bit patterns):
 *   q [N][Hq][d], k, v [N][Hkv*d]; conv_w_k, conv_w_v [C][4] with C = Hkv*d;
 *   q_norm_w, k_norm_w [d]; conv_state_k/v [num_state_slots][3][C] (in/out);
 *   slot_mapping [N]; k_cache, v_cache [num_blocks][Hkv][block_size][d] (in/out);
 *   q_out [N][Hq][d].
 * Optional outputs (NULL to skip): kc_f64 / vc_f64 [N][C] = the conv sums
 * before rounding; kc_bf16 / vc_bf16 [N][C] = the rounded conv outputs.
 * Returns ORACLE_ERR_INDEX (and writes nothing further) when an index is out
 * of range.
 */
int oracle_prologue(int B, const int32_t *cu_seqlens_q, int Hq, int Hkv, int d,
                    const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const float *conv_w_k, const float *conv_w_v,
                    const float *q_norm_w, const float *k_norm_w, double eps,
                    const int32_t *state_slot, int num_state_slots,
                    uint16_t *conv_state_k, uint16_t *conv_state_v,
                    const int32_t *slot_mapping, int block_size, int num_blocks,
                    uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache,
                    double *kc_f64, double *vc_f64, uint16_t *kc_bf16, uint16_t *vc_bf16)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (Hq % Hkv) != 0 || block_size <= 0)
        return ORACLE_ERR_ARG;
    const int C = Hkv * d;
    const int N = cu_seqlens_q[B];
    for (int b = 0; b < B; ++b) {
        if (cu_seqlens_q[b] > cu_seqlens_q[b + 1] || cu_seqlens_q[b] < 0) return ORACLE_ERR_ARG;
        if (state_slot[b] < 0 || state_slot[b] >= num_state_slots) return ORACLE_ERR_INDEX;
    }
    for (int t = 0; t < N; ++t) {
        if (slot_mapping[t] < 0 || slot_mapping[t] / block_size >= num_blocks) return ORACLE_ERR_INDEX;
    }

    uint16_t *kc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(N > 0 ? N : 1) * C);
    uint16_t *vc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(N > 0 ? N : 1) * C);
    if (!kc || !vc) { free(kc); free(vc); return ORACLE_ERR_NOMEM; }

    /* Steps 1 and 2: conv and state carry, one sequence and one channel at a time. */
    for (int b = 0; b < B; ++b) {
        const int start = cu_seqlens_q[b];
        const int n = cu_seqlens_q[b + 1] - start;
        const size_t slot = (size_t)state_slot[b];
        for (int stream = 0; stream < 2; ++stream) {
            const uint16_t *x = stream == 0 ? k : v;
            const float *w = stream == 0 ? conv_w_k : conv_w_v;
            uint16_t *state = stream == 0 ? conv_state_k : conv_state_v;
            uint16_t *y16 = stream == 0 ? kc : vc;
            double *y64 = stream == 0 ? kc_f64 : vc_f64;
            for (int c = 0; c < C; ++c) {
                /* xs[0..2] = carried rows (oldest first), xs[3+t] = new row t */
                const int len = 3 + n;
                uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)len);
                if (!xs) { free(kc); free(vc); return ORACLE_ERR_NOMEM; }
                for (int r = 0; r < 3; ++r) xs[r] = state[(slot * 3 + r) * C + c];
                for (int t = 0; t < n; ++t) xs[3 + t] = x[(size_t)(start + t) * C + c];
                for (int t = 0; t < n; ++t) {
                    double acc = 0.0;
                    for (int tap = 0; tap < 4; ++tap)
                        acc += (double)w[c * 4 + tap] * bf16_bits_to_f64(xs[t + tap]);
                    if (y64) y64[(size_t)(start + t) * C + c] = acc;
                    y16[(size_t)(start + t) * C + c] = oracle_f64_to_bf16(acc);
                }
                for (int r = 0; r < 3; ++r) state[(slot * 3 + r) * C + c] = xs[n + r];
                free(xs);
            }
        }
    }
    if (kc_bf16) memcpy(kc_bf16, kc, sizeof(uint16_t) * (size_t)N * C);
    if (vc_bf16) memcpy(vc_bf16, vc, sizeof(uint16_t) * (size_t)N * C);

    /* Step 3: RMSNorm of Q (per token and query head) and of the conv'd K. */
    for (int t = 0; t < N; ++t) {
        for (int h = 0; h < Hq; ++h) {
            const uint16_t *xq = q + ((size_t)t * Hq + h) * d;
            double ss = 0.0;
            for (int i = 0; i < d; ++i) { double a = bf16_bits_to_f64(xq[i]); ss += a * a; }
            const double inv = 1.0 / sqrt(ss / d + eps);
            for (int i = 0; i < d; ++i)
                q_out[((size_t)t * Hq + h) * d + i] =
                    oracle_f64_to_bf16(bf16_bits_to_f64(xq[i]) * inv * (double)q_norm_w[i]);
        }
        /* Step 4 folded per token: normed K and conv'd V go to the token's slot. */
        const int32_t slot = slot_mapping[t];
        const size_t blk = (size_t)(slot / block_size), off = (size_t)(slot % block_size);
        for (int hk = 0; hk < Hkv; ++hk) {
            const uint16_t *xk = kc + (size_t)t * C + (size_t)hk * d;
            double ss = 0.0;
            for (int i = 0; i < d; ++i) { double a = bf16_bits_to_f64(xk[i]); ss += a * a; }
            const double inv = 1.0 / sqrt(ss / d + eps);
            const size_t base = ((blk * Hkv + hk) * block_size + off) * d;
            for (int i = 0; i < d; ++i) {
                k_cache[base + i] = oracle_f64_to_bf16(bf16_bits_to_f64(xk[i]) * inv * (double)k_norm_w[i]);
                v_cache[base + i] = vc[(size_t)t * C + (size_t)hk * d + i];
            }
        }
    }
    free(kc);
    free(vc);
    return ORACLE_OK;
}

/*
 * Attention with the relative-position bias: step 5 above.
 *
 *   q [N][Hq][d] (the normalised queries), r [N][Hq][d_r], P [Hq][rel_extent][d_r] fp32
 *   (P_h[k][delta] stored at P[h][delta][k]: the d_r weights of one distance are contiguous),
 *   k_cache, v_cache [num_blocks][Hkv][block_size][d], block_table [B][max_blocks].
 * Sequence b has q_len = cu_seqlens_q[b+1]-cu_seqlens_q[b] new tokens, which
 * sit at positions seqlen_k[b]-q_len+t; key j sits at position j and lives in
 * block block_table[b][j / block_size] at offset j % block_size.
 * window = 0 means full attention; otherwise key j is visible from query
 * position i iff 0 <= i-j < window.  softmax_scale <= 0 means 1/sqrt(d).
 * log_scale_base <= 1 disables the length-dependent logit scaling.
 *
 * rows: NULL computes every token row; otherwise the n_rows token indices
 * listed, and out/lse are compact: out [n_rows][Hq][d], lse [n_rows][Hq].
 * Rows are independent; OpenMP spreads (row, head) pairs over n_threads
 * threads (0 = the OpenMP default).
 */
int oracle_attention(int B, const int32_t *cu_seqlens_q, const int32_t *seqlen_k,
                     int Hq, int Hkv, int d, int d_r, int rel_extent, int window,
                     double softmax_scale, double log_scale_base,
                     const uint16_t *q, const uint16_t *r, const float *P,
                     const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_table, int max_blocks, int block_size, int num_blocks,
                     const int32_t *rows, int n_rows,
                     double *out, double *lse, int n_threads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (Hq % Hkv) != 0 || block_size <= 0 ||
        d_r < 0 || rel_extent < 0 || window < 0)
        return ORACLE_ERR_ARG;
    const int N = cu_seqlens_q[B];
    const int g = Hq / Hkv;
    const double scale = softmax_scale > 0.0 ? softmax_scale : 1.0 / sqrt((double)d);
    const int nr = rows ? n_rows : N;

    /* token -> sequence lookup and index validation */
    int32_t *seq_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    if (!seq_of) return ORACLE_ERR_NOMEM;
    for (int b = 0; b < B; ++b) {
        const int ql = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        if (ql < 0 || seqlen_k[b] < ql) { free(seq_of); return ORACLE_ERR_ARG; }
        const int nblk = (seqlen_k[b] + block_size - 1) / block_size;
        if (nblk > max_blocks) { free(seq_of); return ORACLE_ERR_ARG; }
        for (int i = 0; i < nblk; ++i) {
            const int32_t blk = block_table[(size_t)b * max_blocks + i];
            if (blk < 0 || blk >= num_blocks) { free(seq_of); return ORACLE_ERR_INDEX; }
        }
        for (int t = cu_seqlens_q[b]; t < cu_seqlens_q[b + 1]; ++t) seq_of[t] = b;
    }
    for (int ri = 0; ri < nr; ++ri) {
        const int t = rows ? rows[ri] : ri;
        if (t < 0 || t >= N) { free(seq_of); return ORACLE_ERR_INDEX; }
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *s = NULL;
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        int cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (long long task = 0; task < (long long)nr * Hq; ++task) {
            const int ri = (int)(task / Hq), h = (int)(task % Hq);
            const int t = rows ? rows[ri] : ri;
            const int b = seq_of[t];
            const int q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            const int i = seqlen_k[b] - q_len + (t - cu_seqlens_q[b]);   /* query position */
            const int hk = h / g;
            const double lam = oracle_log_scale((double)seqlen_k[b], log_scale_base);
            int j_lo = 0;
            if (window > 0 && i - window + 1 > 0) j_lo = i - window + 1;
            const int nk = i - j_lo + 1;
            if (nk > cap) { free(s); cap = nk; s = (double *)malloc(sizeof(double) * (size_t)cap); }
            if (!s || !acc) { status = ORACLE_ERR_NOMEM; continue; }
            const uint16_t *qv = q + ((size_t)t * Hq + h) * d;
            const uint16_t *rv = r ? r + ((size_t)t * Hq + h) * d_r : NULL;
            double m = -INFINITY;
            for (int j = j_lo; j <= i; ++j) {
                const size_t blk = (size_t)block_table[(size_t)b * max_blocks + j / block_size];
                const uint16_t *kv = k_cache + ((blk * Hkv + hk) * block_size + (size_t)(j % block_size)) * d;
                double dot = 0.0;
                for (int e = 0; e < d; ++e) dot += bf16_bits_to_f64(qv[e]) * bf16_bits_to_f64(kv[e]);
                double bias = 0.0;
                const int delta = i - j;
                if (delta < rel_extent && rv) {
                    for (int e = 0; e < d_r; ++e)
                        bias += bf16_bits_to_f64(rv[e]) *
                                (double)P[((size_t)h * rel_extent + delta) * d_r + e];
                }
                const double sj = lam * (scale * dot + bias);
                s[j - j_lo] = sj;
                if (sj > m) m = sj;
            }
            double z = 0.0;
            for (int e = 0; e < d; ++e) acc[e] = 0.0;
            for (int j = j_lo; j <= i; ++j) {
                const double p = exp(s[j - j_lo] - m);
                z += p;
                const size_t blk = (size_t)block_table[(size_t)b * max_blocks + j / block_size];
                const uint16_t *vv = v_cache + ((blk * Hkv + hk) * block_size + (size_t)(j % block_size)) * d;
                for (int e = 0; e < d; ++e) acc[e] += p * bf16_bits_to_f64(vv[e]);
            }
            double *o = out + ((size_t)ri * Hq + h) * d;
            for (int e = 0; e < d; ++e) o[e] = acc[e] / z;
            if (lse) lse[(size_t)ri * Hq + h] = m + log(z);
        }
        free(s);
        free(acc);
    }
    free(seq_of);
    return status;
}

/*
 * The attention-output ShortConv with the residual add and the RMSNorm: step 6 above.
 *
 * Layouts (row-major, bf16 as raw uint16 bit patterns):
 *   y, residual, h_out, out [N][D]; conv_w [D][4] (w[c][3] weighs the current token);
 *   norm_w [D]; conv_state [num_state_slots][3][D] (in/out, oldest row first).
 * Optional output (NULL to skip): conv_bf16 [N][D] = the rounded conv outputs.
 * h_out may be the residual array itself (each element is read before it is written).
 * Returns ORACLE_ERR_INDEX (and writes nothing) when a state slot is out of range.
 */
int oracle_output_conv(int B, const int32_t *cu_seqlens_q, int D,
                       const uint16_t *y, const float *conv_w,
                       const int32_t *state_slot, int num_state_slots, uint16_t *conv_state,
                       const uint16_t *residual, const float *norm_w, double eps,
                       uint16_t *h_out, uint16_t *out, uint16_t *conv_bf16)
{
    if (B < 0 || D <= 0) return ORACLE_ERR_ARG;
    const int N = cu_seqlens_q[B];
    for (int b = 0; b < B; ++b) {
        if (cu_seqlens_q[b] > cu_seqlens_q[b + 1] || cu_seqlens_q[b] < 0) return ORACLE_ERR_ARG;
        if (state_slot[b] < 0 || state_slot[b] >= num_state_slots) return ORACLE_ERR_INDEX;
    }
    uint16_t *cv = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(N > 0 ? N : 1) * D);
    uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(3 + (N > 0 ? N : 1)));
    if (!cv || !xs) { free(cv); free(xs); return ORACLE_ERR_NOMEM; }

    /* The conv and the state carry, one sequence and one channel at a time (as step 1). */
    for (int b = 0; b < B; ++b) {
        const int start = cu_seqlens_q[b];
        const int n = cu_seqlens_q[b + 1] - start;
        const size_t slot = (size_t)state_slot[b];
        for (int c = 0; c < D; ++c) {
            for (int r = 0; r < 3; ++r) xs[r] = conv_state[(slot * 3 + r) * D + c];
            for (int t = 0; t < n; ++t) xs[3 + t] = y[(size_t)(start + t) * D + c];
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int tap = 0; tap < 4; ++tap)
                    acc += (double)conv_w[(size_t)c * 4 + tap] * bf16_bits_to_f64(xs[t + tap]);
                cv[(size_t)(start + t) * D + c] = oracle_f64_to_bf16(acc);
            }
            for (int r = 0; r < 3; ++r) conv_state[(slot * 3 + r) * D + c] = xs[n + r];
        }
    }
    if (conv_bf16) memcpy(conv_bf16, cv, sizeof(uint16_t) * (size_t)N * D);

    /* The residual add, then the RMSNorm of each token's new residual row. */
    for (int t = 0; t < N; ++t) {
        double ss = 0.0;
        for (int c = 0; c < D; ++c) {
            const size_t i = (size_t)t * D + c;
            /* the fp64 sum of two bf16 values is exact when their exponents differ by at
             * most 44; beyond that the smaller is far below half a bf16 ulp of the larger,
             * which is then the correctly rounded sum either way */
            const uint16_t h = oracle_f64_to_bf16(bf16_bits_to_f64(residual[i]) + bf16_bits_to_f64(cv[i]));
            h_out[i] = h;
            const double a = bf16_bits_to_f64(h);
            ss += a * a;
        }
        const double inv = 1.0 / sqrt(ss / D + eps);
        for (int c = 0; c < D; ++c) {
            const size_t i = (size_t)t * D + c;
            out[i] = oracle_f64_to_bf16(bf16_bits_to_f64(h_out[i]) * inv * (double)norm_w[c]);
        }
    }
    free(cv);
    free(xs);
    return ORACLE_OK;
}

/*
 * E4M3 (OCP FP8, "E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * subnormals; no infinities; the largest finite magnitude is 448 (S.1111.110) and
 * S.1111.111 is NaN.
 */
double oracle_e4m3_to_f64(uint8_t c) {
    const int sgn = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9)                 /* m/8 * 2^(1-7) */
                            : ldexp(8.0 + (double)m, e - 10);     /* (1 + m/8) * 2^(e-7) */
    return sgn ? -v : v;
}

/* The nearest E4M3 value to x, ties to the even code; magnitudes past 448 saturate to 448. */
uint8_t oracle_f64_to_e4m3(double x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sgn | 0x7E);
    /* candidates are the 127 finite non-negative codes, in increasing order of value */
    int best = 0;
    double best_d = a;                           /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sgn | (uint8_t)best);
}

/*
 * Step 7: quantise `rows` rows of `width` bf16 values (x, row-major) to E4M3 codes with
 * one power-of-two scale per row (scales receive 2^k as fp32).
 */
int oracle_quantize_rows_e4m3(const uint16_t *x, int rows, int width, uint8_t *codes, float *scales) {
    if (rows < 0 || width <= 0) return ORACLE_ERR_ARG;
    for (int r = 0; r < rows; ++r) {
        const uint16_t *xr = x + (size_t)r * width;
        double amax = 0.0;
        for (int i = 0; i < width; ++i) {
            const double a = fabs(bf16_bits_to_f64(xr[i]));
            if (a > amax) amax = a;
        }
        int k = 0;
        if (amax > 0.0) {
            k = -24;
            while (ldexp(448.0, k) < amax) ++k;
        }
        scales[r] = (float)ldexp(1.0, k);
        for (int i = 0; i < width; ++i)
            codes[(size_t)r * width + i] = oracle_f64_to_e4m3(ldexp(bf16_bits_to_f64(xr[i]), -k));
    }
    return ORACLE_OK;
}

/* Round n doubles to bf16 bit patterns (ties to even), as oracle_f64_to_bf16 does one. */
void oracle_round_bf16_array(const double *x, long long n, uint16_t *out) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(x[i]);
}
