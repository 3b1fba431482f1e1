// api.cu -- the extern "C" entry points of libinkattn.so: host-side validation, TMA
// descriptor setup, the decode split heuristic, and the launches.
//
// Nothing here computes on the host: every step of the path runs in the kernels of
// prologue.cu, qkvr.cu, output_conv.cu, prefill_tc.cu and decode.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/inkattn.h"
#include "internal.h"

namespace inkattn {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNsDefault = 1000000000ull;   // 1 s, as the kernels' default

// ---------------------------------------------------------------- device checks

std::atomic<int> g_dev_ok[kMaxDevices];       // 0 unknown, 1 sm_103, 2 other
std::atomic<int> g_dev_sms[kMaxDevices];

inkattn_status check_device(int *sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return INKATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return INKATTN_ERR_UNSUPPORTED;
    int ok = g_dev_ok[dev].load(std::memory_order_acquire);
    if (ok == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return INKATTN_ERR_CUDA;
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        ok = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_ok[dev].store(ok, std::memory_order_release);
    }
    if (sms_out) *sms_out = g_dev_sms[dev].load(std::memory_order_relaxed);
    return ok == 1 ? INKATTN_OK : INKATTN_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- TMA encode

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

// ---------------------------------------------------------------- validation

inkattn_status validate_prologue(const inkattn_prologue_params *p) {
    if (!p || p->struct_size != sizeof(inkattn_prologue_params)) return INKATTN_ERR_INVALID_ARG;
    if (p->B < 1 || p->N_tok < 0 || p->max_seqlen_q < 0 || p->Hq < 1 || p->Hkv < 1 ||
        p->Hq % p->Hkv != 0 || p->num_blocks < 1 || p->num_state_slots < 1 || !(p->eps >= 0.f))
        return INKATTN_ERR_INVALID_ARG;
    if (p->N_tok > 0 && p->max_seqlen_q < 1) return INKATTN_ERR_INVALID_ARG;
    if (p->B > 65535 || p->Hq > 65535) return INKATTN_ERR_INVALID_ARG;   // (query rows of a tile: 32-bit offsets)
    if ((long long)p->num_blocks * 64 > INT_MAX) return INKATTN_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || p->block_size != kBlock) return INKATTN_ERR_UNSUPPORTED;
    const void *ptrs16[] = {p->q, p->k, p->v, p->conv_state_k, p->conv_state_v, p->q_out,
                            p->k_cache, p->v_cache};
    for (const void *ptr : ptrs16)
        if (!ptr || !aligned(ptr, 16)) return INKATTN_ERR_INVALID_ARG;
    const void *ptrs4[] = {p->conv_w_k, p->conv_w_v, p->q_norm_w, p->k_norm_w, p->cu_seqlens_q,
                           p->state_slot, p->slot_mapping};
    for (const void *ptr : ptrs4)
        if (!ptr || !aligned(ptr, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->dev_status && !aligned(p->dev_status, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype != INKATTN_KV_BF16 && p->kv_dtype != INKATTN_KV_E4M3) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype == INKATTN_KV_E4M3 &&
        (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 16) || !aligned(p->v_scale, 16)))
        return INKATTN_ERR_INVALID_ARG;
    return INKATTN_OK;
}

inkattn_status validate_output_conv(const inkattn_output_conv_params *p) {
    if (!p || p->struct_size != sizeof(inkattn_output_conv_params)) return INKATTN_ERR_INVALID_ARG;
    if (p->B < 1 || p->B > 65535 || p->N_tok < 0 || p->max_seqlen_q < 0 || p->num_state_slots < 1 ||
        !(p->eps >= 0.f))
        return INKATTN_ERR_INVALID_ARG;
    if (p->D < 8 || p->D > 32768 || p->D % 8 != 0) return INKATTN_ERR_INVALID_ARG;
    if (p->N_tok > 0 && p->max_seqlen_q < 1) return INKATTN_ERR_INVALID_ARG;
    const void *ptrs16[] = {p->y, p->conv_w, p->norm_w, p->conv_state, p->residual, p->h_out, p->out};
    for (const void *ptr : ptrs16)
        if (!ptr || !aligned(ptr, 16)) return INKATTN_ERR_INVALID_ARG;
    const void *ptrs4[] = {p->cu_seqlens_q, p->state_slot};
    for (const void *ptr : ptrs4)
        if (!ptr || !aligned(ptr, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->dev_status && !aligned(p->dev_status, 4)) return INKATTN_ERR_INVALID_ARG;
    // h_out may be the residual array itself, but no other output may overlap an input
    const size_t row = (size_t)p->N_tok * p->D * 2;
    auto overlap = [](const void *a, size_t na, const void *b, size_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return na && nb && x < y + nb && y < x + na;
    };
    if (overlap(p->out, row, p->y, row) || overlap(p->out, row, p->residual, row) ||
        overlap(p->out, row, p->h_out, row) || overlap(p->h_out, row, p->y, row) ||
        (p->h_out != p->residual && overlap(p->h_out, row, p->residual, row)))
        return INKATTN_ERR_INVALID_ARG;
    return INKATTN_OK;
}

inkattn_status validate_qkvr(const inkattn_qkvr_params *p) {
    if (!p || p->struct_size != sizeof(inkattn_qkvr_params)) return INKATTN_ERR_INVALID_ARG;
    if (p->B < 1 || p->B > INKATTN_QKVR_MAX_SEQS || p->N_tok < 0 || p->max_seqlen_q < 0 || p->Hq < 1 ||
        p->Hkv < 1 || p->Hq % p->Hkv != 0 || p->Hq > 1024 || p->num_blocks < 1 || p->num_state_slots < 1 ||
        !(p->eps >= 0.f))
        return INKATTN_ERR_INVALID_ARG;
    if (p->N_tok > 0 && p->max_seqlen_q < 1) return INKATTN_ERR_INVALID_ARG;
    if (p->d_r < 1 || p->d_r > 1024 || ((long long)p->Hq * p->d_r) % 8 != 0) return INKATTN_ERR_INVALID_ARG;
    if (p->d_model < 8 || p->d_model % 8 != 0 || p->d_model > (1 << 20)) return INKATTN_ERR_INVALID_ARG;
    if ((long long)p->num_blocks * 64 > INT_MAX) return INKATTN_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || p->block_size != kBlock) return INKATTN_ERR_UNSUPPORTED;
    const void *ptrs16[] = {p->x, p->w, p->conv_state_k_in, p->conv_state_v_in, p->conv_state_k_out,
                            p->conv_state_v_out, p->q_out, p->r_out, p->k_cache, p->v_cache};
    for (const void *ptr : ptrs16)
        if (!ptr || !aligned(ptr, 16)) return INKATTN_ERR_INVALID_ARG;
    const void *ptrs4[] = {p->conv_w_k, p->conv_w_v, p->q_norm_w, p->k_norm_w, p->cu_seqlens_q,
                           p->state_slot, p->slot_mapping};
    for (const void *ptr : ptrs4)
        if (!ptr || !aligned(ptr, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->dev_status && !aligned(p->dev_status, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->y_out && !aligned(p->y_out, 16)) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype != INKATTN_KV_BF16 && p->kv_dtype != INKATTN_KV_E4M3) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype == INKATTN_KV_E4M3 &&
        (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 16) || !aligned(p->v_scale, 16)))
        return INKATTN_ERR_INVALID_ARG;
    // the new state is written while a sequence's first tile still reads the old one,
    // unless every sequence fits one tile
    if ((p->conv_state_k_out == p->conv_state_k_in || p->conv_state_v_out == p->conv_state_v_in) &&
        p->max_seqlen_q > INKATTN_QKVR_TILE_TOKENS)
        return INKATTN_ERR_INVALID_ARG;
    // no output overlaps an input or another output (in == out for the states excepted)
    const size_t F = (size_t)(p->Hq + 2 * p->Hkv) * kHeadDim + (size_t)p->Hq * p->d_r;
    const size_t st = (size_t)p->num_state_slots * 3 * p->Hkv * kHeadDim * 2;
    const size_t cache = (size_t)p->num_blocks * p->Hkv * 64 * kHeadDim * (p->kv_dtype == INKATTN_KV_E4M3 ? 1 : 2);
    struct Range { const void *a; size_t n; };
    const Range ins[] = {{p->x, (size_t)p->N_tok * p->d_model * 2}, {p->w, F * p->d_model * 2},
                         {p->conv_state_k_in, st}, {p->conv_state_v_in, st}};
    const Range outs[] = {{p->q_out, (size_t)p->N_tok * p->Hq * kHeadDim * 2},
                          {p->r_out, (size_t)p->N_tok * p->Hq * p->d_r * 2},
                          {p->k_cache, cache}, {p->v_cache, cache},
                          {p->conv_state_k_out, st}, {p->conv_state_v_out, st},
                          {p->y_out, p->y_out ? (size_t)p->N_tok * F * 2 : 0}};
    auto overlap = [](const Range &x, const Range &y) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(x.a), b = reinterpret_cast<uintptr_t>(y.a);
        return x.n && y.n && a < b + y.n && b < a + x.n;
    };
    constexpr int kOuts = sizeof(outs) / sizeof(outs[0]);
    for (int o = 0; o < kOuts; ++o) {
        for (int i = 0; i < 4; ++i) {
            const bool same_state = (o == 4 && i == 2 && outs[o].a == ins[i].a) ||
                                    (o == 5 && i == 3 && outs[o].a == ins[i].a);
            if (!same_state && overlap(outs[o], ins[i])) return INKATTN_ERR_INVALID_ARG;
        }
        for (int o2 = o + 1; o2 < kOuts; ++o2)
            if (overlap(outs[o], outs[o2])) return INKATTN_ERR_INVALID_ARG;
    }
    return INKATTN_OK;
}

// x and w are read by TMA: device memory of the current device (as for validate_locations)
inkattn_status validate_qkvr_locations(const inkattn_qkvr_params *p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return INKATTN_ERR_INVALID_ARG;
    }
    const void *ptrs[] = {p->x, p->w};
    for (const void *ptr : ptrs) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
            (void)cudaGetLastError();
            return INKATTN_ERR_INVALID_ARG;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return INKATTN_ERR_INVALID_ARG;
    }
    return INKATTN_OK;
}

inkattn_status validate_attn(const inkattn_attn_params *p) {
    if (!p || p->struct_size != sizeof(inkattn_attn_params)) return INKATTN_ERR_INVALID_ARG;
    if (p->B < 1 || p->B > 65535 || p->N_tok < 0 || p->max_seqlen_q < 0 || p->max_seqlen_k < 0 ||
        p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0 || p->Hq > 65535 || p->num_blocks < 1 ||
        p->max_blocks_per_seq < 1 || p->rel_extent < 0 || p->window < 0)
        return INKATTN_ERR_INVALID_ARG;
    if (p->N_tok > 0 && (p->max_seqlen_q < 1 || p->max_seqlen_k < p->max_seqlen_q))
        return INKATTN_ERR_INVALID_ARG;
    if ((long long)p->max_blocks_per_seq * kBlock < p->max_seqlen_k) return INKATTN_ERR_INVALID_ARG;
    if ((long long)p->num_blocks * p->Hkv * kBlock >= (1ll << 31)) return INKATTN_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || p->block_size != kBlock) return INKATTN_ERR_UNSUPPORTED;
    if (p->out_dtype != INKATTN_DTYPE_BF16 && p->out_dtype != INKATTN_DTYPE_F32) return INKATTN_ERR_INVALID_ARG;
    if (!(p->softmax_scale == p->softmax_scale) || !(p->log_scale_base == p->log_scale_base))
        return INKATTN_ERR_INVALID_ARG;
    const void *ptrs16[] = {p->q, p->k_cache, p->v_cache, p->out};
    for (const void *ptr : ptrs16)
        if (!ptr || !aligned(ptr, 16)) return INKATTN_ERR_INVALID_ARG;
    const void *ptrs4[] = {p->cu_seqlens_q, p->seqlen_k, p->block_table};
    for (const void *ptr : ptrs4)
        if (!ptr || !aligned(ptr, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->lse && !aligned(p->lse, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->dev_status && !aligned(p->dev_status, 4)) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype != INKATTN_KV_BF16 && p->kv_dtype != INKATTN_KV_E4M3) return INKATTN_ERR_INVALID_ARG;
    if (p->kv_dtype == INKATTN_KV_E4M3 &&
        (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 16) || !aligned(p->v_scale, 16)))
        return INKATTN_ERR_INVALID_ARG;
    if (p->rel_extent > 0) {
        if (p->d_r != 32) return INKATTN_ERR_UNSUPPORTED;
        if (!p->r || !p->P || !aligned(p->r, 16) || !aligned(p->P, 16)) return INKATTN_ERR_INVALID_ARG;
    }
    return INKATTN_OK;
}

// q, k_cache and v_cache are read by TMA through tensor maps, and the prefill kernel
// multicasts each K/V tile to the two CTAs of a head pair: the maps must cover memory of
// this GPU alone.  Each must be device memory of the current device; host memory (pinned
// or not), managed memory and another GPU's memory reached through unified addressing are
// rejected.  A pointer whose location the runtime cannot report is rejected too.
inkattn_status validate_locations(const inkattn_attn_params *p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return INKATTN_ERR_INVALID_ARG;
    }
    const bool f8 = p->kv_dtype == INKATTN_KV_E4M3;
    const void *q = p->q;
    const void *ptrs[] = {q, p->k_cache, p->v_cache, f8 ? static_cast<const void *>(p->k_scale) : q,
                          f8 ? static_cast<const void *>(p->v_scale) : q};
    for (const void *ptr : ptrs) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
            (void)cudaGetLastError();
            return INKATTN_ERR_INVALID_ARG;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return INKATTN_ERR_INVALID_ARG;
    }
    return INKATTN_OK;
}

AttnScalars scalars(const inkattn_attn_params &p) {
    AttnScalars s;
    s.scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)kHeadDim);
    s.group = p.Hq / p.Hkv;
    return s;
}

inkattn_status launch_status(cudaError_t e) { return e == cudaSuccess ? INKATTN_OK : INKATTN_ERR_CUDA; }

}  // namespace

// Decode split heuristic ([vLLM TML Inkling サポート, §低レイテンシコレクティブとカーネル
// "FA4 Kernel"]: num_splits from batch size, TP size and KV length; TP = 1 here).
// Cost model in units of one 64-key K+V block moved at the full HBM rate: a CTA streams
// `per` blocks at min(its own rate, HBM / active CTAs), so a wave with a CTAs costs
// per * max(r, a), where r is the number of CTAs that saturate HBM; the split partials add
// their write + read traffic and the combine launch a fixed cost.
int pick_splits(const inkattn_attn_params &p, int num_sms) {
    const int g = p.Hq / p.Hkv;
    long long nblk = (p.max_seqlen_k + kBlock - 1) / kBlock;
    if (p.window > 0) {
        const long long span = ((long long)p.window + p.max_seqlen_q + kBlock - 1) / kBlock + 1;
        if (span < nblk) nblk = span;
    }
    if (nblk < 1) nblk = 1;
    const long long units = (long long)p.B * p.Hkv;
    const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * kDecodeCtasPerSm;
    const double r = kDecodeHbmSmFrac * (double)slots;
    const long long rows_per_unit = (long long)p.max_seqlen_q * g;
    const double block_bytes = 2.0 * kBlock * kHeadDim * 2;   // K + V of one block
    // With a relative bias, two splits cut the keys at the band's start instead of halving
    // them (csrc/decode_tc.cu): the CTAs streaming the keys before the band come first in the
    // grid and the short band CTAs, whose bias tables take the longest, run beside them on
    // the SMs the last wave leaves free.  That pays when the streaming CTAs alone keep HBM
    // busy and the band is a small part of the keys; halves are then not a choice.
    const bool band_split = p.rel_extent > 0;
    const long long band_blk = ((long long)p.rel_extent + p.max_seqlen_q + kBlock - 1) / kBlock + 2;
    int best = 1;
    double best_cost = 1e300;
    for (int S = 1; S <= kDecodeMaxSplits; ++S) {
        const long long per = (nblk + S - 1) / S;
        if (S > 1 && per < kDecodeMinSplitBlocks) break;
        if (band_split && S == 2) continue;
        const long long ctas = units * S;
        const long long full = ctas / slots, rest = ctas - full * slots;
        double waves = (double)full * fmax(r, (double)slots);
        if (rest > 0) waves += fmax(r, (double)rest);
        double cost = (double)per * waves;
        if (S > 1) {
            const double ws_bytes = 2.0 * units * rows_per_unit * S * (kHeadDim + 1) * 4.0;
            cost += ws_bytes / block_bytes + kCombineCostBlocks;
        }
        if (cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = S;
        }
    }
    if (band_split && best == 1 && (double)units >= r && nblk >= 4 * band_blk) return 2;
    return best;
}

namespace {

size_t ws_o_bytes(const inkattn_attn_params &p, int S) {
    const size_t b = (size_t)p.N_tok * p.Hq * S * kHeadDim * 4;
    return (b + 255) & ~(size_t)255;
}
size_t ws_lse_bytes(const inkattn_attn_params &p, int S) {
    const size_t b = (size_t)p.N_tok * p.Hq * S * 4;
    return (b + 255) & ~(size_t)255;
}

inkattn_status validate_decode_shape(const inkattn_attn_params &p) {
    const int g = p.Hq / p.Hkv;
    if (p.max_seqlen_q > 16 || (long long)p.max_seqlen_q * g > kDecodeMaxRows) return INKATTN_ERR_UNSUPPORTED;
    return INKATTN_OK;
}

inkattn_status resolve_splits(const inkattn_attn_params &p, int requested, int *S_out) {
    if (requested < 0 || requested > kDecodeMaxSplits) return INKATTN_ERR_INVALID_ARG;
    if (requested > 0) {
        *S_out = requested;
        return INKATTN_OK;
    }
    int sms = 0;
    inkattn_status st = check_device(&sms);
    if (st != INKATTN_OK) return st;
    *S_out = pick_splits(p, sms);
    return INKATTN_OK;
}

}  // namespace

size_t decode_workspace_bytes(const inkattn_attn_params &p, int S) {
    return S > 1 ? ws_o_bytes(p, S) + ws_lse_bytes(p, S) : 0;
}

inkattn_status validate_decode_call(const inkattn_attn_params *p, int *sms) {
    inkattn_status st = validate_attn(p);
    if (st != INKATTN_OK) return st;
    if ((st = validate_decode_shape(*p)) != INKATTN_OK) return st;
    if ((st = validate_locations(p)) != INKATTN_OK) return st;
    return check_device(sms);
}

const KernelDebug &kernel_debug() {
    static const KernelDebug d = [] {
        KernelDebug k{kWaitLimitNsDefault, 0};
        if (const char *s = std::getenv("INKATTN_TEST_WAIT_LIMIT_US")) {
            const long long us = std::atoll(s);
            if (us >= 100 && us <= 10000000) k.wait_ns = (uint64_t)us * 1000ull;
        }
        if (const char *s = std::getenv("INKATTN_TEST_WITHHOLD_ARRIVAL")) k.withhold = std::atoi(s) == 1;
        return k;
    }();
    return d;
}

bool make_cache_map(CUtensorMap *map, const void *base, long long rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_cache_map_e4m3(CUtensorMap *map, const void *base, long long rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
    cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)kBlock};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_qkvr_maps(const inkattn_qkvr_params &p, CUtensorMap *xmap, CUtensorMap *wmap) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    const long long F = (long long)(p.Hq + 2 * p.Hkv) * kHeadDim + (long long)p.Hq * p.d_r;
    cuuint64_t strides[1] = {(cuuint64_t)p.d_model * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t xdims[2] = {(cuuint64_t)p.d_model, (cuuint64_t)(p.N_tok > 0 ? p.N_tok : 1)};
    cuuint64_t wdims[2] = {(cuuint64_t)p.d_model, (cuuint64_t)F};
    return enc(xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<inkattn_bf16 *>(p.x), xdims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
           enc(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<inkattn_bf16 *>(p.w), wdims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_q_map(CUtensorMap *map, const void *base, int n_tok, int hq, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hq, (cuuint64_t)(n_tok > 0 ? n_tok : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hq * kHeadDim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_q_group_map(CUtensorMap *map, const void *base, int n_tok, int hq, int group, int tokens) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hq, (cuuint64_t)(n_tok > 0 ? n_tok : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hq * kHeadDim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace inkattn

using namespace inkattn;

extern "C" {

const char *inkattn_status_string(inkattn_status s) {
    switch (s) {
        case INKATTN_OK: return "ok";
        case INKATTN_ERR_INVALID_ARG: return "invalid argument";
        case INKATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case INKATTN_ERR_CUDA: return "CUDA runtime error";
        case INKATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case INKATTN_ERR_DEVICE_BOUNDS: return "device index out of bounds";
    }
    return "unknown status";
}

int inkattn_abi_version(void) { return INKATTN_ABI_VERSION; }

inkattn_status inkattn_prologue(const inkattn_prologue_params *p, void *stream) {
    inkattn_status st = validate_prologue(p);
    if (st != INKATTN_OK) return st;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    if (p->N_tok == 0) return INKATTN_OK;
    return launch_status(launch_prologue(*p, static_cast<cudaStream_t>(stream)));
}

inkattn_status inkattn_output_conv(const inkattn_output_conv_params *p, void *stream) {
    inkattn_status st = validate_output_conv(p);
    if (st != INKATTN_OK) return st;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    if (p->N_tok == 0) return INKATTN_OK;
    return launch_status(launch_output_conv(*p, static_cast<cudaStream_t>(stream)));
}

inkattn_status inkattn_qkvr_prologue(const inkattn_qkvr_params *p, void *stream) {
    inkattn_status st = validate_qkvr(p);
    if (st != INKATTN_OK) return st;
    int sms = 0;
    if ((st = check_device(&sms)) != INKATTN_OK) return st;
    if ((st = validate_qkvr_locations(p)) != INKATTN_OK) return st;
    // no tokens and the states in place: nothing to do
    if (p->N_tok == 0 && p->conv_state_k_out == p->conv_state_k_in && p->conv_state_v_out == p->conv_state_v_in)
        return INKATTN_OK;
    CUtensorMap xmap, wmap;
    if (!make_qkvr_maps(*p, &xmap, &wmap)) return INKATTN_ERR_CUDA;
    return launch_status(launch_qkvr(*p, xmap, wmap, sms, static_cast<cudaStream_t>(stream)));
}

namespace {

// The prefill over a bf16 cache, once the call is validated.
inkattn_status run_prefill_bf16(const inkattn_attn_params &p, cudaStream_t stream) {
    CUtensorMap qmap, kmap, vmap;
    const long long rows = (long long)p.num_blocks * p.Hkv * kBlock;
    if (!make_q_map(&qmap, p.q, p.N_tok, p.Hq, kPrefillTcRows) ||
        !make_cache_map(&kmap, p.k_cache, rows) || !make_cache_map(&vmap, p.v_cache, rows))
        return INKATTN_ERR_CUDA;
    if (p.rel_extent == 0)   // no bias band: two query tiles per CTA
        return launch_status(launch_prefill_2q(p, scalars(p), qmap, kmap, vmap, stream));
    return launch_status(launch_prefill_tc(p, scalars(p), qmap, kmap, vmap, stream));
}

// Workspace of the prefill over an E4M3 cache: bf16 K and V copies of B * max_blocks_per_seq
// blocks, then their block table, each piece 256-byte aligned.
size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }
size_t prefill_copy_bytes(const inkattn_attn_params &p) {
    return (size_t)p.B * p.max_blocks_per_seq * p.Hkv * kBlock * kHeadDim * 2;
}
size_t prefill_ws_bytes(const inkattn_attn_params &p) {
    return 2 * round256(prefill_copy_bytes(p)) + round256((size_t)p.B * p.max_blocks_per_seq * 4);
}

}  // namespace

inkattn_status inkattn_prefill(const inkattn_attn_params *p, void *stream) {
    inkattn_status st = validate_attn(p);
    if (st != INKATTN_OK) return st;
    if (p->kv_dtype != INKATTN_KV_BF16) return INKATTN_ERR_UNSUPPORTED;   // (inkattn_prefill_e4m3)
    if ((st = validate_locations(p)) != INKATTN_OK) return st;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    if (p->N_tok == 0) return INKATTN_OK;
    return run_prefill_bf16(*p, static_cast<cudaStream_t>(stream));
}

size_t inkattn_prefill_workspace_bytes(const inkattn_attn_params *p) {
    if (validate_attn(p) != INKATTN_OK || p->kv_dtype != INKATTN_KV_E4M3) return 0;
    return prefill_ws_bytes(*p);
}

inkattn_status inkattn_prefill_e4m3(const inkattn_attn_params *p, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    inkattn_status st = validate_attn(p);
    if (st != INKATTN_OK) return st;
    if (p->kv_dtype != INKATTN_KV_E4M3) return INKATTN_ERR_INVALID_ARG;     // (inkattn_prefill)
    // the copy's rows are addressed by TMA as 32-bit coordinates
    if ((long long)p->B * p->max_blocks_per_seq * p->Hkv * kBlock >= (1ll << 31)) return INKATTN_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < prefill_ws_bytes(*p))
        return INKATTN_ERR_INVALID_ARG;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    if ((st = validate_locations(p)) != INKATTN_OK) return st;
    {   // the copy is read by TMA too: device memory of this GPU
        int dev = -1;
        cudaPointerAttributes a;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&a, workspace) != cudaSuccess) {
            (void)cudaGetLastError();
            return INKATTN_ERR_INVALID_ARG;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return INKATTN_ERR_INVALID_ARG;
    }
    if (p->N_tok == 0) return INKATTN_OK;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const size_t copy = round256(prefill_copy_bytes(*p));
    inkattn_bf16 *k16 = reinterpret_cast<inkattn_bf16 *>(ws);
    inkattn_bf16 *v16 = reinterpret_cast<inkattn_bf16 *>(ws + copy);
    int32_t *table = reinterpret_cast<int32_t *>(ws + 2 * copy);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = launch_status(launch_dequant_e4m3(*p, k16, v16, table, s))) != INKATTN_OK) return st;
    inkattn_attn_params q = *p;
    q.k_cache = k16;
    q.v_cache = v16;
    q.kv_dtype = INKATTN_KV_BF16;
    q.k_scale = nullptr;
    q.v_scale = nullptr;
    q.block_table = table;
    q.num_blocks = p->B * p->max_blocks_per_seq;
    return run_prefill_bf16(q, s);
}

int inkattn_decode_num_splits(const inkattn_attn_params *p, int num_sms) {
    if (validate_attn(p) != INKATTN_OK || validate_decode_shape(*p) != INKATTN_OK || num_sms < 1) return 0;
    return pick_splits(*p, num_sms);
}

size_t inkattn_decode_workspace_bytes(const inkattn_attn_params *p, int num_splits) {
    if (validate_attn(p) != INKATTN_OK) return 0;
    int S = 0;
    if (resolve_splits(*p, num_splits, &S) != INKATTN_OK || S <= 1) return 0;
    return ws_o_bytes(*p, S) + ws_lse_bytes(*p, S);
}

inkattn_status inkattn_decode(const inkattn_attn_params *p, int num_splits, void *workspace,
                              size_t workspace_bytes, void *stream) {
    inkattn_status st = validate_attn(p);
    if (st != INKATTN_OK) return st;
    if ((st = validate_decode_shape(*p)) != INKATTN_OK) return st;
    if (num_splits < 0 || num_splits > kDecodeMaxSplits) return INKATTN_ERR_INVALID_ARG;
    if ((st = validate_locations(p)) != INKATTN_OK) return st;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    int S = 0;
    if ((st = resolve_splits(*p, num_splits, &S)) != INKATTN_OK) return st;
    float *ws_o = nullptr, *ws_lse = nullptr;
    if (S > 1) {
        const size_t need = ws_o_bytes(*p, S) + ws_lse_bytes(*p, S);
        if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return INKATTN_ERR_INVALID_ARG;
        ws_o = static_cast<float *>(workspace);
        ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + ws_o_bytes(*p, S));
    }
    if (p->N_tok == 0) return INKATTN_OK;
    CUtensorMap qmap, kmap, vmap;
    const long long rows = (long long)p->num_blocks * p->Hkv * kBlock;
    auto cache_map = p->kv_dtype == INKATTN_KV_E4M3 ? make_cache_map_e4m3 : make_cache_map;
    if (!cache_map(&kmap, p->k_cache, rows) || !cache_map(&vmap, p->v_cache, rows) ||
        !make_q_group_map(&qmap, p->q, p->N_tok, p->Hq, p->Hq / p->Hkv, p->max_seqlen_q))
        return INKATTN_ERR_CUDA;
    return launch_status(launch_decode_tc(*p, scalars(*p), S, ws_o, ws_lse, qmap, kmap, vmap,
                                          static_cast<cudaStream_t>(stream)));
}

inkattn_status inkattn_combine(const inkattn_attn_params *p, int num_splits, const void *workspace,
                               size_t workspace_bytes, void *stream) {
    inkattn_status st = validate_attn(p);
    if (st != INKATTN_OK) return st;
    if ((st = validate_decode_shape(*p)) != INKATTN_OK) return st;
    if (num_splits < 0 || num_splits > kDecodeMaxSplits) return INKATTN_ERR_INVALID_ARG;
    if ((st = check_device(nullptr)) != INKATTN_OK) return st;
    int S = 0;
    if ((st = resolve_splits(*p, num_splits, &S)) != INKATTN_OK) return st;
    if (S <= 1 || p->N_tok == 0) return INKATTN_OK;
    const size_t need = ws_o_bytes(*p, S) + ws_lse_bytes(*p, S);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return INKATTN_ERR_INVALID_ARG;
    const float *ws_o = static_cast<const float *>(workspace);
    const float *ws_lse = reinterpret_cast<const float *>(static_cast<const char *>(workspace) + ws_o_bytes(*p, S));
    return launch_status(launch_combine(*p, S, ws_o, ws_lse, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
