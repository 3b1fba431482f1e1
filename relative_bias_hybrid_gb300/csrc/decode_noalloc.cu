// decode_noalloc.cu -- inkattn_decode_noalloc: the split-KV decode and its combine,
// with the split partials held in a fixed-size static device buffer instead of a
// workspace the caller allocates.
//
// Why it exists: some callers cannot call cudaMalloc at the point where they decode.
// Plugin hosts own every byte of device memory and hand the plugin only its inputs and
// outputs; serving loops must never allocate on the hot path, because an allocation can
// synchronise the device.  The call itself still makes CUDA runtime calls (device and
// pointer queries, tensor-map encoding) and launches kernels, so it is not meant for
// places where no CUDA call at all is allowed.
//
// It adds nothing to the computation: it makes the checks inkattn_decode makes, resolves
// the split count, points the existing inkattn_decode / inkattn_combine entry points at the
// static buffer, and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/inkattn.h"
#include "context_cache.h"
#include "internal.h"

namespace inkattn {
namespace {

// The split partials (fp32 outputs and log-sum-exps) of every call.  This is static
// device memory: each GPU on which this part of the library is loaded holds these
// INKATTN_DECODE_NOALLOC_MAX_BYTES until the process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_decode_scratch[INKATTN_DECODE_NOALLOC_MAX_BYTES];

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique ID of the context current on this thread, through the runtime's driver entry
// points (no link against the driver library).  False when none is current.
bool current_context_id(unsigned long long *id) {
    std::call_once(g_ctx_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

ContextCache<32> g_scratch_cache;

// Device address of g_decode_scratch in the current context.  In host code the symbol
// names a host-side stand-in, not device memory, so the address comes from
// cudaGetSymbolAddress, made with the caller's context current; it is cached per context.
inkattn_status scratch_address(void **out) {
    auto lookup = [](void **v) {
        if (cudaGetSymbolAddress(v, g_decode_scratch) == cudaSuccess) return true;
        (void)cudaGetLastError();
        return false;
    };
    unsigned long long id = 0;
    if (current_context_id(&id))
        return g_scratch_cache.get(id, lookup, out) ? INKATTN_OK : INKATTN_ERR_CUDA;
    // no context reported: look up without caching
    return lookup(out) && *out ? INKATTN_OK : INKATTN_ERR_CUDA;
}

}  // namespace
}  // namespace inkattn

extern "C" inkattn_status inkattn_decode_noalloc(const inkattn_attn_params *p, int num_splits, void *stream) {
    using namespace inkattn;
    if (num_splits < 0 || num_splits > kDecodeMaxSplits) return INKATTN_ERR_INVALID_ARG;
    // the checks of inkattn_decode first, so that bad params or an unsupported device get
    // the same status here
    int sms = 0;
    inkattn_status st = validate_decode_call(p, &sms);
    if (st != INKATTN_OK) return st;
    int S = num_splits;
    if (S == 0) {
        // the heuristic's choice, lowered until the partials fit the static buffer
        S = pick_splits(*p, sms);
        while (S > 1 && decode_workspace_bytes(*p, S) > (size_t)INKATTN_DECODE_NOALLOC_MAX_BYTES) --S;
    }
    const size_t need = decode_workspace_bytes(*p, S);
    if (need > (size_t)INKATTN_DECODE_NOALLOC_MAX_BYTES) return INKATTN_ERR_INVALID_ARG;
    void *ws = nullptr;
    if (need > 0 && (st = scratch_address(&ws)) != INKATTN_OK) return st;
    if ((st = inkattn_decode(p, S, ws, need, stream)) != INKATTN_OK) return st;
    return inkattn_combine(p, S, ws, need, stream);
}
