// decode_noalloc.cu -- inkattn_decode_noalloc: the split-KV decode and its combine,
// with the split partials held in a fixed-size static device buffer instead of a
// workspace the caller allocates.
//
// Why it exists: some callers cannot call cudaMalloc at the point where they decode.
// Examples are code that runs inside a host function enqueued on a stream (CUDA API
// calls are not allowed there), plugin hosts that own every byte of device memory and
// hand the plugin only its inputs and outputs, and serving loops that must never
// allocate on the hot path because an allocation can synchronise the device.
//
// It adds nothing to the computation: it resolves the split count, points the existing
// inkattn_decode / inkattn_combine entry points at the static buffer, and returns.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/inkattn.h"
#include "internal.h"

namespace inkattn {
namespace {

// The split partials (fp32 outputs and log-sum-exps) of every call.  This is static
// device memory: each GPU on which this part of the library is loaded holds these
// INKATTN_DECODE_NOALLOC_MAX_BYTES until the process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_decode_scratch[INKATTN_DECODE_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the symbol
// names a host-side stand-in, not device memory, so the address must come from
// cudaGetSymbolAddress; it is looked up once per device and cached.
inkattn_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return INKATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return INKATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return INKATTN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return INKATTN_OK;
}

}  // namespace
}  // namespace inkattn

extern "C" inkattn_status inkattn_decode_noalloc(const inkattn_attn_params *p, int num_splits, void *stream) {
    if (!p || num_splits < 0 || num_splits > inkattn::kDecodeMaxSplits) return INKATTN_ERR_INVALID_ARG;
    int S = num_splits;
    if (S == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return INKATTN_ERR_CUDA;
        S = inkattn_decode_num_splits(p, sms);
        // 0 only for params inkattn_decode rejects: let it report which status applies
        if (S == 0) return inkattn_decode(p, 1, nullptr, 0, stream);
    }
    const size_t need = S > 1 ? inkattn_decode_workspace_bytes(p, S) : 0;
    if (need > (size_t)INKATTN_DECODE_NOALLOC_MAX_BYTES) return INKATTN_ERR_INVALID_ARG;
    void *ws = nullptr;
    if (need > 0) {
        const inkattn_status st = inkattn::scratch_address(&ws);
        if (st != INKATTN_OK) return st;
    }
    inkattn_status st = inkattn_decode(p, S, ws, need, stream);
    if (st != INKATTN_OK) return st;
    return inkattn_combine(p, S, ws, need, stream);
}
