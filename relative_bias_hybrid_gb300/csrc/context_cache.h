// context_cache.h -- a small thread-safe map from a CUDA context's unique ID to a pointer
// that was looked up with that context current.  Device addresses belong to a context:
// after cudaDeviceReset, or for a caller that makes its own (non-primary) context current,
// an address cached per device index would point into another or a destroyed context.
// Context IDs (cuCtxGetId) are never reused within a process, so a cached entry can only
// be found again by the context it was looked up in.
//
// Plain C++ without CUDA types, so that its logic can be checked on a machine without a GPU.
#pragma once

#include <mutex>

namespace inkattn {

template <int kEntries>
class ContextCache {
  public:
    // The pointer cached for context `id`; on a miss, lookup(&ptr) is called (it returns
    // false on failure) and its result is cached while free entries are left (beyond that
    // every call of a new context looks up again).
    template <class Lookup>
    bool get(unsigned long long id, Lookup &&lookup, void **out) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < n_; ++i) {
            if (ids_[i] == id) {
                *out = vals_[i];
                return true;
            }
        }
        void *v = nullptr;
        if (!lookup(&v) || v == nullptr) return false;
        if (n_ < kEntries) {
            ids_[n_] = id;
            vals_[n_] = v;
            ++n_;
        }
        *out = v;
        return true;
    }

  private:
    std::mutex mu_;
    unsigned long long ids_[kEntries] = {};
    void *vals_[kEntries] = {};
    int n_ = 0;
};

}  // namespace inkattn
