// Device addresses of the library's file-scope __device__ arrays, cached per
// CUDA context.
//
// Host code cannot use a __device__ variable's name as an address: it names a
// host-side stand-in.  The device address comes from cudaGetSymbolAddress,
// and it belongs to the context that is current when the lookup runs.  A
// process can hold several contexts on one device (the primary context and
// driver-API contexts a host framework creates), and a device reset destroys
// the primary context and makes a new one on next use.  So addresses are
// cached by context, and a context is identified by cuCtxGetId, whose ids are
// unique for the life of the process: an address looked up in a context that
// has since been destroyed is never handed out for a later one.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace path {

// Unique id of the context current on the calling thread.  If the runtime has
// not yet made a context current here, `bind` is called once first (any
// runtime call that initialises the device's primary context will do).
inline cudaError_t current_context_id(unsigned long long *id, cudaError_t (*bind)(void *),
                                      void *bind_arg) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    static cudaError_t resolve_err = cudaSuccess;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            resolve_err = cudaErrorNotSupported;
            return;
        }
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            resolve_err = cudaErrorNotSupported;
            return;
        }
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (resolve_err != cudaSuccess) return resolve_err;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    if (!ctx) {
        cudaError_t e = bind(bind_arg);
        if (e != cudaSuccess) return e;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    }
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

// Cache of one symbol's device address per context.  `lookup` calls
// cudaGetSymbolAddress for the symbol (in the .cu file that defines it).
class PerContextAddress {
  public:
    using Lookup = cudaError_t (*)(void **);
    explicit PerContextAddress(Lookup lookup) : lookup_(lookup) {}

    cudaError_t get(void **out) {
        unsigned long long id = 0;
        void *fresh = nullptr;
        cudaError_t e = current_context_id(&id, &PerContextAddress::bind_by_lookup, this);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < n_; ++i)
            if (ids_[i] == id) {
                *out = addrs_[i];
                return cudaSuccess;
            }
        e = lookup_(&fresh);
        if (e != cudaSuccess) return e;
        // keep the most recent kSlots contexts (oldest entry replaced)
        const int slot = n_ < kSlots ? n_++ : (int)(next_++ % kSlots);
        ids_[slot] = id;
        addrs_[slot] = fresh;
        *out = fresh;
        return cudaSuccess;
    }

  private:
    static constexpr int kSlots = 64;
    static cudaError_t bind_by_lookup(void *self) {
        void *p = nullptr;
        return static_cast<PerContextAddress *>(self)->lookup_(&p);
    }
    Lookup lookup_;
    std::mutex mu_;
    unsigned long long ids_[kSlots] = {};
    void *addrs_[kSlots] = {};
    int n_ = 0;
    unsigned next_ = 0;
};

}  // namespace path
