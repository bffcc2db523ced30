// gdn_context.h -- identity of the calling thread's current CUDA context
// (internal).
//
// The library caches a few per-device addresses of its own __device__
// variables (the error word, the no-alloc prefill scratch).  Those addresses
// belong to the context the module was loaded in: after the caller destroys
// that context (cudaDeviceReset) and the runtime makes a new one, the module
// is loaded again, possibly elsewhere.  A cache entry therefore records the
// unique id of the context it was looked up in and is looked up again when
// the current context's id differs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace gdn {

// Unique id of the current context of the calling thread, or 0 if there is
// none yet or the driver does not offer the query (callers then look the
// address up on every call).  Driver entry points are fetched once through
// the runtime; the library does not link the driver library itself.
inline unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of a __device__ symbol of this module on the current
// device, cached per device and context.  `cache_addr` / `cache_ctx` are the
// caller's per-device slots, guarded by `mu`.
template <typename T>
cudaError_t symbol_address(const T &symbol, void **out, void **cache_addr, unsigned long long *cache_ctx,
                           std::mutex &mu) {
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (*cache_addr && id != 0 && *cache_ctx == id) {
        *out = *cache_addr;
        return cudaSuccess;
    }
    void *a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, symbol);
    if (e != cudaSuccess || !a) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    // the lookup may have made the context current: take its id now
    *cache_ctx = current_context_id();
    *cache_addr = *cache_ctx != 0 ? a : nullptr;
    *out = a;
    return cudaSuccess;
}

}  // namespace gdn
