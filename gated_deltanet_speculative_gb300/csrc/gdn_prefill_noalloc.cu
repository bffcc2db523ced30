// gdn_prefill_noalloc.cu -- gdn_prefill for callers that cannot allocate.
//
// Some callers have no way to hand the prefill its workspace: code running
// where cudaMalloc is off limits (inside another runtime's memory pool that
// owns the whole device, a latency-bound serving loop where cudaMalloc's
// implicit device-wide synchronisation would stall every other stream, or a
// plugin interface that offers no scratch argument).  gdn_prefill_noalloc
// runs the same prefill kernels with their scratch in the file-scope device
// array below, so the call itself allocates nothing.
//
// Costs and limits of that choice:
//  - the array (GDN_PREFILL_NOALLOC_SCRATCH_BYTES = 64 MiB) is device memory
//    that stays reserved, until the process exits, on every GPU where this
//    module is loaded;
//  - sizes whose workspace (gdn_prefill_workspace_size) exceeds it are
//    refused with GDN_EWORKSPACE before anything is enqueued;
//  - every call uses the same array.  Two calls whose work overlaps on the
//    GPU (different streams, or different host threads on one device) race
//    on it; serialise them.  Nothing in it has to start at zero: each call's
//    kernels write every scratch byte they later read (the norm reads O only
//    for tokens of sequences the scan ran), so the previous call's leftovers
//    are never read.
//  - the array's name is only a host-side stand-in in host code; its device
//    address is looked up with that device current, after the arguments
//    have passed the host checks, by the first call made on that device, and
//    again by the first call after the device's context was destroyed and
//    made anew (cudaDeviceReset).  That lookup may load the module, so make
//    the first call on a device before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdn.h"
#include "gdn_context.h"
#include "gdn_prefill_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_PREFILL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_prefill_scratch on the current device.
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
    return gdn::symbol_address(g_prefill_scratch, out, &g_scratch_ptr[dev], &g_scratch_ctx[dev], g_scratch_mu) ==
                   cudaSuccess
               ? GDN_OK
               : GDN_ECUDA;
}

}  // namespace

extern "C" int gdn_prefill_noalloc(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                                   const int32_t *slot, const int32_t *cu_seqlens, int32_t n_seqs,
                                   int32_t n_tokens, const gdn_rows *rows, int32_t chunk, void *stream) {
    // every host check first: a refused call makes no CUDA call at all
    int rc = gdn::prefill_validate(dims, w, cache, slot, cu_seqlens, n_seqs, n_tokens, rows, chunk);
    if (rc != GDN_OK) return rc;
    const size_t need = gdn_prefill_workspace_size(dims, n_seqs, n_tokens, chunk);
    if (need == 0) return GDN_EINVAL;
    if (need > (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES) return GDN_EWORKSPACE;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != GDN_OK) return rc;
    // everything on the caller's stream: no side stream or event is made here
    return gdn::prefill_entry(dims, w, cache, slot, cu_seqlens, n_seqs, n_tokens, rows, chunk, scratch,
                              (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES, stream, false);
}
