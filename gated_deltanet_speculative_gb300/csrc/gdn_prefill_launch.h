// gdn_prefill_launch.h -- host-side entry to the chunked prefill kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

#include "gdn_prefill.cuh"

namespace gdn {

// Floats in one (chunk, value head) block of the prefill workspace.
size_t prefill_chunk_floats(int D);
// Enqueue prep, scan and norm so that they run after earlier work on `st`
// and later work on `st` runs after them.  pipelined: for d = 128, overlap the
// scan with the prep through a side stream of this module (made once per
// device); otherwise everything runs on `st`.
cudaError_t launch_prefill(int D, const PrefillParams &p, cudaStream_t st, bool pipelined);

// One CTA waits, with the prefill kernels' bounded mbarrier wait, for a
// phase that nothing completes; after `polls` polls it raises
// GDN_DERR_TIMEOUT in *err and returns.  Nothing is in flight meanwhile.
cudaError_t launch_wait_selftest(unsigned polls, int *err, cudaStream_t st);

// gdn_prefill's host checks of every argument except the workspace (a
// GDN_* status; nothing is enqueued and no CUDA call is made).
int prefill_validate(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                     const int32_t *cu_seqlens, int32_t n_seqs, int32_t n_tokens, const gdn_rows *rows,
                     int32_t chunk);

// gdn_prefill's validation and launch with the plan chosen by the caller
// (gdn_prefill: pipelined; gdn_prefill_noalloc: everything on `stream`).
int prefill_entry(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                  const int32_t *cu_seqlens, int32_t n_seqs, int32_t n_tokens, const gdn_rows *rows, int32_t chunk,
                  void *workspace, size_t workspace_bytes, void *stream, bool pipelined);

}  // namespace gdn
