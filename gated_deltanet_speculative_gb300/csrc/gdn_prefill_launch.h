// gdn_prefill_launch.h -- host-side entry to the chunked prefill kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

#include "gdn_prefill.cuh"

namespace gdn {

// Floats in one (chunk, value head) block of the prefill workspace.
size_t prefill_chunk_floats(int D);
// Enqueue prep, scan and norm on `st`.
cudaError_t launch_prefill(int D, const PrefillParams &p, cudaStream_t st);

}  // namespace gdn
