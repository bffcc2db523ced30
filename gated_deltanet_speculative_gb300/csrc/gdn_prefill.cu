// gdn_prefill.cu -- launchers of the chunked prefill kernels (prep, scan, norm).
#include <cuda_runtime.h>

#include "gdn_prefill.cuh"
#include "gdn_prefill_launch.h"

namespace gdn {

namespace {

template <int D, int C, int DS, int NT>
cudaError_t launch(const PrefillParams &p, cudaStream_t st) {
    using Prep = PrepSmem<D, C>;
    using Scan = ScanSmem<D, C, DS>;
    constexpr bool TC = (D == 128 && C == 64);   // tensor-core prep and scan for d = 128
    cudaError_t e;
    if constexpr (TC) {
        e = cudaFuncSetAttribute(gdn_prefill_prep_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrepTcSmem);
        if (e != cudaSuccess) return e;
        gdn_prefill_prep_tc_kernel<C><<<dim3(p.Hv, p.max_chunks), kPrepTcThreads, kPrepTcSmem, st>>>(p);
    } else {
        e = cudaFuncSetAttribute(gdn_prefill_prep_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Prep::kBytes);
        if (e != cudaSuccess) return e;
        gdn_prefill_prep_kernel<D, C><<<dim3(p.Hv, p.max_chunks), kPrepThreads, Prep::kBytes, st>>>(p);
    }
    if constexpr (TC) {
        e = cudaFuncSetAttribute(gdn_prefill_scan_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanTcSmem);
        if (e != cudaSuccess) return e;
        gdn_prefill_scan_tc_kernel<C><<<dim3(p.Hv, p.n_seqs), kScanTcThreads, kScanTcSmem, st>>>(p);
    } else {
        e = cudaFuncSetAttribute(gdn_prefill_scan_kernel<D, C, DS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Scan::kBytes);
        if (e != cudaSuccess) return e;
        gdn_prefill_scan_kernel<D, C, DS, NT><<<dim3(D / DS, p.Hv, p.n_seqs), NT, Scan::kBytes, st>>>(p);
    }
    const size_t items = (size_t)p.n_tokens * p.Hv;
    const unsigned blocks = (unsigned)((items + kNormThreads / 32 - 1) / (kNormThreads / 32));
    gdn_prefill_norm_kernel<D><<<blocks, kNormThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_chunk_floats(int D) {
    switch (D) {
        case 32: return ChunkBlock<32, kPrefillChunk>::kFloats;
        case 64: return ChunkBlock<64, kPrefillChunk>::kFloats;
        default: return ChunkBlock<128, kPrefillChunk>::kFloats;
    }
}

cudaError_t launch_prefill(int D, const PrefillParams &p, cudaStream_t st) {
    switch (D) {
        case 32: return launch<32, kPrefillChunk, 32, 256>(p, st);
        case 64: return launch<64, kPrefillChunk, 32, 512>(p, st);
        default: return launch<128, kPrefillChunk, 64, 512>(p, st);
    }
}

}  // namespace gdn
