// gdn_launch.h -- host-side launchers of the GDN kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include "gdn_rows.cuh"

namespace gdn {

// One template instantiation set per head width; each lives in its own
// translation unit (gdn_rows_d<D>.cu) so the build compiles them in parallel.
cudaError_t launch_rows_d32(int mode, const RowParams &p, int n_streams, cudaStream_t st);
cudaError_t launch_rows_d64(int mode, const RowParams &p, int n_streams, cudaStream_t st);
cudaError_t launch_rows_d128(int mode, const RowParams &p, int n_streams, cudaStream_t st);

template <int D>
cudaError_t launch_rows(int mode, const RowParams &p, int n_streams, cudaStream_t st) {
    const dim3 grid(p.Hv, n_streams), block(kRowThreads);
    if (mode == kStep) {
        // clusters of the G value heads that share a key head: the in-place
        // tail shift of the shared q/k channels waits for all of them
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = p.G;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, gdn_rows_kernel<D, kStep>, p);
    }
    if (mode == kWindow) gdn_rows_kernel<D, kWindow><<<grid, block, 0, st>>>(p);
    else if (mode == kWindowLog) gdn_rows_kernel<D, kWindowLog><<<grid, block, 0, st>>>(p);
    else gdn_rows_kernel<D, kTree><<<grid, block, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
