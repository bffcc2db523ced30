// gdn_launch.h -- host-side launchers of the GDN kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gdn_rows.cuh"

namespace gdn {

// One template instantiation set per head width; each lives in its own
// translation unit (gdn_rows_d<D>.cu) so the build compiles them in parallel.
cudaError_t launch_rows_d32(int mode, const RowParams &p, int n_streams, cudaStream_t st);
cudaError_t launch_rows_d64(int mode, const RowParams &p, int n_streams, cudaStream_t st);
cudaError_t launch_rows_d128(int mode, const RowParams &p, int n_streams, cudaStream_t st);

// Steps in clusters of the G value heads that share a key head (the in-place
// tail shift of the shared q/k channels waits for all of them), each head's
// state rows split over P CTAs of the cluster.
template <int D, int P>
cudaError_t launch_step(const RowParams &p, int n_streams, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Hv * P, n_streams);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.G * P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // The step may be scheduled before the previous kernel ends (it waits for
    // it, griddepcontrol.wait, before touching memory), which hides the launch
    // gap between back-to-back steps; a previous kernel that does not signal
    // its dependents simply runs to its end first.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gdn_rows_kernel<D, kStep, P>, p);
}

// Row slices per step CTA: double P while the cluster stays within 8 CTAs,
// every warp keeps at least one state row, and the grid stays within two
// CTAs per SM.
inline int step_slices(int D, int G, int Hv, int n_streams) {
    static std::atomic<int> n_sm[64];   // per device, 0 until first asked (any thread may fill it)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    int sms = n_sm[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 1;
        n_sm[dev].store(sms, std::memory_order_relaxed);
    }
    int P = 1;
    while (P * 2 * G <= 8 && P * 2 <= D / 8 && (long long)Hv * n_streams * P * 2 <= 2LL * sms) P *= 2;
    return P;
}

template <int D>
cudaError_t launch_rows(int mode, const RowParams &p, int n_streams, cudaStream_t st) {
    const dim3 grid(p.Hv, n_streams), block(kRowThreads);
    if (mode == kStep) {
        const int P = step_slices(D, p.G, p.Hv, n_streams);
        if constexpr (D >= 64)
            if (P == 8) return launch_step<D, 8>(p, n_streams, st);
        if (P == 4) return launch_step<D, 4>(p, n_streams, st);
        if (P == 2) return launch_step<D, 2>(p, n_streams, st);
        return launch_step<D, 1>(p, n_streams, st);
    }
    if (mode == kWindow) gdn_rows_kernel<D, kWindow><<<grid, block, 0, st>>>(p);
    else if (mode == kWindowLog) gdn_rows_kernel<D, kWindowLog><<<grid, block, 0, st>>>(p);
    else if (mode == kTreeLog) gdn_rows_kernel<D, kTreeLog><<<grid, block, 0, st>>>(p);
    else gdn_rows_kernel<D, kTree><<<grid, block, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
