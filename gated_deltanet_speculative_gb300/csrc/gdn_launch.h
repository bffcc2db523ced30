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

// SMs of the current device (0 if unknown), cached per device.
inline int sm_count() {
    static std::atomic<int> n_sm[64];   // per device, 0 until first asked (any thread may fill it)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int sms = n_sm[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
        n_sm[dev].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

// Row slices per step CTA: double P while the cluster stays within 8 CTAs,
// every warp keeps at least one state row, and the grid stays within two
// CTAs per SM.
inline int step_slices(int D, int G, int Hv, int n_streams) {
    const int sms = sm_count();
    if (sms == 0) return 1;
    int P = 1;
    while (P * 2 * G <= 8 && P * 2 <= D / 8 && (long long)Hv * n_streams * P * 2 <= 2LL * sms) P *= 2;
    return P;
}

// Windows and trees of few streams split each head's state rows over P CTAs
// of a cluster of P (they shift no tail in place, so a cluster is one
// head's slices): double P while the cluster stays within 8 CTAs, every warp
// keeps at least one state row, and every CTA still has an SM of its own.
// A window CTA runs its rows one after another, so a slice that shares an
// SM gains little: on the GB300, 27B-like heads, one stream x 16 rows took
// 35.5 / 25.2 / 27.3 / 29.3 us at P = 1 / 2 / 4 / 8, two streams 35.5 /
// 35.5 / 33.4 / 47.8, four 58.0 / 64.2 / 58.0 / 78.5.
inline int window_slices(int D, int Hv, int n_streams) {
    const int sms = sm_count();
    if (sms == 0) return 1;
    int P = 1;
    while (P * 2 <= 8 && P * 2 <= D / 8 && (long long)Hv * n_streams * P * 2 <= (long long)sms) P *= 2;
    return P;
}

template <int D, int MODE, int P>
cudaError_t launch_window_sliced(const RowParams &p, int n_streams, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Hv * P, n_streams);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gdn_rows_kernel<D, MODE, P>, p);
}

template <int D, int MODE>
cudaError_t launch_window_mode(const RowParams &p, int n_streams, cudaStream_t st) {
    const int P = window_slices(D, p.Hv, n_streams);
    if constexpr (D >= 64)
        if (P == 8) return launch_window_sliced<D, MODE, 8>(p, n_streams, st);
    if (P == 4) return launch_window_sliced<D, MODE, 4>(p, n_streams, st);
    if (P == 2) return launch_window_sliced<D, MODE, 2>(p, n_streams, st);
    gdn_rows_kernel<D, MODE><<<dim3(p.Hv, n_streams), kRowThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_rows(int mode, const RowParams &p, int n_streams, cudaStream_t st) {
    if (mode == kStep) {
        const int P = step_slices(D, p.G, p.Hv, n_streams);
        if constexpr (D >= 64)
            if (P == 8) return launch_step<D, 8>(p, n_streams, st);
        if (P == 4) return launch_step<D, 4>(p, n_streams, st);
        if (P == 2) return launch_step<D, 2>(p, n_streams, st);
        return launch_step<D, 1>(p, n_streams, st);
    }
    if (mode == kWindow) return launch_window_mode<D, kWindow>(p, n_streams, st);
    if (mode == kWindowLog) return launch_window_mode<D, kWindowLog>(p, n_streams, st);
    if (mode == kTreeLog) return launch_window_mode<D, kTreeLog>(p, n_streams, st);
    return launch_window_mode<D, kTree>(p, n_streams, st);
}

}  // namespace gdn
