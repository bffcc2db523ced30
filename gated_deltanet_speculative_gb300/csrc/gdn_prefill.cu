// gdn_prefill.cu -- launchers of the chunked prefill kernels (prep, scan, norm).
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_prefill.cuh"
#include "gdn_prefill_launch.h"

namespace gdn {

namespace {

// Chunk groups of a pipelined tensor-core prefill: prep of group g runs on
// the caller's stream, the scan of group g on a high-priority side stream as
// soon as that prep is done, so the scan (one CTA per head and sequence, far
// fewer than the SMs) overlaps the prep of the groups after it.  Both kernels
// hold one CTA per SM, so a scan CTA waits for a prep CTA to retire; more
// groups pipeline more finely but pay that wait (and a state round trip
// through the slot) more often.  On GB300, 27B-like heads: 1 / 2 / 4 / 6 /
// 10 / 16 groups took 0.81 / 0.72 / 0.68 / 0.72 / 0.77 / 0.72 ms for one
// 4722-token prompt and 1.10 / 1.13 / 1.07 / 1.08 / 1.16 / 1.24 ms for
// 512 + 1024 + 2048 + 4096 tokens.
constexpr int kPrefillGroups = 4;

struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t start = nullptr, ready = nullptr, done = nullptr;
};
constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];
std::mutex g_side_mu;   // one pipelined enqueue at a time (they share the side stream's events)

// The side stream and events of the current device, made on first use
// (call with g_side_mu held).
cudaError_t side_stream(SideStream **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideStream &ss = g_side[dev];
    if (!ss.stream) {
        int lo = 0, hi = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
        cudaStream_t s = nullptr;
        if ((e = cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, hi)) != cudaSuccess) return e;
        cudaEvent_t ev[3] = {};
        for (auto &x : ev)
            if ((e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming)) != cudaSuccess) return e;
        ss.start = ev[0];
        ss.ready = ev[1];
        ss.done = ev[2];
        ss.stream = s;
    }
    *out = &ss;
    return cudaSuccess;
}

template <int D, int C, int DS, int NT>
cudaError_t launch(const PrefillParams &p0, cudaStream_t st, bool pipelined) {
    using Prep = PrepSmem<D, C>;
    using Scan = ScanSmem<D, C, DS>;
    constexpr bool TC = (D == 128 && C == 64);   // tensor-core prep and scan for d = 128
    PrefillParams p = p0;
    p.c_lo = 0;
    p.c_hi = p.max_chunks;
    const size_t items = (size_t)p.n_tokens * p.Hv;
    const unsigned norm_blocks = (unsigned)((items + kNormThreads / 32 - 1) / (kNormThreads / 32));
    cudaError_t e;
    if constexpr (TC) {
        e = cudaFuncSetAttribute(gdn_prefill_prep_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrepTcSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_prefill_scan_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanTcSmem);
        if (e != cudaSuccess) return e;
        const int groups = pipelined ? min(p.max_chunks, kPrefillGroups) : 1;
        if (groups <= 1) {
            gdn_prefill_prep_tc_kernel<C><<<dim3(p.Hv, p.max_chunks), kPrepTcThreads, kPrepTcSmem, st>>>(p);
            gdn_prefill_scan_tc_kernel<C><<<dim3(p.Hv, p.n_seqs), kScanTcThreads, kScanTcSmem, st>>>(p);
            gdn_prefill_norm_kernel<D><<<norm_blocks, kNormThreads, 0, st>>>(p);
            return cudaGetLastError();
        }
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *ss = nullptr;
        if ((e = side_stream(&ss)) != cudaSuccess) return e;
        // the side stream starts after the caller's earlier work ...
        if ((e = cudaEventRecord(ss->start, st)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->stream, ss->start, 0)) != cudaSuccess) return e;
        const int per = (p.max_chunks + groups - 1) / groups;
        for (int lo = 0; lo < p.max_chunks; lo += per) {
            p.c_lo = lo;
            p.c_hi = min(p.max_chunks, lo + per);
            gdn_prefill_prep_tc_kernel<C><<<dim3(p.Hv, p.c_hi - p.c_lo), kPrepTcThreads, kPrepTcSmem, st>>>(p);
            // (a recorded event may be recorded again once a wait on it is enqueued)
            if ((e = cudaEventRecord(ss->ready, st)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(ss->stream, ss->ready, 0)) != cudaSuccess) return e;
            gdn_prefill_scan_tc_kernel<C><<<dim3(p.Hv, p.n_seqs), kScanTcThreads, kScanTcSmem, ss->stream>>>(p);
        }
        gdn_prefill_norm_kernel<D><<<norm_blocks, kNormThreads, 0, ss->stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // ... and the caller's stream continues after all of it
        if ((e = cudaEventRecord(ss->done, ss->stream)) != cudaSuccess) return e;
        return cudaStreamWaitEvent(st, ss->done, 0);
    } else {
        e = cudaFuncSetAttribute(gdn_prefill_prep_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Prep::kBytes);
        if (e != cudaSuccess) return e;
        gdn_prefill_prep_kernel<D, C><<<dim3(p.Hv, p.max_chunks), kPrepThreads, Prep::kBytes, st>>>(p);
        e = cudaFuncSetAttribute(gdn_prefill_scan_kernel<D, C, DS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Scan::kBytes);
        if (e != cudaSuccess) return e;
        gdn_prefill_scan_kernel<D, C, DS, NT><<<dim3(D / DS, p.Hv, p.n_seqs), NT, Scan::kBytes, st>>>(p);
        gdn_prefill_norm_kernel<D><<<norm_blocks, kNormThreads, 0, st>>>(p);
        return cudaGetLastError();
    }
}

}  // namespace

size_t prefill_chunk_floats(int D) {
    switch (D) {
        case 32: return ChunkBlock<32, kPrefillChunk>::kFloats;
        case 64: return ChunkBlock<64, kPrefillChunk>::kFloats;
        default: return ChunkBlock<128, kPrefillChunk>::kFloats;
    }
}

cudaError_t launch_prefill(int D, const PrefillParams &p, cudaStream_t st, bool pipelined) {
    switch (D) {
        case 32: return launch<32, kPrefillChunk, 32, 256>(p, st, pipelined);
        case 64: return launch<64, kPrefillChunk, 32, 512>(p, st, pipelined);
        default: return launch<128, kPrefillChunk, 64, 512>(p, st, pipelined);
    }
}

}  // namespace gdn
