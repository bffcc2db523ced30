// gdn_prefill.cu -- launchers of the chunked prefill kernels (prep, scan, norm).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "gdn_prefill.cuh"
#include "gdn_prefill_launch.h"

namespace gdn {

// The bounded-wait failure path without a hang or a fault: the mbarrier is
// initialised for one arrival that never comes, no copy or MMA refers to it,
// so the wait runs out after `polls` polls, the error word records it, and
// the CTA leaves with nothing in flight.
__global__ void gdn_wait_selftest_kernel(uint32_t polls, int *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, polls)) raise_error(err, GDN_DERR_TIMEOUT);
}

cudaError_t launch_wait_selftest(unsigned polls, int *err, cudaStream_t st) {
    gdn_wait_selftest_kernel<<<1, 32, 0, st>>>(polls, err);
    return cudaGetLastError();
}

namespace {

// Chunk groups of a pipelined tensor-core prefill: prep of group g runs on
// the caller's stream, the scan of group g on a high-priority side stream as
// soon as that prep is done, so the scan (one CTA per head and sequence, far
// fewer than the SMs) overlaps the prep of the groups after it; the norm of
// group g runs on a third stream after that scan, so it never holds up the
// next scan.  Only the last group's scan and norm cannot overlap any prep,
// so with several sequences the groups shrink: each takes kGroupShare of the
// chunks left (at least kGroupMin).  A large share measured best there: a
// group's scan runs one chain per sequence it touches, so the scans of mixed
// groups take many SMs and starve a concurrent prep, and most of the prep is
// better done on all SMs first (512/1024/2048/4096 tokens: share 0.35 ->
// 0.817 ms, 0.75 -> 0.754 ms, one group 0.814 ms).  One sequence uses
// round_groups below.  How much of the GPU a prep may take while a scan runs
// is set in the launch loop.
constexpr double kGroupShare = 0.75;
constexpr int kGroupMin = 4;
constexpr int kMaxGroups = 64;

// Group boundaries of `chunks` chunks into b[0..n]; returns n.
int chunk_groups(int chunks, int (&b)[kMaxGroups + 1]) {
    int n = 0, at = 0;
    b[0] = 0;
    while (at < chunks && n < kMaxGroups) {
        const int left = chunks - at;
        int take = (int)(left * kGroupShare + 0.999);
        take = take < kGroupMin ? kGroupMin : take;
        if (left - take < kGroupMin || n == kMaxGroups - 1) take = left;
        at += take;
        b[++n] = at;
    }
    return n;
}

// Groups for one sequence, sized in whole prep rounds (a round = one item
// per CTA of the prep grid, a prep item taking about as long as a scan
// launch needs for one round's chunks): the first group fills kRounds0
// rounds of all n_sm SMs, each later one kRounds rounds of the n_sm - Hv SMs
// a prep keeps while a scan runs; the last takes what is left.
constexpr int kRounds0 = 2;
constexpr int kRounds = 2;
int round_groups(int chunks, int n_sm, int Hk, int Hv, int (&b)[kMaxGroups + 1]) {
    int first = kRounds0 * n_sm / Hk, later = kRounds * (n_sm - Hv) / Hk;
    first = first < 1 ? 1 : first;
    later = later < 1 ? 1 : later;
    int n = 0, at = 0;
    b[0] = 0;
    while (at < chunks && n < kMaxGroups) {
        int take = n == 0 ? first : later;
        if (chunks - at < take || n == kMaxGroups - 1) take = chunks - at;
        at += take;
        b[++n] = at;
    }
    return n;
}

// SMs of the current device (0 if unknown).
int sm_count() {
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

struct SideStream {
    cudaStream_t stream = nullptr;   // scans, highest priority
    cudaStream_t norm = nullptr;     // norms
    cudaEvent_t start = nullptr, ready = nullptr, scanned = nullptr, done = nullptr;
};
constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];
std::mutex g_side_mu;   // one pipelined enqueue at a time (they share the side stream's events)

// The side streams and events of the current device, made on first use
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
        cudaStream_t s = nullptr, sn = nullptr;
        cudaEvent_t ev[4] = {};
        e = cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, hi);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&sn, cudaStreamNonBlocking, lo);
        for (auto &x : ev)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
        if (e != cudaSuccess) {   // give back what was made; the next call tries again
            for (auto &x : ev)
                if (x) cudaEventDestroy(x);
            if (sn) cudaStreamDestroy(sn);
            if (s) cudaStreamDestroy(s);
            return e;
        }
        ss.start = ev[0];
        ss.ready = ev[1];
        ss.scanned = ev[2];
        ss.done = ev[3];
        ss.norm = sn;
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
    const dim3 norm_grid(p.Hv * kNormSplit, p.max_chunks);   // every chunk of the pass
    cudaError_t e;
    if constexpr (TC) {
        e = cudaFuncSetAttribute(gdn_prefill_prep_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrepTcSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_prefill_scan_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanTcSmem);
        if (e != cudaSuccess) return e;
        int bounds[kMaxGroups + 1];
        const int n_sm = sm_count() > 0 ? sm_count() : 1;
        const bool hold_one = p.n_seqs == 1 && n_sm - p.Hv >= p.Hk;
        const int groups = !pipelined ? 1
                           : hold_one ? round_groups(p.max_chunks, n_sm, p.Hk, p.Hv, bounds)
                                      : chunk_groups(p.max_chunks, bounds);
        if (groups <= 1) {   // one launch each; the prep grid takes at most one CTA per SM
            const int items = (p.c_hi - p.c_lo) * p.Hk;
            gdn_prefill_prep_tc_kernel<C><<<items < n_sm ? items : n_sm, kPrepTcThreads, kPrepTcSmem, st>>>(p);
            gdn_prefill_scan_tc_kernel<C><<<dim3(p.Hv, p.n_seqs), kScanTcThreads, kScanTcSmem, st>>>(p);
            gdn_prefill_norm_chunks_kernel<D, C><<<norm_grid, kNormThreads, 0, st>>>(p);
            return cudaGetLastError();
        }
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *ss = nullptr;
        if ((e = side_stream(&ss)) != cudaSuccess) return e;
        // the side streams start after the caller's earlier work ...
        if ((e = cudaEventRecord(ss->start, st)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->stream, ss->start, 0)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->norm, ss->start, 0)) != cudaSuccess) return e;
        for (int g = 0; g < groups; ++g) {
            p.c_lo = bounds[g];
            p.c_hi = bounds[g + 1];
            // A prep launched while a scan runs must leave the scan its SMs: when
            // a scan launch ends, the next one is dispatched a few microseconds
            // later, and prep CTAs still waiting for an SM would take the freed
            // ones and keep them for a whole prep item.  With one sequence the
            // scan is Hv CTAs, so every prep after the first runs as a
            // persistent grid of the other SMs.  With several, the number of
            // scan CTAs per group depends on the lengths (device data), so only
            // the second group's prep, which becomes ready together with the
            // first scan, starts with a launch small enough to leave one
            // sequence's scan its SMs.
            PrefillParams pp = p;
            int grid = (p.c_hi - p.c_lo) * p.Hk;
            if (g >= 1 && hold_one) {
                grid = grid < n_sm - p.Hv ? grid : n_sm - p.Hv;
            } else if (g == 1) {
                const int a = (n_sm - p.Hv) / p.Hk;
                if (a >= 1 && p.c_lo + a < p.c_hi) {
                    pp.c_hi = p.c_lo + a;
                    gdn_prefill_prep_tc_kernel<C><<<a * p.Hk, kPrepTcThreads, kPrepTcSmem, st>>>(pp);
                    pp.c_lo = pp.c_hi;
                    pp.c_hi = p.c_hi;
                    grid = (pp.c_hi - pp.c_lo) * p.Hk;
                }
            }
            gdn_prefill_prep_tc_kernel<C><<<grid, kPrepTcThreads, kPrepTcSmem, st>>>(pp);
            // (a recorded event may be recorded again once a wait on it is enqueued)
            if ((e = cudaEventRecord(ss->ready, st)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(ss->stream, ss->ready, 0)) != cudaSuccess) return e;
            gdn_prefill_scan_tc_kernel<C><<<dim3(p.Hv, p.n_seqs), kScanTcThreads, kScanTcSmem, ss->stream>>>(p);
            if ((e = cudaEventRecord(ss->scanned, ss->stream)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(ss->norm, ss->scanned, 0)) != cudaSuccess) return e;
            gdn_prefill_norm_chunks_kernel<D, C><<<dim3(p.Hv * kNormSplit, p.c_hi - p.c_lo), kNormThreads, 0, ss->norm>>>(p);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // ... and the caller's stream continues after all of it (the last
        // norm follows the last scan)
        if ((e = cudaEventRecord(ss->done, ss->norm)) != cudaSuccess) return e;
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
        gdn_prefill_norm_chunks_kernel<D, C><<<norm_grid, kNormThreads, 0, st>>>(p);
        return cudaGetLastError();
    }
}

}  // namespace

size_t prefill_chunk_floats(int D) {
    switch (D) {
        case 32: return ChunkBlock<32, kPrefillChunk>::kFloats;
        case 64: return ChunkBlock<64, kPrefillChunk>::kFloats;
        default: return TcBlock::kBytes / 4;   // d = 128: the tensor-core layout
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
