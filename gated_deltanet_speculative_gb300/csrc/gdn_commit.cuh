// gdn_commit.cuh -- commit of each stream's accepted path (TensorFold #747,
// first note: "commit only each stream's accepted path"; TensorFold #932,
// Qwen3.5 CUDA note: recorded rows let the lane core "keep partial copies").
//
// One CTA per (value head h, stream s) copies the recorded [D x D] fp32 tile
// of the kept row into the stream's slot, plus 1/Hv of the kept row's conv
// tail.  Pure copy: 128-bit loads that bypass L1 and stream out of L2,
// 128-bit stores.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

struct CommitParams {
    int Hv, D, CH;
    float *state;             // [n_slots, Hv, D, D]
    uint16_t *tail;           // bf16 [n_slots, 3, CH]
    int n_slots;
    const int *slot;          // [S]
    const int *keep_row;      // [S]
    int n_rows;
    const float *rec_state;   // [R, Hv, D, D]
    const uint16_t *rec_tail; // bf16 [R, 3, CH]
    int *err;
};

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) gdn_commit_kernel(const CommitParams p) {
    const int h = blockIdx.x, s = blockIdx.y;
    const int kr = p.keep_row[s];
    if (kr == -1) return;   // nothing accepted: the slot keeps its bits
    const int sl = p.slot[s];
    if (kr < -1 || kr >= p.n_rows || sl < 0 || sl >= p.n_slots) {
        if (h == 0 && threadIdx.x == 0)
            raise_error(p.err, (sl < 0 || sl >= p.n_slots) ? GDN_DERR_SLOT : GDN_DERR_KEEP);
        return;
    }
    const size_t tile4 = (size_t)p.D * p.D / 4;
    const float4 *src = reinterpret_cast<const float4 *>(p.rec_state) + ((size_t)kr * p.Hv + h) * tile4;
    float4 *dst = reinterpret_cast<float4 *>(p.state) + ((size_t)sl * p.Hv + h) * tile4;
    // 8 loads in flight per thread before the first store
    constexpr int kUnroll = 8;
    for (size_t base = 0; base < tile4; base += (size_t)kUnroll * kCommitThreads) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t i = base + (size_t)u * kCommitThreads + threadIdx.x;
            if (i < tile4) v[u] = __ldcs(src + i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t i = base + (size_t)u * kCommitThreads + threadIdx.x;
            if (i < tile4) dst[i] = v[u];
        }
    }

    // this CTA's share of the tail, in 16-byte units (3*CH*2 is a multiple of 16)
    const size_t units = (size_t)3 * p.CH / 8;
    const size_t lo = units * h / p.Hv, hi = units * (h + 1) / p.Hv;
    const uint4 *tsrc = reinterpret_cast<const uint4 *>(p.rec_tail + (size_t)kr * 3 * p.CH);
    uint4 *tdst = reinterpret_cast<uint4 *>(p.tail + (size_t)sl * 3 * p.CH);
    for (size_t i = lo + threadIdx.x; i < hi; i += kCommitThreads) tdst[i] = __ldcs(tsrc + i);
}

}  // namespace gdn
