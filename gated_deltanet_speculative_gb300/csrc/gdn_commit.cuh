// gdn_commit.cuh -- commit of each stream's accepted path (TensorFold #747,
// first note: of a shared round, each stream keeps only its accepted rows;
// TensorFold #932, Qwen3.5 CUDA note: the recorded rows are what lets the
// engine keep a stream's partially accepted window).
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
    const int *row_ptr;       // [S + 1] each stream's packed rows
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
    const int sl = p.slot[s], r0 = p.row_ptr[s], r1 = p.row_ptr[s + 1];
    // the kept row must be one of the stream's own rows (a stream keeps only
    // its own accepted path)
    const bool bad_slot = sl < 0 || sl >= p.n_slots;
    const bool bad_keep = r0 < 0 || r1 > p.n_rows || kr < r0 || kr >= r1;
    if (bad_slot || bad_keep) {
        if (h == 0 && threadIdx.x == 0) raise_error(p.err, bad_slot ? GDN_DERR_SLOT : GDN_DERR_KEEP);
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

// Commit by index (pooled records): the kept row's state and tail were
// recorded in pool entry rec_slot[r] of the cache itself, so stream s keeps
// them by taking that entry as its slot; its previous entry is handed back
// in freed[s] (-1 when nothing is committed).  One thread per stream.
struct SwapParams {
    int *slot;               // [S] in/out
    const int *row_ptr;      // [S + 1]
    const int *keep_row;     // [S]
    const int *rec_slot;     // [R]
    int *freed;              // [S] or nullptr
    int n_streams, n_rows, n_slots;
    int *err;
};

constexpr int kSwapThreads = 128;

__global__ void __launch_bounds__(kSwapThreads) gdn_commit_swap_kernel(const SwapParams p) {
    const int s = blockIdx.x * kSwapThreads + threadIdx.x;
    // Launched as a programmatic dependent of the window before it: while
    // that kernel finishes, ask L2 for the index words (only a hint; they
    // are read after the wait, when the previous kernel's writes are visible).
    if (s < p.n_streams) {
        prefetch_l2(p.keep_row + s);
        prefetch_l2(p.row_ptr + s);
        prefetch_l2(p.slot + s);
    }
    for (int i = s * 32; i < p.n_rows; i += gridDim.x * kSwapThreads * 32) prefetch_l2(p.rec_slot + i);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (s >= p.n_streams) return;
    // the four index words at once, then the kept row's entry
    const int kr = p.keep_row[s];
    const int r0 = p.row_ptr[s], r1 = p.row_ptr[s + 1], old = p.slot[s];
    int out = -1;
    if (kr != -1) {
        const bool bad_keep = r0 < 0 || r1 > p.n_rows || kr < r0 || kr >= r1;
        const int ne = bad_keep ? -1 : p.rec_slot[kr];
        const bool bad_slot = !bad_keep && (ne < 0 || ne >= p.n_slots || ne == old);
        if (bad_keep || bad_slot) {
            raise_error(p.err, bad_keep ? GDN_DERR_KEEP : GDN_DERR_SLOT);
        } else {
            p.slot[s] = ne;
            out = old;
        }
    }
    if (p.freed) p.freed[s] = out;
}

// Replay commit: slot[s] <- the committed state advanced along the kept path
// of the stream's logged window, one rank-1 update per row,  S <- u k^T + a S
// with the same rounding as the window (fma(u_i, k_j, a * S_ij)), so the
// result equals the state the window would have recorded for the kept row,
// bit for bit.  The path of a chain is rows row_ptr[s] .. keep_row[s]; that
// of a tree (TREE) the kept node's root-to-node path through the parent
// indices, root first.  The conv tail is the kept row's recorded tail.
// (TensorFold #932, tree note: the commit re-applies the accepted rows' logs
// to the committed state in a single pass, trees included.)
struct ReplayParams {
    int Hk, Hv, G, CH;
    float *state;
    uint16_t *tail;
    int n_slots;
    const int *slot;
    const int *row_ptr;
    const int *parent;        // [R] window-local parents (trees only)
    const int *keep_row;
    int n_rows;
    const float *log_a;       // [R, Hv]
    const float *log_u;       // [R, Hv, D]
    const float *log_k;       // [R, Hk, D]
    const uint16_t *rec_tail; // bf16 [R, 3, CH]
    int *err;
};

constexpr int kReplayThreads = 256;

template <int D, bool TREE = false>
__global__ void __launch_bounds__(kReplayThreads) gdn_commit_replay_kernel(const ReplayParams p) {
    constexpr int RPW = D / 8, CPL = D / 32;
    __shared__ __align__(16) float us[GDN_MAX_WINDOW][D];
    __shared__ __align__(16) float ks[GDN_MAX_WINDOW][D];
    __shared__ float as[GDN_MAX_WINDOW];
    __shared__ int path[TREE ? GDN_MAX_WINDOW : 1];   // trees: window-local rows of the kept path, root first
    __shared__ int path_len;
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kr = __ldg(p.keep_row + s);
    if (kr == -1) return;   // nothing accepted: the slot keeps its bits
    const int sl = __ldg(p.slot + s), r0 = __ldg(p.row_ptr + s), r1 = __ldg(p.row_ptr + s + 1);
    const bool bad_slot = sl < 0 || sl >= p.n_slots;
    const bool bad_keep = r0 < 0 || r1 > p.n_rows || kr < r0 || kr >= r1 || kr - r0 >= GDN_MAX_WINDOW;
    if (bad_slot || bad_keep) {
        if (h == 0 && tid == 0) raise_error(p.err, bad_slot ? GDN_DERR_SLOT : GDN_DERR_KEEP);
        return;
    }
    int n = kr - r0 + 1;
    if constexpr (TREE) {
        // the kept node's ancestors: parents lie below their children, so
        // the walk ends within kr - r0 + 1 steps; the path's rows in
        // ascending order are its rows from the root down
        __shared__ int par[GDN_MAX_WINDOW];
        if (tid < n) par[tid] = __ldg(p.parent + r0 + tid);
        __syncthreads();
        if (tid == 0) {
            unsigned mask = 0;
            int m = n - 1, ok = 1;
            while (m >= 0) {
                mask |= 1u << m;
                const int pm = par[m];
                if (pm < -1 || pm >= m) {
                    ok = 0;
                    break;
                }
                m = pm;
            }
            int len = 0;
            for (int i = 0; i < n; ++i)
                if ((mask >> i) & 1u) path[len++] = i;
            path_len = ok ? len : -1;
        }
        __syncthreads();
        n = path_len;
        if (n < 0) {
            if (h == 0 && tid == 0) raise_error(p.err, GDN_DERR_PARENT);
            return;
        }
    }
    const int kh = h / p.G;
    auto row_of = [&](int t) { return TREE ? r0 + path[t] : r0 + t; };   // packed row of path step t
    for (int i = tid; i < n * D / 4; i += kReplayThreads) {   // the path's logs into shared memory
        const int t = i / (D / 4), c4 = (i - t * (D / 4)) * 4;
        const size_t r = (size_t)row_of(t);
        cp_async16(&us[t][c4], p.log_u + (r * p.Hv + h) * D + c4);
        cp_async16(&ks[t][c4], p.log_k + (r * p.Hk + kh) * D + c4);
    }
    if (tid < n) as[tid] = __ldg(p.log_a + (size_t)row_of(tid) * p.Hv + h);
    // The tile streams through registers in blocks of RB rows a warp, the
    // next block's loads in flight while the current one is replayed: each
    // element's updates depend on that element alone, so the blocks can be
    // taken in any order and the arithmetic is that of the whole tile.
    constexpr int RB = RPW < 4 ? RPW : 4, NB = RPW / RB;
    float *tile = p.state + ((size_t)sl * p.Hv + h) * D * D;
    float cur[RB][CPL], nxt[RB][CPL];
    auto load_block = [&](float (&x)[RB][CPL], int b) {
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int c = 0; c < CPL; ++c) x[r][c] = tile[(size_t)(warp * RPW + b * RB + r) * D + lane * CPL + c];
    };
    load_block(cur, 0);
    cp_async_wait_all();
    __syncthreads();
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b + 1 < NB) load_block(nxt, b + 1);
        for (int t = 0; t < n; ++t) {
            const float a = as[t];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float ur = us[t][warp * RPW + b * RB + r];
#pragma unroll
                for (int c = 0; c < CPL; ++c) cur[r][c] = __fmaf_rn(ur, ks[t][lane * CPL + c], __fmul_rn(a, cur[r][c]));
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int c = 0; c < CPL; ++c) tile[(size_t)(warp * RPW + b * RB + r) * D + lane * CPL + c] = cur[r][c];
        if (b + 1 < NB) {
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int c = 0; c < CPL; ++c) cur[r][c] = nxt[r][c];
        }
    }
    // this CTA's share of the kept row's tail, in 16-byte units
    const size_t units = (size_t)3 * p.CH / 8;
    const size_t lo = units * h / p.Hv, hi = units * (h + 1) / p.Hv;
    const uint4 *tsrc = reinterpret_cast<const uint4 *>(p.rec_tail + (size_t)kr * 3 * p.CH);
    uint4 *tdst = reinterpret_cast<uint4 *>(p.tail + (size_t)sl * 3 * p.CH);
    for (size_t i = lo + tid; i < hi; i += kReplayThreads) tdst[i] = __ldcs(tsrc + i);
}

}  // namespace gdn
