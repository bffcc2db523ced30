// gdn_rows.cuh -- the GDN row kernel: one-row steps, chain windows and tree
// windows share this one template, so their arithmetic is the same code.
//
// Work decomposition (one CTA per (value head h, stream s); 8 warps):
//   warp w owns state rows i in [w*D/8, (w+1)*D/8) of the [D x D] fp32 tile,
//   lane l owns columns j in [l*D/32, (l+1)*D/32).  The tile stays in
//   registers for the whole window, so it crosses HBM once on the way in and
//   once per recorded row on the way out.
//
// Steps, windows and trees may also split the tile's rows over P CTAs of a
// cluster (P slices of D/P rows; every state row evolves from its own row,
// k, q and the gates alone), when the (stream, head) units alone would
// leave SMs idle.  Each row's sums stay inside one warp with the same lane
// layout, so a sliced step or window equals an unsliced one bit for bit; the
// RMSNorm, the only step that mixes rows, sums o^2 in one order whatever the
// slicing (a slice's rows are an aligned lane group of the butterfly), and
// the slices complete that sum through distributed shared memory.
//
// Per row (TensorFold #932, Qwen3.5 CUDA engine note: gated delta rule and
// causal convolution; tree note: taps and recurrence follow each row's
// branch):
//   a1  resolve the row's parent and its three conv ancestors
//   a2  conv (width 4, kept tail) + SiLU for the head's q, k, v channels
//   a3  L2 norm of q and k, q scaled
//   a4  decay a = exp(-exp(A_log) softplus(a_in + dt_bias)), beta = sigmoid(b_in)
//   a5  p = S k and S q in one pass over the tile (one reduce-scatter),
//       u = beta (v - a p),  S <- a S + u k^T,  o = a (S q) + u (k . q)
//       -- algebraically S' = a S (I - beta k k^T) + beta v k^T, o = S' q
//   a6  record S and the conv tail after the row (windows and trees)
//   a7  y = o / sqrt(mean o^2 + eps) * w_norm * SiLU(z), rounded to bf16
#pragma once

#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {

// kWindowLog / kTreeLog: a chain or tree window that logs each row's decay,
// write u and key instead of recording its state (TensorFold #932, tree
// note: per-row logs of the decay, the write vector and the key replace the
// recorded states, and the commit replays them).  A logged tree node whose
// parent is not the node visited just before it rebuilds the parent's state
// from the committed slot by re-applying the logged rows of the path down to
// the parent, with the forward pass's own rounding, so it continues from
// the same bits the recorded tree would have re-read.
enum RowMode : int { kStep = 0, kWindow = 1, kTree = 2, kWindowLog = 3, kTreeLog = 4 };

struct RowParams {
    int Hk, Hv, G, CH;
    float q_scale, eps_l2, eps_rms;
    const uint16_t *conv_w;   // bf16 [CH, 4]
    const float *A_log;       // [Hv]
    const float *dt_bias;     // [Hv]
    const uint16_t *norm_w;   // bf16 [D]
    float *state;             // [n_slots, Hv, D, D]
    uint16_t *tail;           // bf16 [n_slots, 3, CH]
    int n_slots;
    const uint16_t *mixed;    // bf16 [R, CH]
    const uint16_t *z;        // bf16 [R, Hv, D]
    const uint16_t *a;        // bf16 [R, Hv]
    const uint16_t *b;        // bf16 [R, Hv]
    uint16_t *y;              // bf16 [R, Hv, D]
    const int *slot;          // [S]
    const int *row_ptr;       // [S + 1] (windows, trees)
    const int *parent;        // [R] (trees)
    int n_rows;
    float *rec_state;         // [R, Hv, D, D], or the state pool (pooled records)
    uint16_t *rec_tail;       // bf16 [R, 3, CH], or the tail pool (pooled records)
    const int *rec_slot;      // [R] pooled records: row r is recorded at entry rec_slot[r]; else nullptr
    float *log_a;             // [R, Hv] decay (logged modes)
    float *log_u;             // [R, Hv, D] write u = b (v - a S k) (logged modes)
    float *log_k;             // [R, Hk, D] normalised key (logged modes)
    int *err;                 // device error word
    int early_state;          // steps: read slot, state, tail and weights before the wait (the kernel
                              // before this one writes none of them)
    // d >= 64: tensor maps of the staged inputs (TMA), encoded per call on the host
    int box_rows;             // rows of one mixed / z box: 1 for steps, min(16, R) otherwise
    CUtensorMap map_mixed;    // [R rows][CH] bf16, box [box_rows][D]
    CUtensorMap map_tail;     // [n_slots * 3 rows][CH] bf16, box [3][D]
    CUtensorMap map_z;        // [R][Hv][D] bf16, box [box_rows][1][D]
};

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kMaxRows = GDN_MAX_WINDOW;
constexpr uint32_t kRowWaitLimit = 1u << 22;   // polls of the staging mbarrier before giving up

// Unclustered windows and trees of d >= 64 stage their inputs with TMA.
// d = 32 (a parity geometry, whose 3-row tail block is not a multiple of 128
// bytes), steps and row-sliced windows and trees use 16-byte cp.async: a
// step has one row to stage, and clustered CTAs must not leave early on a
// staging timeout, which would strand their partners at the cluster
// barriers.
template <int D, int MODE, int P>
__host__ __device__ constexpr bool rows_use_tma() { return D >= 64 && MODE != kStep && P == 1; }

template <int D>
struct __align__(128) RowSmem {
    // The staging areas come first: a TMA box lands on a 128-byte boundary
    // (for d = 64 and 128 every box start below is one).
    union {
        // staged bf16 conv inputs of this head's q, k and v channels, part by
        // part: rows 0..2 are the committed tail (oldest first), row 3 + t is
        // window row t
        uint16_t xin[3][kMaxRows + 3][D];
        float o[kMaxRows][D];   // written by the recurrence, after the conv
    } u;
    uint16_t z[kMaxRows][D];
    float q[kMaxRows][D];
    float k[kMaxRows][D];
    float v[kMaxRows][D];
    uint16_t cw[3 * D][4];   // conv weights of this head's q | k | v channels
    uint16_t nw[D];          // RMSNorm weight
    float decay[kMaxRows];
    float beta[kMaxRows];
    float kq[kMaxRows];
    // conv ancestors m = 1, 2, 3 steps back along the branch: e >= 0 is a
    // window-local row, e < 0 is row 3 + e of the committed tail; either way
    // the ancestor's staged row is 3 + e
    int anc[kMaxRows][3];
    int parent[kMaxRows];
    int recidx[kMaxRows];   // where each row's state and tail are recorded (row r0 + t, or its pool entry)
    int reused[kMaxRows];   // tree: re-read later by a child that does not follow it
    int order[kMaxRows];    // tree: depth-first preorder (children in row order); else 0, 1, ...
    int bad;
};

template <int CPL>
__device__ __forceinline__ void load_cols(float (&x)[CPL], const float *src) {
    if constexpr (CPL == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (CPL == 2) {
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = __ldcg(src);
    }
}

template <int CPL>
__device__ __forceinline__ void store_cols(float *dst, const float (&x)[CPL], bool streaming) {
    if constexpr (CPL == 4) {
        const float4 t = make_float4(x[0], x[1], x[2], x[3]);
        if (streaming) __stcs(reinterpret_cast<float4 *>(dst), t);
        else *reinterpret_cast<float4 *>(dst) = t;
    } else if constexpr (CPL == 2) {
        const float2 t = make_float2(x[0], x[1]);
        if (streaming) __stcs(reinterpret_cast<float2 *>(dst), t);
        else *reinterpret_cast<float2 *>(dst) = t;
    } else {
        if (streaming) __stcs(dst, x[0]);
        else *dst = x[0];
    }
}

template <int D, int RPW, int CPL>
__device__ __forceinline__ void load_tile(float (&S)[RPW][CPL], const float *tile, int warp, int lane) {
#pragma unroll
    for (int r = 0; r < RPW; ++r) load_cols<CPL>(S[r], tile + (size_t)(warp * RPW + r) * D + lane * CPL);
}

template <int D, int RPW, int CPL>
__device__ __forceinline__ void store_tile(float *tile, const float (&S)[RPW][CPL], int warp, int lane,
                                           bool streaming) {
#pragma unroll
    for (int r = 0; r < RPW; ++r) store_cols<CPL>(tile + (size_t)(warp * RPW + r) * D + lane * CPL, S[r], streaming);
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// The two halves of a cluster barrier, for a CTA that only needs to know
// that every CTA of its cluster has started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Global conv channel of element e of part (0 = q, 1 = k, 2 = v) of value head h.
template <int D>
__device__ __forceinline__ int channel_of(int part, int e, int Hk, int kh, int h) {
    return part == 0 ? kh * D + e : (part == 1 ? (Hk + kh) * D + e : 2 * Hk * D + h * D + e);
}

// Store v at the same shared-memory variable of CTA `rank` of this cluster.
__device__ __forceinline__ void st_cluster_f32(const float *local, uint32_t rank, float v) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

template <int D, int MODE, int P = 1>
__global__ void __launch_bounds__(kRowThreads, 2) gdn_rows_kernel(const __grid_constant__ RowParams p) {
    static_assert(P == 1 || D / (kRowWarps * P) >= 1, "every warp keeps at least one state row");
    constexpr int RPW = D / (kRowWarps * P);      // state rows per warp
    constexpr int CPL = D / 32;                   // state columns per lane
    constexpr int NV = 2 * RPW;                   // partial sums per lane: S k and S q
    constexpr int SHIFT = 5 - Log2<NV>::value;    // lane l holds total (l >> SHIFT)
    constexpr int SEG = D * 2 / 16;               // 16-byte chunks in one q, k or v segment
    constexpr int CHUNKS = 3 * SEG;               // 16-byte chunks in a staged row
    constexpr bool TMA = rows_use_tma<D, MODE, P>();
    static_assert(NV >= 2 && NV <= 32, "unsupported head width");
    constexpr bool TREE = MODE == kTree || MODE == kTreeLog;
    constexpr bool LOG = MODE == kWindowLog || MODE == kTreeLog;
    // sliced RMSNorm: exchange per-slice partial sums (P >= 4) or gather the
    // o rows (P = 2; measured faster there)
    constexpr bool kPartials = P >= 4;

    __shared__ RowSmem<D> sm;
    __shared__ __align__(8) uint64_t stage_bar;   // TMA staging completes here
    __shared__ int stage_fail;                    // a staging wait gave up
    // the whole o vector of each row, gathered from the slices
    // sliced: this slice's o rows (at their row index), and every slice's
    // partial sum of o^2 per row, gathered through distributed shared memory
    __shared__ float o_all[P > 1 && MODE != kStep ? kMaxRows : 1][P > 1 ? D : 1];
    __shared__ float part_all[P > 1 && MODE != kStep ? kMaxRows : 1][P];
    // logged trees: every row's write u (to rebuild a parent's state) and,
    // per node, the set of rows on its root-to-node path (bit m = row m)
    __shared__ float u_rows[MODE == kTreeLog ? kMaxRows : 1][MODE == kTreeLog ? D : 1];
    __shared__ int path_mask[MODE == kTreeLog ? kMaxRows : 1];
    const int h = blockIdx.x / P, s = blockIdx.y;
    const int sli = blockIdx.x % P;               // row slice: state rows [row0, row0 + D/P)
    const int row0 = sli * (D / P);
    // cluster rank of slice 0 of this head: a step's cluster holds the G value
    // heads of its key head (G * P CTAs), a window's only the P slices of one head
    const int crank0 = MODE == kStep ? (h % p.G) * P : 0;
    if constexpr (P > 1) cluster_arrive_relaxed();   // "started"; waited on before the first remote store
    // Steps are launched as programmatic dependents of the kernel before them
    // (decode runs them back to back, layer after layer): the CTAs may be
    // scheduled while that kernel finishes, and wait here, before their first
    // global access, until it has completed and its writes are visible, so
    // ordering is that of a plain launch; then they let the next step be
    // scheduled in turn.
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kh = h / p.G;
    const size_t CH = (size_t)p.CH;
    // The slot word, the conv and norm weights, and (steps) the state tile
    // and the committed tail: issued by issue_state(), before the wait for a
    // step launched with early_state, else after it.
    int sl = 0;
    float A_log = 0.0f, dt_bias = 0.0f;
    float S[RPW][CPL];
    const size_t tile = (size_t)D * D;
    auto issue_state = [&](bool tile_and_tail) {
        sl = __ldg(p.slot + s);
        for (int i = tid; i < 3 * D / 2; i += kRowThreads) {   // two channels (16 bytes) per copy
            const int part = i / (D / 2), e0 = (i - part * (D / 2)) * 2;
            cp_async16(&sm.cw[part * D + e0][0], p.conv_w + (size_t)channel_of<D>(part, e0, p.Hk, kh, h) * 4);
        }
        if (tid < D / 8) cp_async16(&sm.nw[tid * 8], p.norm_w + tid * 8);
        A_log = __ldg(p.A_log + h);
        dt_bias = __ldg(p.dt_bias + h);
        if (tile_and_tail && sl >= 0 && sl < p.n_slots) {
            load_tile<D, RPW, CPL>(S, p.state + ((size_t)sl * p.Hv + h) * tile + (size_t)row0 * D, warp, lane);
            const uint16_t *tl = p.tail + (size_t)sl * 3 * CH;
            for (int i = tid; i < 3 * CHUNKS; i += kRowThreads) {   // the three committed tail rows
                const int row = i / CHUNKS, ch = i - row * CHUNKS;
                const int part = ch / SEG, off = (ch - part * SEG) * 8;
                cp_async16(&sm.u.xin[part][row][off], tl + (size_t)row * CH + channel_of<D>(part, off, p.Hk, kh, h));
            }
        }
    };
    const bool early = MODE == kStep && p.early_state;   // uniform over the grid
    if constexpr (MODE == kStep) {
        if (early) {
            // The kernel before writes none of the slot words, the cache or
            // the weights (the caller's promise): read them now, while it
            // finishes; only the row's inputs wait.
            issue_state(true);
            if (warp == 0 && sli == 0) {   // ask L2 for the input row's q, k, v segments and z
                if (lane >= 10 && lane <= 12)
                    prefetch_l2_bulk(p.mixed + (size_t)s * CH + channel_of<D>(lane - 10, 0, p.Hk, kh, h),
                                     (uint32_t)(D * 2));
                if (lane == 13) prefetch_l2_bulk(p.z + ((size_t)s * p.Hv + h) * D, (uint32_t)(D * 2));
            }
        } else {
            // While the kernel before this step finishes, ask L2 for what the step
            // reads that no kernel of the layer loop writes: this slice of the
            // committed state tile, the head's conv weights and tail, and the
            // step's input row.  Prefetches only move lines into L2, which every
            // write reaches, so they cannot change a result.  The slot word is
            // read on the L2 path (no L1 line survives across the wait) and only
            // chooses what to prefetch; the step reads it again after the wait.
            if (warp == 0) {
                const int sl0 = __ldcg(p.slot + s);
                if (sl0 >= 0 && sl0 < p.n_slots) {
                    if (lane == 0)
                        prefetch_l2_bulk(p.state + ((size_t)sl0 * p.Hv + h) * D * D + (size_t)row0 * D,
                                         (uint32_t)(D / P * D * 4));
                    if (sli == 0 && lane >= 1 && lane <= 9) {   // tail rows x (q, k, v) segments
                        const int m = (lane - 1) / 3, part = (lane - 1) % 3;
                        prefetch_l2_bulk(p.tail + ((size_t)sl0 * 3 + m) * CH + channel_of<D>(part, 0, p.Hk, kh, h),
                                         (uint32_t)(D * 2));
                    }
                }
                if (sli == 0 && lane >= 10 && lane <= 12) {   // the input row's q, k, v segments
                    const int part = lane - 10;
                    prefetch_l2_bulk(p.mixed + (size_t)s * CH + channel_of<D>(part, 0, p.Hk, kh, h), (uint32_t)(D * 2));
                }
                if (sli == 0 && lane == 13) prefetch_l2_bulk(p.z + ((size_t)s * p.Hv + h) * D, (uint32_t)(D * 2));
                if (sli == 0 && lane >= 14 && lane <= 16) {   // conv weights of the three segments
                    const int part = lane - 14;
                    prefetch_l2_bulk(p.conv_w + (size_t)channel_of<D>(part, 0, p.Hk, kh, h) * 4, (uint32_t)(D * 8));
                }
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        // A window or tree lets a kernel launched after it as a programmatic
        // dependent (the index commit) be scheduled as soon as every CTA of
        // this grid has started: that kernel waits for this grid's end
        // (griddepcontrol.wait) before it reads or writes anything.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    const bool lead = (h % p.G) == 0;    // this CTA writes the q/k channels shared by its key-head group

    // ---- a1: the stream's slot and rows (the same few words in every thread)
    // While those words are in flight: the conv and norm weights (independent
    // of every index), so that no later phase waits on a load of its own.
    if (!early) issue_state(false);
    int r0 = s, n = 1;
    if (MODE != kStep) {
        r0 = __ldg(p.row_ptr + s);
        n = __ldg(p.row_ptr + s + 1) - r0;
    }
    {
        int bad = (sl < 0 || sl >= p.n_slots) ? GDN_DERR_SLOT : 0;
        if (MODE != kStep && (r0 < 0 || n < 0 || n > kMaxRows || r0 > p.n_rows - n)) bad |= GDN_DERR_ROWS;
        if (bad || n == 0) {   // uniform over the CTA and over its cluster (same stream)
            if (bad && h == 0 && tid == 0) raise_error(p.err, bad);
            cp_async_wait_all();   // no copy may land after the CTA has left
            return;
        }
    }

    // The committed state tile goes to registers; the loads stay in flight
    // while the conv inputs are staged and processed.
    float *slot_tile = p.state + ((size_t)sl * p.Hv + h) * tile;
    if (!early) load_tile<D, RPW, CPL>(S, slot_tile + (size_t)row0 * D, warp, lane);

    // Stage the committed tail and the window's rows (this head's q, k and v
    // channels) and the z rows into shared memory.  d >= 64: seven TMA box
    // loads issued by one thread onto one mbarrier (per part a [3][D] box of
    // the tail and a [box_rows][D] box of the rows, and a [box_rows][D] box
    // of z; box rows past the window are other streams' rows or zeros, and
    // are never read).  d = 32: 16-byte cp.async.
    const uint16_t *tail = p.tail + (size_t)sl * 3 * CH;
    if constexpr (TMA) {
        if (tid == 0) {
            stage_fail = 0;
            tc::mbar_init(&stage_bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            tc::fence_async_smem();
            tc::mbar_expect_tx(&stage_bar, (uint32_t)((3 * (3 + p.box_rows) + p.box_rows) * D * 2));
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                const int c = channel_of<D>(part, 0, p.Hk, kh, h);
                tc::tma_load_2d(&sm.u.xin[part][0][0], &p.map_tail, c, sl * 3, &stage_bar);
                tc::tma_load_2d(&sm.u.xin[part][3][0], &p.map_mixed, c, r0, &stage_bar);
            }
            tc::tma_load_3d(&sm.z[0][0], &p.map_z, 0, h, r0, &stage_bar);
        }
    } else {
        for (int i = early ? 3 * CHUNKS + tid : tid; i < (n + 3) * CHUNKS; i += kRowThreads) {   // (early: tail staged)
            const int row = i / CHUNKS, ch = i - row * CHUNKS;
            const int part = ch / SEG, off = (ch - part * SEG) * 8;
            const int c = channel_of<D>(part, off, p.Hk, kh, h);
            const uint16_t *src = row < 3 ? tail + (size_t)row * CH + c : p.mixed + (size_t)(r0 + row - 3) * CH + c;
            cp_async16(&sm.u.xin[part][row][off], src);
        }
        for (int i = tid; i < n * SEG; i += kRowThreads) {
            const int t = i / SEG, ch = i - t * SEG;
            cp_async16(&sm.z[t][ch * 8], p.z + ((size_t)(r0 + t) * p.Hv + h) * D + ch * 8);
        }
    }
    if (TREE && tid < n) sm.parent[tid] = __ldg(p.parent + r0 + tid);
    // ---- a4: gates
    if (tid == 0) sm.bad = 0;
    if (MODE == kStep && tid == 0) {   // the row follows the slot: its taps are the tail's rows 2, 1, 0
        sm.parent[0] = -1;
        sm.reused[0] = 0;
        sm.order[0] = 0;
        sm.anc[0][0] = -1;
        sm.anc[0][1] = -2;
        sm.anc[0][2] = -3;
    }
    // A step's gates are computed by the last thread while warps 0-2 convert
    // the row (its a and b are loaded here, beside the row's inputs); the
    // rows of a window or tree are computed here, one thread each.
    constexpr int kGateThread = kRowThreads - 1;
    uint16_t step_a = 0, step_b = 0;
    if constexpr (MODE == kStep) {
        if (tid == kGateThread) {
            step_a = p.a[(size_t)r0 * p.Hv + h];
            step_b = p.b[(size_t)r0 * p.Hv + h];
        }
    } else if (tid < n) {
        sm.recidx[tid] = p.rec_slot ? __ldg(p.rec_slot + r0 + tid) : r0 + tid;
        const size_t gi = (size_t)(r0 + tid) * p.Hv + h;
        const float ain = bf_bits(p.a[gi]);
        const float bin = bf_bits(p.b[gi]);
        const float g = -__fmul_rn(expf(A_log), softplusf_rn(__fadd_rn(ain, dt_bias)));
        sm.decay[tid] = expf(g);
        sm.beta[tid] = sigmoidf_rn(bin);
    }
    cp_async_wait_all();
    __syncthreads();
    if constexpr (TMA) {
        // bounded: on a timeout the error word says so, the stream's outputs
        // are skipped, and the CTA still waits (bounded) for its copies
        // before it leaves
        if (!tc::mbar_wait(&stage_bar, 0, kRowWaitLimit)) {
            raise_error(p.err, GDN_DERR_TIMEOUT);
            tc::mbar_wait(&stage_bar, 0, kRowWaitLimit);
            stage_fail = 1;
        }
        __syncthreads();
        if (stage_fail) return;   // uniform: read after the barrier
    }

    // ---- each row's parent and conv ancestors along its branch -------------
    // (a step's one row follows the slot: set with its gates, below)
    if constexpr (MODE != kStep) {
        // Each row's thread checks its own parent and record entry ...
        if (tid < n) {
            const int par = TREE ? sm.parent[tid] : tid - 1;
            int bad = (par < -1 || par >= tid) ? GDN_DERR_PARENT : 0;
            // a pooled record must be a pool entry other than the stream's slot
            const int ri = sm.recidx[tid];
            if (p.rec_slot && (ri < 0 || ri >= p.n_slots || ri == sl)) bad |= GDN_DERR_SLOT;
            if (bad) atomicOr(&sm.bad, bad);
            sm.parent[tid] = par;
            sm.reused[tid] = 0;
            sm.order[tid] = tid;
        }
        __syncthreads();
        if (sm.bad) {   // uniform over the CTA and over its cluster (same stream)
            if (h == 0 && tid == 0) raise_error(p.err, sm.bad);
            return;
        }
        // ... then walks up to three parents for its conv ancestors
        if (tid < n) {
            int node = tid, tail_next = 2;
            for (int m = 0; m < 3; ++m) {
                if (node >= 0) node = sm.parent[node];
                if (node >= 0) {
                    sm.anc[tid][m] = node;
                } else {
                    sm.anc[tid][m] = tail_next - 3;
                    --tail_next;
                }
            }
        }
        if (TREE && warp == 0) {
            // Visit order: a tree depth first, children (and roots) in row order,
            // so that a node follows its parent wherever it can and the parent's
            // state is still in registers (only a node's later children reload
            // it).  Lane t < n takes node t: its ancestor-or-self set by walking
            // up, subtree sizes by ballot over those sets, and its preorder slot
            // = its depth + the subtree sizes of the earlier siblings of every
            // node on its root-to-node path.
            const bool live = lane < n;
            const int par = live ? sm.parent[lane] : -1;
            uint32_t anc = live ? (1u << lane) : 0u;
            for (int p_ = par, step = 0; step < kMaxRows; ++step) {
                const bool up = p_ >= 0;
                if (!__any_sync(kFull, up)) break;
                if (up) anc |= 1u << p_;
                const int pp = __shfl_sync(kFull, par, up ? p_ : 0);
                p_ = up ? pp : -1;
            }
            int nsub = 0;
            for (int b = 0; b < n; ++b) {
                const uint32_t m = __ballot_sync(kFull, live && ((anc >> b) & 1u));
                if (lane == b) nsub = __popc(m);
            }
            int before = 0;   // subtree sizes of the earlier siblings
            for (int q = 0; q < n; ++q) {
                const int pq = __shfl_sync(kFull, par, q), nq = __shfl_sync(kFull, nsub, q);
                if (live && q < lane && pq == par) before += nq;
            }
            int pre = __popc(anc) - 1;
            for (int a = 0; a < n; ++a) {
                const int ba = __shfl_sync(kFull, before, a);
                if ((anc >> a) & 1u) pre += ba;
            }
            if (live) sm.order[pre] = lane;
            __syncwarp();
            if (live && pre > 0 && par >= 0 && par != sm.order[pre - 1]) sm.reused[par] = 1;
            if constexpr (MODE == kTreeLog)
                if (live) path_mask[lane] = (int)anc;
        }
        __syncthreads();
    }

    if (MODE == kStep && tid == kGateThread) {   // (no conv item falls to this thread)
        const float g = -__fmul_rn(expf(A_log), softplusf_rn(__fadd_rn(bf_bits(step_a), dt_bias)));
        sm.decay[0] = expf(g);
        sm.beta[0] = sigmoidf_rn(bf_bits(step_b));
    }
    // ---- a2: conv over the branch's four taps, then SiLU (4 channels each) --
    static_assert(MODE != kStep || 3 * D / 4 <= kGateThread, "a step's conv items stop short of the gate thread");
    for (int i = tid; i < n * (3 * D / 4); i += kRowThreads) {
        const int t = i / (3 * D / 4);
        const int cc = (i - t * (3 * D / 4)) * 4;
        const int part = cc / D, e = cc - part * D;
        const uint4 *wp = reinterpret_cast<const uint4 *>(&sm.cw[cc][0]);
        const uint4 wa = wp[0], wb = wp[1];
        const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        // taps, oldest first: 3, 2 and 1 steps back along the branch, then the row
        const uint2 x0 = *reinterpret_cast<const uint2 *>(&sm.u.xin[part][3 + sm.anc[t][2]][e]);
        const uint2 x1 = *reinterpret_cast<const uint2 *>(&sm.u.xin[part][3 + sm.anc[t][1]][e]);
        const uint2 x2 = *reinterpret_cast<const uint2 *>(&sm.u.xin[part][3 + sm.anc[t][0]][e]);
        const uint2 x3 = *reinterpret_cast<const uint2 *>(&sm.u.xin[part][3 + t][e]);
        float *dst = part == 0 ? &sm.q[t][e] : (part == 1 ? &sm.k[t][e] : &sm.v[t][e]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int sh = (j & 1) * 16;
            const uint32_t a0 = (j < 2 ? x0.x : x0.y) >> sh, a1 = (j < 2 ? x1.x : x1.y) >> sh;
            const uint32_t a2 = (j < 2 ? x2.x : x2.y) >> sh, a3 = (j < 2 ? x3.x : x3.y) >> sh;
            float acc = __fmul_rn(bf_bits(wv[2 * j] & 0xffffu), bf_bits(a0 & 0xffffu));
            acc = __fmaf_rn(bf_bits(wv[2 * j] >> 16), bf_bits(a1 & 0xffffu), acc);
            acc = __fmaf_rn(bf_bits(wv[2 * j + 1] & 0xffffu), bf_bits(a2 & 0xffffu), acc);
            acc = __fmaf_rn(bf_bits(wv[2 * j + 1] >> 16), bf_bits(a3 & 0xffffu), acc);
            dst[j] = silu(acc);
        }
    }
    // ---- a6 (tail): the three newest inputs after each row, oldest first ----
    const int own_lo = lead ? 0 : 2 * SEG;   // chunks this CTA owns: v always, q/k if lead
    const int per_row = CHUNKS - own_lo;
    if (MODE != kStep && sli == 0) {   // slice 0 of a sliced window writes them
        for (int i = tid; i < n * 3 * per_row; i += kRowThreads) {
            const int t = i / (3 * per_row);
            const int rem = i - t * 3 * per_row;
            const int m = rem / per_row;
            const int ch = own_lo + rem - m * per_row;
            const int src_row = m == 2 ? 3 + t : 3 + sm.anc[t][1 - m];
            const int part = ch / SEG, off = (ch - part * SEG) * 8;
            const int c = channel_of<D>(part, off, p.Hk, kh, h);
            *reinterpret_cast<uint4 *>(p.rec_tail + ((size_t)sm.recidx[t] * 3 + m) * CH + c) =
                *reinterpret_cast<const uint4 *>(&sm.u.xin[part][src_row][off]);
        }
    }
    __syncthreads();

    // The in-place tail shift of a step: every CTA of the cluster (the key
    // head's value heads, and their row slices) must have staged the old tail
    // before the lead slices overwrite it.  Unsliced steps wait for that here;
    // sliced steps shift after the cluster barrier that gathers o, which every
    // slice reaches only after its staging.
    auto shift_tail = [&]() {
        for (int i = tid; i < (sli == 0 ? 3 * per_row : 0); i += kRowThreads) {   // slice 0 of each head
            const int m = i / per_row;
            const int ch = own_lo + i - m * per_row;
            const int part = ch / SEG, off = (ch - part * SEG) * 8;
            const int c = channel_of<D>(part, off, p.Hk, kh, h);
            *reinterpret_cast<uint4 *>(p.tail + ((size_t)sl * 3 + m) * CH + c) =
                *reinterpret_cast<const uint4 *>(&sm.u.xin[part][m + 1][off]);
        }
    };
    if (MODE == kStep && P == 1) {
        cluster_sync_all();
        shift_tail();
    }

    // ---- a3: L2 norm of q and k ------------------------------------------------
    for (int j = warp; j < 2 * n; j += kRowWarps) {
        float *x = (j & 1) ? sm.k[j >> 1] : sm.q[j >> 1];
        float xv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) xv[c] = x[lane * CPL + c];
        float ss = __fmul_rn(xv[0], xv[0]);
#pragma unroll
        for (int c = 1; c < CPL; ++c) ss = __fmaf_rn(xv[c], xv[c], ss);
        ss = warp_sum(ss);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss, p.eps_l2)));
        const float scale = (j & 1) ? 1.0f : p.q_scale;
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[lane * CPL + c] = __fmul_rn(__fmul_rn(xv[c], inv), scale);
    }
    __syncthreads();

    for (int t = warp; t < n; t += kRowWarps) {   // k . q of each row
        float acc = __fmul_rn(sm.k[t][lane * CPL], sm.q[t][lane * CPL]);
#pragma unroll
        for (int c = 1; c < CPL; ++c) acc = __fmaf_rn(sm.k[t][lane * CPL + c], sm.q[t][lane * CPL + c], acc);
        acc = warp_sum(acc);
        if (lane == 0) sm.kq[t] = acc;
    }
    if (LOG) {   // the rows' decay (every head) and normalised key (lead head of the group)
        if (tid < n && sli == 0) p.log_a[(size_t)(r0 + tid) * p.Hv + h] = sm.decay[tid];
        if (lead && sli == 0)
            for (int i = tid; i < n * D; i += kRowThreads)
                p.log_k[((size_t)(r0 + i / D) * p.Hk + kh) * D + i % D] = sm.k[i / D][i % D];
    }
    __syncthreads();
    if constexpr (P > 1) cluster_wait();   // every slice has started: remote stores are safe

    // ---- a5 + a6: the recurrence, row by row; no CTA barrier inside --------
    const int vi = lane >> SHIFT;
    for (int j = 0; j < n; ++j) {
        const int t = TREE ? sm.order[j] : j;   // the row (node) in hand
        if (TREE && j > 0) {
            const int par = sm.parent[t];
            if (par != sm.order[j - 1]) {
                if constexpr (MODE == kTree) {
                    load_tile<D, RPW, CPL>(S, (par < 0 ? slot_tile : p.rec_state + ((size_t)sm.recidx[par] * p.Hv + h) * tile) +
                                                  (size_t)row0 * D,
                                           warp, lane);
                } else {
                    // the committed state, then the logged rows from the root
                    // down to the parent (ancestors have smaller indices, so
                    // ascending order is root first), each as in the forward
                    // pass:  S <- fma(u, k, a S)
                    load_tile<D, RPW, CPL>(S, slot_tile + (size_t)row0 * D, warp, lane);
                    if (par >= 0) {
                        __syncwarp();   // this warp's rows of u_rows, written in earlier iterations
                        const int mask = path_mask[par];
                        for (int m = 0; m <= par; ++m) {
                            if (!((mask >> m) & 1)) continue;
                            const float dm = sm.decay[m];
                            float km[CPL];
#pragma unroll
                            for (int c = 0; c < CPL; ++c) km[c] = sm.k[m][lane * CPL + c];
#pragma unroll
                            for (int r = 0; r < RPW; ++r) {
                                const float ur = u_rows[m][warp * RPW + r];
#pragma unroll
                                for (int c = 0; c < CPL; ++c) S[r][c] = __fmaf_rn(ur, km[c], __fmul_rn(dm, S[r][c]));
                            }
                        }
                    }
                }
            }
        }
        float kk[CPL], qq[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            kk[c] = sm.k[t][lane * CPL + c];
            qq[c] = sm.q[t][lane * CPL + c];
        }
        float part[NV];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            float pk = __fmul_rn(S[r][0], kk[0]);
            float pq = __fmul_rn(S[r][0], qq[0]);
#pragma unroll
            for (int c = 1; c < CPL; ++c) {
                pk = __fmaf_rn(S[r][c], kk[c], pk);
                pq = __fmaf_rn(S[r][c], qq[c], pq);
            }
            part[r] = pk;
            part[RPW + r] = pq;
        }
        const float tot = reduce_scatter<NV>(part, lane);   // lanes < 16: S k; lanes >= 16: S q
        const float dec = sm.decay[t], bet = sm.beta[t];
        float u = 0.0f;
        if (lane < 16) u = __fmul_rn(bet, __fsub_rn(sm.v[t][row0 + warp * RPW + vi], __fmul_rn(dec, tot)));
        const float u_pair = __shfl_xor_sync(kFull, u, 16);
        if (lane >= 16 && (lane & ((1 << SHIFT) - 1)) == 0) {
            const int row = row0 + warp * RPW + vi - RPW;
            const float ov = __fmaf_rn(u_pair, sm.kq[t], __fmul_rn(dec, tot));
            if constexpr (P > 1 && !kPartials) {   // into every slice of this head (cluster ranks (h % G) * P + j)
#pragma unroll
                for (int j = 0; j < P; ++j)
                    st_cluster_f32(&o_all[MODE == kStep ? 0 : t][row], (uint32_t)(crank0 + j), ov);
            } else if constexpr (P > 1) {
                o_all[MODE == kStep ? 0 : t][row] = ov;
            } else {
                sm.u.o[t][row] = ov;
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float ur = __shfl_sync(kFull, u, r << SHIFT);
#pragma unroll
            for (int c = 0; c < CPL; ++c) S[r][c] = __fmaf_rn(ur, kk[c], __fmul_rn(dec, S[r][c]));
        }
        if (MODE == kWindow || MODE == kTree) {
            const bool streaming = !(MODE == kTree && sm.reused[t]);
            store_tile<D, RPW, CPL>(p.rec_state + ((size_t)sm.recidx[t] * p.Hv + h) * tile + (size_t)row0 * D, S, warp,
                                    lane, streaming);
        }
        if (LOG && lane < 16 && (lane & ((1 << SHIFT) - 1)) == 0) {
            p.log_u[((size_t)(r0 + t) * p.Hv + h) * D + row0 + warp * RPW + vi] = u;
            if constexpr (MODE == kTreeLog) u_rows[t][warp * RPW + vi] = u;
        }
    }
    if (MODE == kStep) store_tile<D, RPW, CPL>(slot_tile + (size_t)row0 * D, S, warp, lane, false);
    if constexpr (P > 1 && !kPartials) {
        cluster_sync_all();   // every slice's o rows have landed in every slice
        if (MODE == kStep) shift_tail();   // and every slice has staged the old tail long ago
    } else {
        __syncthreads();   // every warp's o rows are in shared memory
    }

    // ---- a7: gated RMSNorm, y in bf16 ----------------------------------------
    // Sum of o^2 over the row: lane l takes rows l*CPL .. l*CPL + CPL - 1,
    // then the xor butterfly 1, 2, 4, .., 16.  Two slices gather each
    // other's o rows and sum the whole row.  With more, a slice's rows are
    // the aligned lane group [row0 / CPL, (row0 + D/P) / CPL): each slice
    // sums its own group's levels, sends that partial to every slice of the
    // head, and all finish the remaining levels from the P partials in the
    // butterfly's pairwise order.  Either way the bits are the unsliced ones.
    constexpr int GL = 32 / P;   // lanes of one slice's rows
    auto lane_ss = [&](const float (&ov)[CPL]) {
        float ss = __fmul_rn(ov[0], ov[0]);
#pragma unroll
        for (int c = 1; c < CPL; ++c) ss = __fmaf_rn(ov[c], ov[c], ss);
        return ss;
    };
    if constexpr (P > 1 && kPartials) {
        for (int t = warp; t < n; t += kRowWarps) {
            const bool mine = lane / GL == sli;
            float ov[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) ov[c] = mine ? o_all[MODE == kStep ? 0 : t][lane * CPL + c] : 0.0f;
            float ss = lane_ss(ov);
#pragma unroll
            for (int off = 1; off < GL; off <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, off));
            if (lane == sli * GL) {   // into every slice of this head (cluster ranks (h % G) * P + j)
#pragma unroll
                for (int j = 0; j < P; ++j)
                    st_cluster_f32(&part_all[MODE == kStep ? 0 : t][sli], (uint32_t)(crank0 + j), ss);
            }
        }
        cluster_sync_all();   // every slice's partials have landed in every slice
        if (MODE == kStep) shift_tail();   // and every slice has staged the old tail long ago
    }
    for (int t = warp; t < n; t += kRowWarps) {
        float ov[CPL];
        float ss;
        if constexpr (P > 1 && !kPartials) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) ov[c] = o_all[MODE == kStep ? 0 : t][lane * CPL + c];
            ss = warp_sum_up(lane_ss(ov));
        } else if constexpr (P > 1) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) ov[c] = o_all[MODE == kStep ? 0 : t][lane * CPL + c];   // own rows only
            float v[P];
#pragma unroll
            for (int q = 0; q < P; ++q) v[q] = part_all[MODE == kStep ? 0 : t][q];
#pragma unroll
            for (int off = 1; off < P; off <<= 1) {
                float w[P];
#pragma unroll
                for (int q = 0; q < P; ++q) w[q] = __fadd_rn(v[q], v[q ^ off]);
#pragma unroll
                for (int q = 0; q < P; ++q) v[q] = w[q];
            }
            ss = v[0];
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) ov[c] = sm.u.o[t][lane * CPL + c];
            ss = warp_sum_up(lane_ss(ov));
        }
        // (the fast reciprocal square root: within a few ulp, far below the
        // output's bf16 rounding, and a short chain on the path to y)
        const float inv = rsqrtf(__fadd_rn(__fmul_rn(ss, 1.0f / D), p.eps_rms));
        const size_t base = ((size_t)(r0 + t) * p.Hv + h) * D + lane * CPL;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            if (P > 1 && (lane * CPL + c < row0 || lane * CPL + c >= row0 + D / P)) continue;   // another slice's
            const float zz = bf_bits(sm.z[t][lane * CPL + c]);
            const float wn = bf_bits(sm.nw[lane * CPL + c]);
            const float yv = __fmul_rn(__fmul_rn(__fmul_rn(ov[c], inv), wn), silu(zz));
            p.y[base + c] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
        }
    }
}

}  // namespace gdn
