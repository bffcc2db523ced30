// gdn_rows.cuh -- the GDN row kernel: one-row steps, chain windows and tree
// windows share this one template, so their arithmetic is the same code.
//
// Work decomposition (one CTA per (value head h, stream s); 8 warps):
//   warp w owns state rows i in [w*D/8, (w+1)*D/8) of the [D x D] fp32 tile,
//   lane l owns columns j in [l*D/32, (l+1)*D/32).  The tile stays in
//   registers for the whole window, so it crosses HBM once on the way in and
//   once per recorded row on the way out.
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

#include "gdn_common.cuh"

namespace gdn {

enum RowMode : int { kStep = 0, kWindow = 1, kTree = 2 };

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
    float *rec_state;         // [R, Hv, D, D]
    uint16_t *rec_tail;       // bf16 [R, 3, CH]
    int *err;                 // device error word
};

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kMaxRows = GDN_MAX_WINDOW;

template <int D>
struct RowSmem {
    float q[kMaxRows][D];
    float k[kMaxRows][D];
    float v[kMaxRows][D];
    float o[kMaxRows][D];
    float decay[kMaxRows];
    float beta[kMaxRows];
    float kq[kMaxRows];
    // conv ancestors m = 1, 2, 3 steps back along the branch: >= 0 is a
    // window-local row, e < 0 is row 3 + e of the committed tail
    int anc[kMaxRows][3];
    int parent[kMaxRows];
    int reused[kMaxRows];   // tree: re-read later by a non-adjacent child
    int slot, r0, n;
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

// Global conv channel of element e of part (0 = q, 1 = k, 2 = v) of value head h.
template <int D>
__device__ __forceinline__ int channel_of(int part, int e, int Hk, int kh, int h) {
    return part == 0 ? kh * D + e : (part == 1 ? (Hk + kh) * D + e : 2 * Hk * D + h * D + e);
}

template <int D, int MODE>
__global__ void __launch_bounds__(kRowThreads, 2) gdn_rows_kernel(const RowParams p) {
    constexpr int RPW = D / kRowWarps;            // state rows per warp
    constexpr int CPL = D / 32;                   // state columns per lane
    constexpr int NV = 2 * RPW;                   // partial sums per lane: S k and S q
    constexpr int SHIFT = 5 - Log2<NV>::value;    // lane l holds total (l >> SHIFT)
    static_assert(NV >= 2 && NV <= 32, "unsupported head width");

    __shared__ RowSmem<D> sm;
    const int h = blockIdx.x, s = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kh = h / p.G;
    const size_t CH = (size_t)p.CH;

    // ---- a1: the stream's rows, each row's parent and conv ancestors -------
    if (tid == 0) {
        int bad = 0;
        const int sl = p.slot[s];
        if (sl < 0 || sl >= p.n_slots) bad |= GDN_DERR_SLOT;
        int r0 = s, n = 1;
        if (MODE != kStep) {
            r0 = p.row_ptr[s];
            const int r1 = p.row_ptr[s + 1];
            n = r1 - r0;
            if (r0 < 0 || r1 > p.n_rows || n < 0 || n > kMaxRows) bad |= GDN_DERR_ROWS;
        }
        if (!bad) {
            for (int t = 0; t < n; ++t) {
                int par = t - 1;
                if (MODE == kTree) {
                    par = p.parent[r0 + t];
                    if (par < -1 || par >= t) {
                        bad |= GDN_DERR_PARENT;
                        break;
                    }
                }
                sm.parent[t] = par;
                sm.reused[t] = 0;
            }
        }
        if (!bad) {
            for (int t = 0; t < n; ++t) {
                int node = t, tail_next = 2;
                for (int m = 0; m < 3; ++m) {
                    if (node >= 0) node = sm.parent[node];
                    if (node >= 0) {
                        sm.anc[t][m] = node;
                    } else {
                        sm.anc[t][m] = tail_next - 3;
                        --tail_next;
                    }
                }
                if (MODE == kTree && sm.parent[t] >= 0 && sm.parent[t] != t - 1) sm.reused[sm.parent[t]] = 1;
            }
        }
        if (bad) {
            if (h == 0) raise_error(p.err, bad);
            n = 0;
        }
        sm.slot = sl;
        sm.r0 = r0;
        sm.n = n;
    }
    __syncthreads();
    const int n = sm.n;
    if (n == 0) return;   // uniform over the CTA and over its cluster (same stream)
    const int sl = sm.slot, r0 = sm.r0;
    const bool lead = (h % p.G) == 0;   // this CTA records the shared q/k tail channels
    const uint16_t *tail = p.tail + (size_t)sl * 3 * CH;

    // ---- a2: conv over the branch's four taps, then SiLU --------------------
    for (int idx = tid; idx < n * 3 * D; idx += kRowThreads) {
        const int t = idx / (3 * D);
        const int cc = idx - t * 3 * D;
        const int part = cc / D;
        const int e = cc - part * D;
        const int c = channel_of<D>(part, e, p.Hk, kh, h);
        uint16_t x[4];   // oldest first; x[3] is the row itself
        x[3] = p.mixed[(size_t)(r0 + t) * CH + c];
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const int an = sm.anc[t][m];
            x[2 - m] = an >= 0 ? p.mixed[(size_t)(r0 + an) * CH + c] : tail[(size_t)(3 + an) * CH + c];
        }
        const uint2 wv = *reinterpret_cast<const uint2 *>(p.conv_w + (size_t)c * 4);
        float acc = __fmul_rn(bf_bits(wv.x & 0xffffu), bf_bits(x[0]));
        acc = __fmaf_rn(bf_bits(wv.x >> 16), bf_bits(x[1]), acc);
        acc = __fmaf_rn(bf_bits(wv.y & 0xffffu), bf_bits(x[2]), acc);
        acc = __fmaf_rn(bf_bits(wv.y >> 16), bf_bits(x[3]), acc);
        const float act = silu(acc);
        if (part == 0) sm.q[t][e] = act;
        else if (part == 1) sm.k[t][e] = act;
        else sm.v[t][e] = act;
        if (MODE != kStep && (part == 2 || lead)) {   // a6: the row's tail
            uint16_t *rt = p.rec_tail + (size_t)(r0 + t) * 3 * CH + c;
            rt[0] = x[1];
            rt[CH] = x[2];
            rt[2 * CH] = x[3];
        }
    }
    __syncthreads();

    if (MODE == kStep) {
        // Every CTA of this key-head group has read the old tail; now shift it
        // in place: the lead CTA moves the shared q/k channels, each CTA its v.
        cluster_sync_all();
        for (int cc = tid; cc < 3 * D; cc += kRowThreads) {
            const int part = cc / D;
            if (part < 2 && !lead) continue;
            const int c = channel_of<D>(part, cc - part * D, p.Hk, kh, h);
            uint16_t *tl = p.tail + (size_t)sl * 3 * CH + c;
            const uint16_t t1 = tl[CH], t2 = tl[2 * CH];
            tl[0] = t1;
            tl[CH] = t2;
            tl[2 * CH] = p.mixed[(size_t)s * CH + c];
        }
    }

    // ---- a3: L2 norm of q and k; a4: gates ----------------------------------
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
    if (tid < n) {
        const size_t gi = (size_t)(r0 + tid) * p.Hv + h;
        const float ain = bf_bits(p.a[gi]);
        const float bin = bf_bits(p.b[gi]);
        const float g = -__fmul_rn(expf(p.A_log[h]), softplusf_rn(__fadd_rn(ain, p.dt_bias[h])));
        sm.decay[tid] = expf(g);
        sm.beta[tid] = sigmoidf_rn(bin);
    }

    // The committed state tile goes to registers while the norms finish.
    const size_t tile = (size_t)D * D;
    float *slot_tile = p.state + ((size_t)sl * p.Hv + h) * tile;
    float S[RPW][CPL];
    load_tile<D, RPW, CPL>(S, slot_tile, warp, lane);
    __syncthreads();

    for (int t = warp; t < n; t += kRowWarps) {   // k . q of each row
        float acc = __fmul_rn(sm.k[t][lane * CPL], sm.q[t][lane * CPL]);
#pragma unroll
        for (int c = 1; c < CPL; ++c) acc = __fmaf_rn(sm.k[t][lane * CPL + c], sm.q[t][lane * CPL + c], acc);
        acc = warp_sum(acc);
        if (lane == 0) sm.kq[t] = acc;
    }
    __syncthreads();

    // ---- a5 + a6: the recurrence, row by row; no CTA barrier inside --------
    const int vi = lane >> SHIFT;
    for (int t = 0; t < n; ++t) {
        if (MODE == kTree && t > 0) {
            const int par = sm.parent[t];
            if (par != t - 1)
                load_tile<D, RPW, CPL>(S, par < 0 ? slot_tile : p.rec_state + ((size_t)(r0 + par) * p.Hv + h) * tile,
                                       warp, lane);
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
        if (lane < 16) u = __fmul_rn(bet, __fsub_rn(sm.v[t][warp * RPW + vi], __fmul_rn(dec, tot)));
        const float u_pair = __shfl_xor_sync(kFull, u, 16);
        if (lane >= 16 && (lane & ((1 << SHIFT) - 1)) == 0)
            sm.o[t][warp * RPW + vi - RPW] = __fmaf_rn(u_pair, sm.kq[t], __fmul_rn(dec, tot));
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float ur = __shfl_sync(kFull, u, r << SHIFT);
#pragma unroll
            for (int c = 0; c < CPL; ++c) S[r][c] = __fmaf_rn(ur, kk[c], __fmul_rn(dec, S[r][c]));
        }
        if (MODE != kStep) {
            const bool streaming = !(MODE == kTree && sm.reused[t]);
            store_tile<D, RPW, CPL>(p.rec_state + ((size_t)(r0 + t) * p.Hv + h) * tile, S, warp, lane, streaming);
        }
    }
    if (MODE == kStep) store_tile<D, RPW, CPL>(slot_tile, S, warp, lane, false);
    __syncthreads();

    // ---- a7: gated RMSNorm, y in bf16 ----------------------------------------
    for (int t = warp; t < n; t += kRowWarps) {
        float ov[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) ov[c] = sm.o[t][lane * CPL + c];
        float ss = __fmul_rn(ov[0], ov[0]);
#pragma unroll
        for (int c = 1; c < CPL; ++c) ss = __fmaf_rn(ov[c], ov[c], ss);
        ss = warp_sum(ss);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / D), p.eps_rms)));
        const size_t base = ((size_t)(r0 + t) * p.Hv + h) * D + lane * CPL;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const float zz = bf_bits(p.z[base + c]);
            const float wn = bf_bits(p.norm_w[lane * CPL + c]);
            const float yv = __fmul_rn(__fmul_rn(__fmul_rn(ov[c], inv), wn), silu(zz));
            p.y[base + c] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
        }
    }
}

}  // namespace gdn
