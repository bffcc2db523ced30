// gdn_prefill.cuh -- chunked prompt prefill of the GDN layer (TensorFold
// #747, first note: the engine's "prompt chain" kernel; prompts that arrive
// together share one prefill pass).
//
// The recurrence S_t = a_t S_{t-1} + u_t k_t^T with u_t = b_t (v_t - a_t
// S_{t-1} k_t) is evaluated chunk by chunk (C rows).  Inside a chunk, with
// G_t = sum_{s<=t} log a_s, gamma_t = exp(G_t), Gamma_ts = exp(G_t - G_s):
//   A  = K K^T,  M = strict_lower(diag(b) (Gamma o A))
//   (I + M) W = diag(b gamma) K,   (I + M) U~ = diag(b) V   (forward substitution)
//   U  = U~ - W S0^T
//   O  = diag(gamma) Q S0^T + lower(Gamma o Q K^T) U
//   S  = gamma_C S0 + U^T diag(gamma_C / gamma) K
// which equals the row-by-row recurrence in exact arithmetic.
//
// Three kernels:
//   prep  (chunk x value head, all chunks in parallel): conv + SiLU, L2 norms,
//         gates, A, Q K^T, the forward substitution; writes the chunk's
//         Q~ = diag(gamma) Q, K~ = diag(gamma_C / gamma) K, W, U~,
//         P = lower(Gamma o Q K^T) and gamma_C to the workspace.
//   scan  (sequence x value head x d_v slice, chunks in order): U, O and the
//         state update; writes O (fp32) to the workspace, and the final state
//         and conv tail to the slot.
//   norm  (token x value head): gated RMSNorm of O, y in bf16.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

struct PrefillParams {
    int Hk, Hv, G, CH;
    float q_scale, eps_l2, eps_rms;
    const uint16_t *conv_w;
    const float *A_log;
    const float *dt_bias;
    const uint16_t *norm_w;
    float *state;
    uint16_t *tail;
    int n_slots;
    const uint16_t *mixed;   // bf16 [T, CH]
    const uint16_t *z;       // bf16 [T, Hv, D]
    const uint16_t *a;       // bf16 [T, Hv]
    const uint16_t *b;       // bf16 [T, Hv]
    uint16_t *y;             // bf16 [T, Hv, D]
    const int *slot;         // [S]
    const int *cu_seqlens;   // [S + 1]
    int n_seqs, n_tokens, max_chunks;
    float *ws_chunks;        // [max_chunks, Hv, chunk block]
    float *ws_out;           // [T, Hv, D] fp32 O
    int *err;
};

constexpr int kPrefillChunk = 64;
constexpr int kPrepThreads = 256;
constexpr int kNormThreads = 256;

// Floats of one (chunk, head) block of the workspace.
template <int D, int C>
struct ChunkBlock {
    static constexpr int kQ = 0;              // Q~ [C][D]
    static constexpr int kK = C * D;          // K~ [C][D]
    static constexpr int kW = 2 * C * D;      // W  [C][D]
    static constexpr int kU = 3 * C * D;      // U~ [C][D]
    static constexpr int kP = 4 * C * D;      // P  [C][C]
    static constexpr int kMisc = 4 * C * D + C * C;   // gamma_C, pad
    static constexpr int kFloats = kMisc + 4;
};

// Locate global chunk gc: its sequence, first token, rows, and the
// sequence's first token.  Returns false past the last chunk or on bad
// cu_seqlens (bad = 1).
__device__ __forceinline__ bool locate_chunk(const PrefillParams &p, int C, int gc, int &seq, int &start, int &n,
                                             int &seq_start, int &bad) {
    int base = 0;
    bad = 0;
    for (int s = 0; s < p.n_seqs; ++s) {
        const int lo = __ldg(p.cu_seqlens + s), hi = __ldg(p.cu_seqlens + s + 1);
        if (lo < 0 || hi < lo || hi > p.n_tokens) {
            bad = 1;
            return false;
        }
        const int nc = (hi - lo + C - 1) / C;
        if (gc < base + nc) {
            seq = s;
            seq_start = lo;
            start = lo + (gc - base) * C;
            n = min(C, hi - start);
            return true;
        }
        base += nc;
    }
    return false;
}

// First global chunk of sequence s (chunks are numbered sequence by
// sequence), or -1 if cu_seqlens[0..s+1] is not a non-decreasing list in
// [0, n_tokens].
__device__ __forceinline__ int chunk_base(const PrefillParams &p, int C, int s) {
    int base = 0;
    for (int i = 0; i <= s; ++i) {
        const int lo = __ldg(p.cu_seqlens + i), hi = __ldg(p.cu_seqlens + i + 1);
        if (lo < 0 || hi < lo || hi > p.n_tokens) return -1;
        if (i < s) base += (hi - lo + C - 1) / C;
    }
    return base;
}

template <int D>
__device__ __forceinline__ int pchannel(int part, int e, int Hk, int kh, int h) {
    return part == 0 ? kh * D + e : (part == 1 ? (Hk + kh) * D + e : 2 * Hk * D + h * D + e);
}

// ---------------------------------------------------------------------------
// prep: one CTA per (value head, global chunk)
// ---------------------------------------------------------------------------
template <int D, int C>
struct PrepSmem {
    static constexpr int LD = D + 4;                    // padded fp32 row
    static constexpr int kQ = 0;                        // q [C][LD]
    static constexpr int kK = C * LD;                   // k [C][LD]
    static constexpr int kV = 2 * C * LD;               // v [C][LD]
    static constexpr int kScratch = 3 * C * LD;         // xin (bf16) then A, QK
    static constexpr int kXinFloats = ((C + 3) * 3 * D * 2 + 15) / 16 * 4;
    static constexpr int AS = C + 4;                    // padded row of A / QK (16-byte aligned)
    static constexpr int kAQK = 2 * C * AS;             // A [C][AS], QK [C][AS]
    static constexpr int kScratchFloats = kXinFloats > kAQK ? kXinFloats : kAQK;
    static constexpr int kVec = kScratch + kScratchFloats;   // g, beta, G, eG, eGC [C] each
    static constexpr int kFloats = kVec + 5 * C + 4;
    static constexpr size_t kBytes = (size_t)kFloats * 4;
};

template <int D, int C>
__global__ void __launch_bounds__(kPrepThreads, 1) gdn_prefill_prep_kernel(const PrefillParams p) {
    using L = PrepSmem<D, C>;
    using B = ChunkBlock<D, C>;
    constexpr int LD = L::LD;
    extern __shared__ __align__(16) float smem[];
    float *q = smem + L::kQ, *k = smem + L::kK, *v = smem + L::kV;
    uint16_t *xin = reinterpret_cast<uint16_t *>(smem + L::kScratch);   // [C+3][3D]
    constexpr int AS = L::AS;
    float *A = smem + L::kScratch;                                     // [C][AS] after the conv
    float *QK = A + C * AS;
    float *g = smem + L::kVec, *beta = g + C, *Gc = beta + C, *eG = Gc + C, *eGC = eG + C;
    __shared__ int info[5];

    const int h = blockIdx.x, gc = blockIdx.y, tid = threadIdx.x;
    const int kh = h / p.G;
    const size_t CH = (size_t)p.CH;
    if (tid == 0) {
        int seq = -1, start = 0, n = 0, seq_start = 0, bad = 0;
        const bool ok = locate_chunk(p, C, gc, seq, start, n, seq_start, bad);
        int sl = ok ? __ldg(p.slot + seq) : -1;
        if (ok && (sl < 0 || sl >= p.n_slots)) bad |= 2;
        if (bad && h == 0) raise_error(p.err, (bad & 1 ? GDN_DERR_SEQLENS : 0) | (bad & 2 ? GDN_DERR_SLOT : 0));
        info[0] = (ok && !bad) ? n : 0;
        info[1] = start;
        info[2] = seq_start;
        info[3] = sl;
    }
    __syncthreads();
    const int n = info[0], start = info[1], seq_start = info[2], sl = info[3];
    if (n == 0) return;

    // stage the conv inputs: rows start-3 .. start+n-1 (before the sequence:
    // the slot's kept tail), this head's q | k | v channels
    constexpr int SEG = D * 2 / 16, CHUNKS = 3 * SEG;
    for (int i = tid; i < (n + 3) * CHUNKS; i += kPrepThreads) {
        const int row = i / CHUNKS, ch = i - row * CHUNKS;
        const int part = ch / SEG, off = (ch - part * SEG) * 8;
        const int c = pchannel<D>(part, off, p.Hk, kh, h);
        const int tok = start - 3 + row;
        const uint16_t *src = tok >= seq_start ? p.mixed + (size_t)tok * CH + c
                                               : p.tail + ((size_t)sl * 3 + (3 - (seq_start - tok))) * CH + c;
        *reinterpret_cast<uint4 *>(xin + (size_t)row * 3 * D + part * D + off) = __ldg(reinterpret_cast<const uint4 *>(src));
    }
    __syncthreads();

    // conv + SiLU (rows >= n are zero)
    for (int i = tid; i < C * 3 * D; i += kPrepThreads) {
        const int t = i / (3 * D), cc = i - t * 3 * D;
        const int part = cc / D, e = cc - part * D;
        float act = 0.0f;
        if (t < n) {
            const int c = pchannel<D>(part, e, p.Hk, kh, h);
            const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + (size_t)c * 4));
            const uint16_t *x = xin + (size_t)t * 3 * D + cc;   // staged row t is 3 back from row t
            float acc = __fmul_rn(bf_bits(wv.x & 0xffffu), bf_bits(x[0]));
            acc = __fmaf_rn(bf_bits(wv.x >> 16), bf_bits(x[3 * D]), acc);
            acc = __fmaf_rn(bf_bits(wv.y & 0xffffu), bf_bits(x[6 * D]), acc);
            acc = __fmaf_rn(bf_bits(wv.y >> 16), bf_bits(x[9 * D]), acc);
            act = silu(acc);
        }
        float *dst = part == 0 ? q : (part == 1 ? k : v);
        dst[t * LD + e] = act;
    }
    __syncthreads();

    // L2 norms of q and k (one warp per vector), gates, chunk-local log decay
    const int lane = tid & 31, warp = tid >> 5;
    constexpr int CPL = D / 32;
    for (int j = warp; j < 2 * n; j += kPrepThreads / 32) {
        float *x = (j & 1) ? k + (j >> 1) * LD : q + (j >> 1) * LD;
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
    if (tid < C) {
        float gg = 0.0f, bb = 0.0f;
        if (tid < n) {
            const size_t gi = (size_t)(start + tid) * p.Hv + h;
            gg = -__fmul_rn(expf(p.A_log[h]), softplusf_rn(__fadd_rn(bf_bits(p.a[gi]), p.dt_bias[h])));
            bb = sigmoidf_rn(bf_bits(p.b[gi]));
        }
        g[tid] = gg;
        beta[tid] = bb;
    }
    __syncthreads();
    if (tid == 0) {
        float run = 0.0f;
        for (int t = 0; t < C; ++t) {
            run = __fadd_rn(run, g[t]);
            Gc[t] = run;
        }
    }
    __syncthreads();

    // A = K K^T and Q K^T: each thread owns rows t = ti + 16 r and columns
    // s = si + 16 c (r, c < 4), so the 8 threads of a 128-bit load phase read
    // 8 consecutive padded rows (distinct banks)
    {
        const int ti = tid / (C / 4), si = tid % (C / 4);
        float accA[4][4] = {}, accQ[4][4] = {};
        for (int j = 0; j < D; j += 4) {
            float4 kt[4], ks[4], qt[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                kt[r] = *reinterpret_cast<const float4 *>(k + (ti + 16 * r) * LD + j);
                qt[r] = *reinterpret_cast<const float4 *>(q + (ti + 16 * r) * LD + j);
                ks[r] = *reinterpret_cast<const float4 *>(k + (si + 16 * r) * LD + j);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    accA[r][c] = __fmaf_rn(kt[r].x, ks[c].x, accA[r][c]);
                    accA[r][c] = __fmaf_rn(kt[r].y, ks[c].y, accA[r][c]);
                    accA[r][c] = __fmaf_rn(kt[r].z, ks[c].z, accA[r][c]);
                    accA[r][c] = __fmaf_rn(kt[r].w, ks[c].w, accA[r][c]);
                    accQ[r][c] = __fmaf_rn(qt[r].x, ks[c].x, accQ[r][c]);
                    accQ[r][c] = __fmaf_rn(qt[r].y, ks[c].y, accQ[r][c]);
                    accQ[r][c] = __fmaf_rn(qt[r].z, ks[c].z, accQ[r][c]);
                    accQ[r][c] = __fmaf_rn(qt[r].w, ks[c].w, accQ[r][c]);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                A[(ti + 16 * r) * AS + si + 16 * c] = accA[r][c];
                QK[(ti + 16 * r) * AS + si + 16 * c] = accQ[r][c];
            }
    }
    if (tid < C) {   // per-row exponentials of the chunk-local log decay
        eG[tid] = expf(Gc[tid]);
        eGC[tid] = expf(__fsub_rn(Gc[n - 1], Gc[tid]));
    }
    __syncthreads();

    // M = strict_lower(diag(b) Gamma o A) in place of A; P = lower(Gamma o QK) to the workspace
    float *blk = p.ws_chunks + ((size_t)gc * p.Hv + h) * B::kFloats;
    for (int i = tid; i < C * C; i += kPrepThreads) {
        const int t = i / C, s = i - t * C;
        const bool live = t < n && s < n;
        const float gam = live ? expf(__fsub_rn(Gc[t], Gc[s])) : 0.0f;
        A[t * AS + s] = (live && s < t) ? __fmul_rn(__fmul_rn(beta[t], gam), A[t * AS + s]) : 0.0f;
        blk[B::kP + i] = (live && s <= t) ? __fmul_rn(gam, QK[t * AS + s]) : 0.0f;
    }
    __syncthreads();

    // Forward substitution (I + M) X = Y, one column per thread, in blocks of
    // 16 rows: first the rows' sums over all earlier blocks (16 independent
    // accumulators), then the 16 x 16 triangular block itself.
    if (tid < 2 * D) {
        const bool isW = tid < D;
        const int col = isW ? tid : tid - D;
        float X[C];
#pragma unroll
        for (int b0 = 0; b0 < C; b0 += 16) {
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = b0 + i;
                acc[i] = isW ? __fmul_rn(__fmul_rn(beta[t], eG[t]), k[t * LD + col])
                             : __fmul_rn(beta[t], v[t * LD + col]);
            }
#pragma unroll
            for (int s4 = 0; s4 < b0; s4 += 4)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(A + (b0 + i) * AS + s4);
                    acc[i] = __fmaf_rn(-m4.x, X[s4], acc[i]);
                    acc[i] = __fmaf_rn(-m4.y, X[s4 + 1], acc[i]);
                    acc[i] = __fmaf_rn(-m4.z, X[s4 + 2], acc[i]);
                    acc[i] = __fmaf_rn(-m4.w, X[s4 + 3], acc[i]);
                }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
#pragma unroll
                for (int j = 0; j < i; ++j) acc[i] = __fmaf_rn(-A[(b0 + i) * AS + b0 + j], X[b0 + j], acc[i]);
                X[b0 + i] = acc[i];
            }
        }
        float *dst = blk + (isW ? B::kW : B::kU);
#pragma unroll
        for (int t = 0; t < C; ++t) dst[t * D + col] = X[t];
    }
    // Q~ = diag(gamma) Q, K~ = diag(gamma_C / gamma) K, gamma_C
    for (int i = tid; i < C * D / 4; i += kPrepThreads) {
        const int t = i / (D / 4), e = (i - t * (D / 4)) * 4;
        const bool live = t < n;
        const float4 q4 = *reinterpret_cast<const float4 *>(q + t * LD + e);
        const float4 k4 = *reinterpret_cast<const float4 *>(k + t * LD + e);
        const float a = live ? eG[t] : 0.0f, c = live ? eGC[t] : 0.0f;
        *reinterpret_cast<float4 *>(blk + B::kQ + t * D + e) =
            make_float4(__fmul_rn(a, q4.x), __fmul_rn(a, q4.y), __fmul_rn(a, q4.z), __fmul_rn(a, q4.w));
        *reinterpret_cast<float4 *>(blk + B::kK + t * D + e) =
            make_float4(__fmul_rn(c, k4.x), __fmul_rn(c, k4.y), __fmul_rn(c, k4.z), __fmul_rn(c, k4.w));
    }
    if (tid == 0) blk[B::kMisc] = eG[n - 1];
}

// ---------------------------------------------------------------------------
// scan: one CTA per (d_v slice, value head, sequence); chunks in order
// ---------------------------------------------------------------------------
template <int D, int C, int DS>
struct ScanSmem {
    static constexpr int LD = D + 4;
    static constexpr int LS = DS + 4;
    static constexpr int kQ = 0;                 // Q~ [C][LD]
    static constexpr int kK = C * LD;            // K~ [C][LD]
    static constexpr int kW = 2 * C * LD;        // W  [C][LD]
    static constexpr int kUt = 3 * C * LD;       // U~ slice [C][LS]
    static constexpr int kP = kUt + C * LS;      // P [C][C+4]
    static constexpr int kS = kP + C * (C + 4);  // S slice [DS][LD]
    static constexpr int kU = kS + DS * LD;      // U [C][LS]
    static constexpr int kFloats = kU + C * LS + 4;
    static constexpr size_t kBytes = (size_t)kFloats * 4;
};

template <int D, int C, int DS, int NT>
__global__ void __launch_bounds__(NT, 1) gdn_prefill_scan_kernel(const PrefillParams p) {
    using L = ScanSmem<D, C, DS>;
    using B = ChunkBlock<D, C>;
    constexpr int LD = L::LD, LS = L::LS;
    extern __shared__ __align__(16) float smem[];
    float *Qs = smem + L::kQ, *Ks = smem + L::kK, *Ws = smem + L::kW, *Uts = smem + L::kUt;
    float *Ps = smem + L::kP, *Ss = smem + L::kS, *Us = smem + L::kU;
    float *gam_s = Us + C * LS;

    const int js = blockIdx.x, h = blockIdx.y, s = blockIdx.z, tid = threadIdx.x;
    const int i0 = js * DS;   // first state row of this slice
    const int base = chunk_base(p, C, s);
    if (base < 0) {
        if (js == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DERR_SEQLENS);
        return;
    }
    const int lo = __ldg(p.cu_seqlens + s), hi = __ldg(p.cu_seqlens + s + 1);
    const int L_s = hi - lo;
    if (L_s == 0) return;
    const int sl = __ldg(p.slot + s);
    if (sl < 0 || sl >= p.n_slots) {
        if (js == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DERR_SLOT);
        return;
    }
    const int n_chunks = (L_s + C - 1) / C;

    float *slot_tile = p.state + ((size_t)sl * p.Hv + h) * D * D + (size_t)i0 * D;
    for (int i = tid; i < DS * D / 4; i += NT) {
        const int r = i / (D / 4), c4 = i - r * (D / 4);
        *reinterpret_cast<float4 *>(Ss + r * LD + c4 * 4) = reinterpret_cast<const float4 *>(slot_tile + r * D)[c4];
    }

    // thread tiles: U and O ([C][DS]) as 4 rows x IC slice columns; the
    // state update as SR rows x 4 columns
    constexpr int TT = C / 4;                // row groups of 4
    constexpr int IC = DS * TT / NT;         // slice columns per thread in U / O
    static_assert(IC >= 1 && IC * NT == DS * TT, "scan tiling");
    constexpr int SR = DS * D / (NT * 4);    // state rows per thread in the update
    static_assert(SR >= 1 && SR * NT * 4 == DS * D, "scan tiling");

    for (int c = 0; c < n_chunks; ++c) {
        const int start = lo + c * C;
        const int n = min(C, hi - start);
        const float *blk = p.ws_chunks + ((size_t)(base + c) * p.Hv + h) * B::kFloats;
        __syncthreads();   // the previous chunk's smem readers are done
        for (int i = tid; i < C * D / 4; i += NT) {
            const int t = i / (D / 4), c4 = (i - t * (D / 4)) * 4;
            cp_async16(Qs + t * LD + c4, blk + B::kQ + t * D + c4);
            cp_async16(Ks + t * LD + c4, blk + B::kK + t * D + c4);
            cp_async16(Ws + t * LD + c4, blk + B::kW + t * D + c4);
        }
        for (int i = tid; i < C * DS / 4; i += NT) {
            const int t = i / (DS / 4), c4 = (i - t * (DS / 4)) * 4;
            cp_async16(Uts + t * LS + c4, blk + B::kU + t * D + i0 + c4);
        }
        for (int i = tid; i < C * C / 4; i += NT) {
            const int t = i / (C / 4), c4 = (i - t * (C / 4)) * 4;
            cp_async16(Ps + t * (C + 4) + c4, blk + B::kP + t * C + c4);
        }
        if (tid == 0) gam_s[0] = blk[B::kMisc];
        cp_async_wait_all();
        if (c + 1 < n_chunks) {   // pull the next chunk's block toward L2 while this one computes
            const char *nxt = reinterpret_cast<const char *>(blk + (size_t)p.Hv * B::kFloats);
            for (int off = tid * 128; off < B::kFloats * 4; off += NT * 128) prefetch_l2(nxt + off);
        }
        __syncthreads();

        // U = U~ - W S0^T and O = Q~ S0^T: thread owns rows t = tg + 16 r
        // (r < 4: the 8 threads of a 128-bit phase read 8 consecutive padded
        // rows) and slice columns ic0 .. ic0 + IC - 1
        const int tg = tid % TT, icg = tid / TT;
        const int ic0 = icg * IC;
        float accU[4][IC], accO[4][IC];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int cI = 0; cI < IC; ++cI) {
                accU[r][cI] = 0.0f;
                accO[r][cI] = 0.0f;
            }
        for (int j = 0; j < D; j += 4) {
            float4 w4[4], q4[4], s4[IC];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                w4[r] = *reinterpret_cast<const float4 *>(Ws + (tg + TT * r) * LD + j);
                q4[r] = *reinterpret_cast<const float4 *>(Qs + (tg + TT * r) * LD + j);
            }
#pragma unroll
            for (int cI = 0; cI < IC; ++cI) s4[cI] = *reinterpret_cast<const float4 *>(Ss + (ic0 + cI) * LD + j);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cI = 0; cI < IC; ++cI) {
                    accU[r][cI] = __fmaf_rn(w4[r].x, s4[cI].x, accU[r][cI]);
                    accU[r][cI] = __fmaf_rn(w4[r].y, s4[cI].y, accU[r][cI]);
                    accU[r][cI] = __fmaf_rn(w4[r].z, s4[cI].z, accU[r][cI]);
                    accU[r][cI] = __fmaf_rn(w4[r].w, s4[cI].w, accU[r][cI]);
                    accO[r][cI] = __fmaf_rn(q4[r].x, s4[cI].x, accO[r][cI]);
                    accO[r][cI] = __fmaf_rn(q4[r].y, s4[cI].y, accO[r][cI]);
                    accO[r][cI] = __fmaf_rn(q4[r].z, s4[cI].z, accO[r][cI]);
                    accO[r][cI] = __fmaf_rn(q4[r].w, s4[cI].w, accO[r][cI]);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int cI = 0; cI < IC; ++cI)
                Us[(tg + TT * r) * LS + ic0 + cI] = __fsub_rn(Uts[(tg + TT * r) * LS + ic0 + cI], accU[r][cI]);
        __syncthreads();

        // O += P U (P is lower triangular), then O to the workspace
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = tg + TT * r;
            for (int s2 = 0; s2 <= t; ++s2) {
                const float pv = Ps[t * (C + 4) + s2];
#pragma unroll
                for (int cI = 0; cI < IC; ++cI) accO[r][cI] = __fmaf_rn(pv, Us[s2 * LS + ic0 + cI], accO[r][cI]);
            }
            if (t < n) {
                float *orow = p.ws_out + ((size_t)(start + t) * p.Hv + h) * D + i0 + ic0;
#pragma unroll
                for (int cI = 0; cI < IC; ++cI) orow[cI] = accO[r][cI];
            }
        }

        // S = gamma_C S0 + U^T K~ : thread owns SR state rows x 4 columns
        {
            const int cg = tid % (D / 4), rg = tid / (D / 4);
            const int jc = cg * 4, r0 = rg * SR;
            const float gC = gam_s[0];
            float accS[SR][4];
#pragma unroll
            for (int r = 0; r < SR; ++r) {
                const float4 s4 = *reinterpret_cast<const float4 *>(Ss + (r0 + r) * LD + jc);
                accS[r][0] = __fmul_rn(gC, s4.x);
                accS[r][1] = __fmul_rn(gC, s4.y);
                accS[r][2] = __fmul_rn(gC, s4.z);
                accS[r][3] = __fmul_rn(gC, s4.w);
            }
            for (int t = 0; t < C; ++t) {
                const float4 k4 = *reinterpret_cast<const float4 *>(Ks + t * LD + jc);
#pragma unroll
                for (int r = 0; r < SR; ++r) {
                    const float u = Us[t * LS + r0 + r];
                    accS[r][0] = __fmaf_rn(u, k4.x, accS[r][0]);
                    accS[r][1] = __fmaf_rn(u, k4.y, accS[r][1]);
                    accS[r][2] = __fmaf_rn(u, k4.z, accS[r][2]);
                    accS[r][3] = __fmaf_rn(u, k4.w, accS[r][3]);
                }
            }
            __syncthreads();   // every reader of S0 (U, O) is done
#pragma unroll
            for (int r = 0; r < SR; ++r)
                *reinterpret_cast<float4 *>(Ss + (r0 + r) * LD + jc) =
                    make_float4(accS[r][0], accS[r][1], accS[r][2], accS[r][3]);
        }
    }
    __syncthreads();
    for (int i = tid; i < DS * D / 4; i += NT) {
        const int r = i / (D / 4), c4 = i - r * (D / 4);
        reinterpret_cast<float4 *>(slot_tile + r * D)[c4] = *reinterpret_cast<const float4 *>(Ss + r * LD + c4 * 4);
    }

    // the slot's new conv tail: the sequence's last three inputs (older ones
    // come from the old tail when the prompt is shorter than three rows);
    // slice 0 of each head writes its v channels, the key group's lead head its q/k
    if (js == 0) {
        const int kh = h / p.G;
        const bool lead = (h % p.G) == 0;
        const size_t CH = (size_t)p.CH;
        for (int cc = tid; cc < 3 * D; cc += NT) {
            const int part = cc / D;
            if (part < 2 && !lead) continue;
            const int ch = pchannel<D>(part, cc - part * D, p.Hk, kh, h);
            uint16_t *tl = p.tail + (size_t)sl * 3 * CH + ch;
            uint16_t old[3] = {tl[0], tl[CH], tl[2 * CH]};
            uint16_t nw[3];
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const int pos = L_s - 3 + m;   // sequence-relative position
                nw[m] = pos >= 0 ? p.mixed[(size_t)(lo + pos) * CH + ch] : old[3 + pos];
            }
            tl[0] = nw[0];
            tl[CH] = nw[1];
            tl[2 * CH] = nw[2];
        }
    }
}

// ---------------------------------------------------------------------------
// norm: one warp per (token, value head): y = O / sqrt(mean O^2 + eps) * w * SiLU(z)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kNormThreads) gdn_prefill_norm_kernel(const PrefillParams p) {
    constexpr int CPL = D / 32;
    const int lane = threadIdx.x & 31;
    const size_t item = (size_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
    if (item >= (size_t)p.n_tokens * p.Hv) return;
    const float *o = p.ws_out + item * D + lane * CPL;
    float ov[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) ov[c] = o[c];
    float ss = __fmul_rn(ov[0], ov[0]);
#pragma unroll
    for (int c = 1; c < CPL; ++c) ss = __fmaf_rn(ov[c], ov[c], ss);
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / D), p.eps_rms)));
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const float zz = bf_bits(p.z[item * D + lane * CPL + c]);
        const float wn = bf_bits(p.norm_w[lane * CPL + c]);
        const float yv = __fmul_rn(__fmul_rn(__fmul_rn(ov[c], inv), wn), silu(zz));
        p.y[item * D + lane * CPL + c] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
    }
}

}  // namespace gdn
