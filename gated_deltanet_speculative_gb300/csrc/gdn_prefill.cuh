// gdn_prefill.cuh -- chunked prompt prefill of the GDN layer (TensorFold
// #747, first note: the engine has a kernel for prompts, and prompts that
// come in together are prefilled in one pass).
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
//   prep  (all chunks in parallel): conv + SiLU, L2 norms, gates, A, Q K^T,
//         the inverse T; writes each chunk's Q~ = diag(gamma) Q (d = 128:
//         Q once per key head, gamma_t per value head), K~ = diag(gamma_C /
//         gamma) K, W, U~, P = lower(Gamma o Q K^T) and gamma_C to the
//         workspace.  d = 128 (tensor cores): one CTA per
//         (key head, chunk) item serves the G value heads of the key head;
//         d = 32, 64 (CUDA cores): one CTA per (value head, chunk).
//   scan  (chunks in order): U, O and the state update; writes O (fp32) to
//         the workspace, and the final state and conv tail to the slot.
//         d = 128: one CTA per (value head, sequence), the state in TMEM;
//         d = 32, 64: one CTA per (value head, sequence, d_v slice).
//   norm  (token x value head): gated RMSNorm of O, y in bf16.
// For d = 128 the launcher runs them per chunk group on three streams (see
// gdn_prefill.cu).
#pragma once

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

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
    int c_lo, c_hi;          // global chunks [c_lo, c_hi) of this launch (tensor-core prep and scan)
    float *ws_chunks;        // [max_chunks, Hv, chunk block]
    float *ws_out;           // [T, Hv, D] fp32 O
    int *err;
};

constexpr int kPrefillChunk = 64;
constexpr uint32_t kPrepWaitLimit = 1u << 22;
constexpr int kPrepThreads = 256;
constexpr int kNormThreads = 256;
constexpr int kNormSplit = 4;   // norm CTAs per (value head, chunk)

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

// The same block as laid out for the tensor-core scan (d = 128, C = 64), in
// bytes.  bf16 operands are pre-split (x = hi + lo, both bf16) and stored in
// the K-major no-swizzle layout of gdn_tc.cuh, hi block then lo block.  Two
// stacked operands, so that each group of the scan is one wide product:
//   [-W; Q]     rows 0..63 -W (rows t), 64..127 Q (rows t), K = j (128):
//               B operand of [U^T | O1^T] = [U~^T | 0] + S0 [-W; Q]^T  (N = 128).
//               Q is the key head's, so only the block of the first value
//               head of a key head holds it; the scan takes it from there.
//   [P; K~^T]   rows 0..63 P (rows t, K = s), 64..191 K~^T (rows j, K = t),
//               K = 64:  B operand of [O2^T | S] += U^T [P; K~^T]^T  (N = 192)
//               and O = diag(gamma) O1 + O2
//   U~^T fp32 [128 i][64 t]           the group-1 accumulator's start
//   gamma_C, then gamma_t [64]
struct TcBlock {
    static constexpr int kWQ = 0;           // [-W; Q~] hi; lo at + kWQLo
    static constexpr int kWQLo = 32768;
    static constexpr int kPK = 65536;       // [P; K~^T] hi; lo at + kPKLo
    static constexpr int kPKLo = 24576;
    static constexpr int kGroup1 = 65536;   // bytes of [-W; Q~]
    static constexpr int kGroup2 = 49152;   // bytes of [P; K~^T]
    static constexpr int kOpBytes = 114688;
    static constexpr int kUt = 114688;
    static constexpr int kMisc = 147456;
    static constexpr int kGam = 147472;     // gamma_t, fp32 [64]
    static constexpr int kBytes = 147728;
    static constexpr int kHalf = 16384;     // bytes of rows 0..63 of a 128-row operand with K = 128
};

// Store 8 consecutive k (k0 multiple of 8) of row r of a K-major bf16
// operand (K columns), split x = hi + lo: hi into `hi_base`, lo into
// `lo_base`, one 16-byte write each.
__device__ __forceinline__ void store_split8(unsigned char *hi_base, unsigned char *lo_base, int r, int k0, int K,
                                             const float (&x)[8]) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) tc::split_bf16x2(x[2 * j], x[2 * j + 1], hw[j], lw[j]);
    const uint32_t off = tc::kmajor_offset(r, k0, K);
    *reinterpret_cast<uint4 *>(hi_base + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(lo_base + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

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

    // conv + SiLU, one channel per thread down the chunk with a sliding
    // window of the four taps (rows >= n are zero)
    for (int cc = tid; cc < 3 * D; cc += kPrepThreads) {
        const int part = cc / D, e = cc - part * D;
        const int c = pchannel<D>(part, e, p.Hk, kh, h);
        const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(p.conv_w + (size_t)c * 4));
        const float w0 = bf_bits(wv.x & 0xffffu), w1 = bf_bits(wv.x >> 16);
        const float w2 = bf_bits(wv.y & 0xffffu), w3 = bf_bits(wv.y >> 16);
        const uint16_t *x = xin + cc;   // staged row t + 3 is row t itself
        float x0 = bf_bits(x[0]), x1 = bf_bits(x[3 * D]), x2 = bf_bits(x[6 * D]);
        float *dst = (part == 0 ? q : (part == 1 ? k : v)) + e;
        for (int t = 0; t < C; ++t) {
            float act = 0.0f;
            if (t < n) {
                const float x3 = bf_bits(x[(size_t)(t + 3) * 3 * D]);
                float acc = __fmul_rn(w0, x0);
                acc = __fmaf_rn(w1, x1, acc);
                acc = __fmaf_rn(w2, x2, acc);
                acc = __fmaf_rn(w3, x3, acc);
                act = __fdividef(acc, 1.0f + __expf(-acc));   // SiLU; prefill matches steps to tolerance
                x0 = x1;
                x1 = x2;
                x2 = x3;
            }
            dst[t * LD] = act;
        }
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
    if (warp == 0) {   // inclusive prefix sum of the log decays, two rows per lane
        const float a0 = g[2 * lane], a1 = g[2 * lane + 1];
        float run = __fadd_rn(a0, a1);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(kFull, run, off);
            if (lane >= off) run = __fadd_rn(run, o);
        }
        const float excl = __shfl_up_sync(kFull, run, 1);
        const float before = lane == 0 ? 0.0f : excl;
        Gc[2 * lane] = __fadd_rn(before, a0);
        Gc[2 * lane + 1] = run;
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
        const float gam = live ? __expf(__fsub_rn(Gc[t], Gc[s])) : 0.0f;
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
// prep on the tensor cores (d = 128, C = 64): a persistent grid of CTAs of
// 512 threads, each taking (key head, global chunk) items of [c_lo, c_hi)
// in turn (the grid may be held below the SM count so that a concurrent
// scan finds free SMs).  An item writes the chunk block (TcBlock) of each
// of the G value heads that share the key head.
// Once per key head (item):
//   the gates of all G value heads (log decays, their prefix sums G_t,
//   gamma_t = exp(G_t), gamma_C / gamma_t, beta_t and the decays a_t);
//   conv + SiLU of the q and k channels (16-row pieces of one channel, no
//   per-row branches); L2 norms, eight rows per warp in one reduce-scatter;
//   MMA 1:  [K; Q] (128 x 128) * K^T -> K K^T and Q K^T, left in TMEM;
//   Q (shared by the value heads) out to the key head's first block, and
//   the K^T operand, the A operand of every head's W product.
// Then for each value head h of the group (its v inputs staged while the
// previous head is worked on):
//   conv + SiLU of h's v channels straight into (diag(b) V)^T (the first
//   head's while MMA 1 runs, each later one's beside the previous head's
//   stores);
//   M = strict_lower(diag(b) Gamma o A), P = lower(Gamma o Q K^T), formed
//   from the TMEM readout of MMA 1 with h's gates; along a row, Gamma is one
//   exponential per 16 columns and products with the decays a_s;
//   T = (I + M)^-1 on the CUDA cores (fp32): 16 x 16 diagonal blocks by
//   forward substitution, the rest by two levels of block doubling;
//   MMA 2:  K^T * T'^T -> W^T with T' = T diag(b gamma) (W = T diag(b gamma) K),
//           (diag(b) V)^T * T^T -> U~^T,
//   while K~^T = (diag(gamma_C / gamma) K)^T goes out for the scan; W and
//   U~^T leave TMEM into stages where T' and T were and go out from there.
// Every MMA operand is split into bf16 hi + lo and multiplied three times
// (hi hi + hi lo + lo hi), accumulating in fp32.
// ---------------------------------------------------------------------------
constexpr int kPrepTcThreads = 512;
constexpr int kPrepTcLD = 132;                 // fp32 row of q and k
// Shared memory (bytes):
constexpr int kPtQ = 0;                        // q fp32 [64][132], kept for every head
constexpr int kPtK = 33792;                    // k fp32 [64][132], kept for every head
constexpr int kPtR1 = 67584;                   // 65536: per head the (diag(b) V)^T operand and
                                               //   T' = T diag(b gamma)
                                               //   (at + 32768), then the W fp32 stage [64][128] in
                                               //   T''s place
constexpr int kPtR2 = kPtR1 + 65536;           // 66304: q | k conv inputs [67][256] bf16, then the
                                               //   [K; Q] operand hi | lo; then per head M, scratch,
                                               //   T fp32 [64][65] and the T operand
                                               //   (at + 49920), then the U~^T fp32 stage [128][64]
                                               //   in the place of T and its operand (at + 33280)
constexpr int kPtR3 = kPtR2 + 66304;           // 17152: v conv inputs [67][128] bf16 of one head
constexpr int kPrepMaxG = 8;                   // value heads per key head (the ABI's limit)
constexpr int kPtVec = kPtR3 + 17152;          // beta, G, eG, eGC, a [kPrepMaxG][64] each
constexpr int kPtCw = kPtVec + 5 * kPrepMaxG * 64 * 4;   // conv weights: q | k channels [256][4], then one head's v [128][4]
constexpr size_t kPrepTcSmem = kPtCw + 384 * 4 * 2;
static_assert(kPrepTcSmem <= 227 * 1024, "the prep's shared memory fits one CTA's opt-in limit");

template <int C>
__global__ void __launch_bounds__(kPrepTcThreads, 1) gdn_prefill_prep_tc_kernel(const PrefillParams p) {
    constexpr int D = 128, LD = kPrepTcLD, AS = C + 1;   // odd row stride: column walks across rows hit distinct banks
    static_assert(C == 64, "the tensor-core block layout is for C = 64");
    static_assert(kPrepTcThreads / 32 * 8 == 2 * C, "the norm step gives each warp eight of the 2C rows");
    static_assert(3 * C * AS * 4 + 16384 <= 66304 && 2 * C * AS * 4 + D * C * 4 <= 66304,
                  "region 2 holds M, scratch, T and the T operand, then the U~^T stage where T was");
    static_assert(32768 + C * D * 4 <= 65536, "region 1 holds the W stage where T' was");
    static_assert(2 * D * C * 2 <= 64 * kPrepTcLD * 4, "q's region holds the K^T operand");
    extern __shared__ __align__(1024) unsigned char psm[];
    float *q = reinterpret_cast<float *>(psm + kPtQ);
    float *k = reinterpret_cast<float *>(psm + kPtK);
    unsigned char *R1 = psm + kPtR1, *R2 = psm + kPtR2;
    uint16_t *xqk = reinterpret_cast<uint16_t *>(R2);           // [C+3][2D] q | k inputs
    uint16_t *xv = reinterpret_cast<uint16_t *>(psm + kPtR3);   // [C+3][D] v inputs of the head in hand
    unsigned char *kq_hi = R2, *kq_lo = R2 + 32768;             // [K; Q] operand (after the conv)
    unsigned char *kt_hi = psm + kPtQ, *kt_lo = kt_hi + 16384;  // K^T [D][C] in q's place, per item
    unsigned char *v_hi = R1, *v_lo = R1 + 16384;               // (b V)^T [D][C]
    unsigned char *tp_hi = R1 + 32768, *tp_lo = tp_hi + 8192;   // T' = T diag(b gamma) [C][C]
    float *A = reinterpret_cast<float *>(R2);                   // M [C][AS]
    float *QK = A + C * AS;                                     // level-2 scratch [C][AS]
    float *T = QK + C * AS;                                     // T [C][AS]
    unsigned char *t_hi = R2 + 49920, *t_lo = t_hi + 8192;      // T operand [C][C]
    // The W and U~^T stages take the places of T' and T, which MMA 2 reads
    // last: a head's W and U~^T leave from there while the next head's v conv
    // writes its operand (region 1's first half), with no barrier between.
    // Rows of 128 / 64 floats, 16-byte pieces XOR-swizzled
    // by the row (bits 2..4 of the column), so that the TMEM readout's
    // column writes and the row-wise reads of the stores both hit distinct
    // banks.
    float *Wf = reinterpret_cast<float *>(R1 + 32768);          // W [C][D]
    float *Uf = reinterpret_cast<float *>(R2 + 2 * C * AS * 4); // U~^T [D][C]
    auto swz = [](int row, int col) { return col ^ ((row & 7) << 2); };
    float *beta_all = reinterpret_cast<float *>(psm + kPtVec);      // [G][C], every head of the key head
    float *Gc_all = beta_all + kPrepMaxG * C;                        // log decays, then their prefix sums
    float *eG_all = Gc_all + kPrepMaxG * C;
    float *eGC_all = eG_all + kPrepMaxG * C;
    float *dec_all = eGC_all + kPrepMaxG * C;                        // per-row decays a_t = exp(g_t)
    uint16_t *cw_qk = reinterpret_cast<uint16_t *>(psm + kPtCw);   // [2D][4]
    uint16_t *cw_v = cw_qk + 2 * D * 4;                              // [D][4] of the head in hand
    __shared__ int info[4];
    __shared__ __align__(8) uint64_t bar_mma;
    __shared__ uint32_t tmem_base;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const size_t CH = (size_t)p.CH;
    if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        tc::mbar_init(&bar_mma, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    bool ok = true;
    uint32_t ph = 0;   // parity of the next bar_mma completion
    const int items = (p.c_hi - p.c_lo) * p.Hk;

#pragma unroll 1
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int kh = item % p.Hk, gc = p.c_lo + item / p.Hk;
    __syncthreads();   // every thread has read the previous item's info
    if (tid == 0) {
        int seq = -1, start = 0, n = 0, seq_start = 0, bad = 0;
        const bool found = locate_chunk(p, C, gc, seq, start, n, seq_start, bad);
        const int sl = found ? __ldg(p.slot + seq) : -1;
        if (found && (sl < 0 || sl >= p.n_slots)) bad |= 2;
        if (bad && kh == 0) raise_error(p.err, (bad & 1 ? GDN_DERR_SEQLENS : 0) | (bad & 2 ? GDN_DERR_SLOT : 0));
        info[0] = (found && !bad) ? n : 0;
        info[1] = start;
        info[2] = seq_start;
        info[3] = sl;
    }
    __syncthreads();
    const int n = info[0], start = info[1], seq_start = info[2], sl = info[3];
    if (n == 0) continue;   // uniform over the CTA

    // conv inputs: rows start-3 .. start+n-1 (the slot's kept tail before the
    // sequence), 16 bytes per copy
    auto src_of = [&](int row, int c) -> const uint16_t * {
        const int tok = start - 3 + row;
        return tok >= seq_start ? p.mixed + (size_t)tok * CH + c
                                : p.tail + ((size_t)sl * 3 + (3 - (seq_start - tok))) * CH + c;
    };
    auto stage_v = [&](int h) {   // head h's v channels into xv and their conv weights into cw_v
        for (int i = tid; i < (n + 3) * (D / 8); i += kPrepTcThreads) {
            const int row = i / (D / 8), off = (i - row * (D / 8)) * 8;
            cp_async16(xv + (size_t)row * D + off, src_of(row, pchannel<D>(2, off, p.Hk, kh, h)));
        }
        if (tid < D / 2) cp_async16(cw_v + tid * 8, p.conv_w + (size_t)pchannel<D>(2, tid * 2, p.Hk, kh, h) * 4);
    };
    for (int i = tid; i < (n + 3) * (2 * D / 8); i += kPrepTcThreads) {   // the key head's q | k channels
        const int row = i / (2 * D / 8), ch = i - row * (2 * D / 8);
        const int part = ch / (D / 8), off = (ch - part * (D / 8)) * 8;
        cp_async16(xqk + (size_t)row * 2 * D + part * D + off, src_of(row, pchannel<D>(part, off, p.Hk, kh, 0)));
    }
    if (tid < D) {   // q | k conv weights, two channels per copy
        const int part = tid / (D / 2), e0 = (tid - part * (D / 2)) * 2;
        cp_async16(cw_qk + (part * D + e0) * 4, p.conv_w + (size_t)pchannel<D>(part, e0, p.Hk, kh, 0) * 4);
    }
    stage_v(kh * p.G);
    // gates of every value head of the key head (rows >= n: beta = 0, log decay 0)
    for (int i = tid; i < p.G * C; i += kPrepTcThreads) {
        const int gi = i / C, t = i - gi * C, h = kh * p.G + gi;
        float gg = 0.0f, bb = 0.0f;
        if (t < n) {
            const size_t ai = (size_t)(start + t) * p.Hv + h;
            gg = -__fmul_rn(expf(p.A_log[h]), softplusf_rn(__fadd_rn(bf_bits(p.a[ai]), p.dt_bias[h])));
            bb = sigmoidf_rn(bf_bits(p.b[ai]));
        }
        Gc_all[gi * C + t] = gg;
        beta_all[gi * C + t] = bb;
        dec_all[gi * C + t] = expf(gg);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int gi = warp; gi < p.G; gi += kPrepTcThreads / 32) {   // inclusive prefix sums, two rows per lane
        float *Gc = Gc_all + gi * C;
        const float a0 = Gc[2 * lane], a1 = Gc[2 * lane + 1];
        float run = __fadd_rn(a0, a1);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(kFull, run, off);
            if (lane >= off) run = __fadd_rn(run, o);
        }
        const float excl = __shfl_up_sync(kFull, run, 1);
        Gc[2 * lane] = __fadd_rn(lane == 0 ? 0.0f : excl, a0);
        Gc[2 * lane + 1] = run;
    }

    // conv + SiLU of q and k: work item (16-row piece, channel), a sliding
    // window of the four taps down the piece.  Rows >= n read unstaged inputs
    // and are replaced by 0 with a select, so the 16 rows carry no branches.
    constexpr int PR = 16;
    auto conv_piece = [&](const uint16_t *x, int stride, const uint16_t *wsm, int t0, float (&act)[PR]) {
        const uint2 wv = *reinterpret_cast<const uint2 *>(wsm);
        const float w0 = bf_bits(wv.x & 0xffffu), w1 = bf_bits(wv.x >> 16);
        const float w2 = bf_bits(wv.y & 0xffffu), w3 = bf_bits(wv.y >> 16);
        float x0 = bf_bits(x[0]), x1 = bf_bits(x[stride]), x2 = bf_bits(x[2 * stride]);
#pragma unroll
        for (int r = 0; r < PR; ++r) {
            const float x3 = bf_bits(x[(size_t)(r + 3) * stride]);
            float acc = __fmul_rn(w0, x0);
            acc = __fmaf_rn(w1, x1, acc);
            acc = __fmaf_rn(w2, x2, acc);
            acc = __fmaf_rn(w3, x3, acc);
            const float sv = __fdividef(acc, 1.0f + __expf(-acc));   // SiLU; prefill matches steps to tolerance
            act[r] = t0 + r < n ? sv : 0.0f;
            x0 = x1;
            x1 = x2;
            x2 = x3;
        }
    };
    for (int it = tid; it < (C / PR) * 2 * D; it += kPrepTcThreads) {
        const int cc = it % (2 * D), t0 = (it / (2 * D)) * PR;   // warp-uniform part and t0
        const int part = cc / D, e = cc - part * D;
        float act[PR];
        conv_piece(xqk + (size_t)t0 * 2 * D + cc, 2 * D, cw_qk + cc * 4, t0, act);
        float *dst = (part == 0 ? q : k) + e;
#pragma unroll
        for (int r = 0; r < PR; ++r) dst[(t0 + r) * LD] = act[r];
    }
    for (int i = tid; i < p.G * C; i += kPrepTcThreads) {   // gamma and gamma_C / gamma of every head
        const int gi = i / C, t = i - gi * C;
        const float *Gc = Gc_all + gi * C;
        eG_all[i] = __expf(Gc[t]);
        eGC_all[i] = __expf(__fsub_rn(Gc[n - 1], Gc[t]));
    }
    __syncthreads();
    // L2 norms of q and k rows, q scaled: warp w takes rows 8w .. 8w+7 of the
    // interleaved list (q row j/2 for even j, k row j/2 for odd j); one
    // reduce-scatter leaves row 8w + (lane >> 2)'s sum of squares in lane
    // `lane`.  Rows >= n are zero and stay zero.
    {
        float4 xv4[8];
        float ss[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int j = warp * 8 + m;
            const float *x = (j & 1) ? k + (j >> 1) * LD : q + (j >> 1) * LD;
            xv4[m] = *reinterpret_cast<const float4 *>(x + lane * 4);
            float a2 = __fmul_rn(xv4[m].x, xv4[m].x);
            a2 = __fmaf_rn(xv4[m].y, xv4[m].y, a2);
            a2 = __fmaf_rn(xv4[m].z, xv4[m].z, a2);
            ss[m] = __fmaf_rn(xv4[m].w, xv4[m].w, a2);
        }
        const float tot = reduce_scatter<8>(ss, lane);
        const int jl = warp * 8 + (lane >> 2);
        const float mine = __fmul_rn(rsqrtf(__fadd_rn(tot, p.eps_l2)), (jl & 1) ? 1.0f : p.q_scale);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int j = warp * 8 + m;
            const float sc = __shfl_sync(kFull, mine, m * 4);
            float *x = (j & 1) ? k + (j >> 1) * LD : q + (j >> 1) * LD;
            *reinterpret_cast<float4 *>(x + lane * 4) = make_float4(__fmul_rn(xv4[m].x, sc), __fmul_rn(xv4[m].y, sc),
                                                                    __fmul_rn(xv4[m].z, sc), __fmul_rn(xv4[m].w, sc));
        }
    }
    __syncthreads();
    for (int it = tid; it < 2 * C * (D / 8); it += kPrepTcThreads) {   // [K; Q] rows r, 8 columns j
        const int r = it % (2 * C), j0 = (it / (2 * C)) * 8;
        const float *src = r < C ? k + r * LD + j0 : q + (r - C) * LD + j0;
        const float4 a4 = *reinterpret_cast<const float4 *>(src), b4 = *reinterpret_cast<const float4 *>(src + 4);
        const float x[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
        store_split8(kq_hi, kq_lo, r, j0, D, x);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // MMA 1: [A; QK] = [K; Q] K^T (TMEM columns 0..63), kept for every head
    if (tid == 0) {
        constexpr uint32_t idn = tc::idesc_bf16(128, C);
        const uint32_t ah = tc::smem_u32(kq_hi), al = tc::smem_u32(kq_lo);
        tc::mma_bf16<D>(tmem_base, ah, ah, idn, false);
        tc::mma_bf16<D>(tmem_base, ah, al, idn, true);
        tc::mma_bf16<D>(tmem_base, al, ah, idn, true);
        tc::mma_commit(&bar_mma);
    }
    {   // Q (rows 64..127 of the [K; Q] operand, hi and lo) into the block of the
        // key head's first value head, where the scan of every value head of
        // the key head takes it (rows >= n are zero)
        unsigned char *lead = reinterpret_cast<unsigned char *>(p.ws_chunks) +
                              ((size_t)gc * p.Hv + (size_t)kh * p.G) * TcBlock::kBytes;
        constexpr int V4 = TcBlock::kHalf / 16;   // 16-byte pieces of one half
        for (int it = tid; it < 2 * V4; it += kPrepTcThreads) {
            const int lo_part = it / V4, e = it - lo_part * V4;
            const unsigned char *src = (lo_part ? kq_lo : kq_hi) + TcBlock::kHalf;
            unsigned char *dst = lead + (lo_part ? TcBlock::kWQLo : 0) + TcBlock::kHalf;
            reinterpret_cast<float4 *>(dst)[e] = reinterpret_cast<const float4 *>(src)[e];
        }
    }
    // K^T (rows j, K = t) in q's place (q is not read again): the A operand
    // of every head's W^T product.  W = T diag(b gamma) K, so W^T = K^T T'^T
    // with T' = T diag(b gamma): only the 64 x 64 factor T' is per head.
    for (int it = tid; it < D * (C / 8); it += kPrepTcThreads) {   // rows j, 8 t
        const int j = it % D, t0 = (it / D) * 8;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = k[(t0 + e) * LD + j];
        store_split8(kt_hi, kt_lo, j, t0, C, x);
    }
    // (MMA 1 is waited for before the first head's M, P: its v conv and
    // operands, the Q copy and K^T overlap it)
    const int quarter = warp & 3, part = warp >> 2;   // 16 warps: lane quarter x column part

    // conv + SiLU of value head gi's v channels (staged in xv, weights in
    // cw_v) straight into the (diag(b) V)^T operand
    auto conv_v = [&](int gv, int first, int count) {   // on threads [first, first + count)
        const float *bv = beta_all + gv * C;
        for (int it = tid - first; it < (C / PR) * D; it += count) {
            const int e = it % D, t0 = (it / D) * PR;
            float act[PR];
            conv_piece(xv + (size_t)t0 * D + e, D, cw_v + e * 4, t0, act);
#pragma unroll
            for (int h8 = 0; h8 < PR; h8 += 8) {
                float vb[8];
#pragma unroll
                for (int e8 = 0; e8 < 8; ++e8) vb[e8] = __fmul_rn(bv[t0 + h8 + e8], act[h8 + e8]);
                store_split8(v_hi, v_lo, e, t0 + h8, C, vb);
            }
        }
    };
    conv_v(0, 0, kPrepTcThreads);
    ok = tc::mbar_wait(&bar_mma, ph, kPrepWaitLimit) && ok;   // MMA 1: [A; QK] in TMEM, region 2 free
    ph ^= 1;
    tc::fence_after_sync();

#pragma unroll 1
    for (int gi = 0; gi < p.G; ++gi) {
        const int h = kh * p.G + gi;
        unsigned char *blk = reinterpret_cast<unsigned char *>(p.ws_chunks) + ((size_t)gc * p.Hv + h) * TcBlock::kBytes;
        const float *beta = beta_all + gi * C, *Gc = Gc_all + gi * C, *eG = eG_all + gi * C, *eGC = eGC_all + gi * C;
        const float *dec = dec_all + gi * C;
        __syncthreads();   // xv and cw_v consumed; this head's v operand, the K^T operand and the
                           // previous head's W and U~^T stores are complete
        if (gi + 1 < p.G) stage_v(h + 1);   // in flight while this head is worked on
        {   // lane r holds row r of [A; QK]; the four warps on a lane quarter take
            // 16 columns each and form M = strict_lower(diag(b) Gamma o A) (into
            // shared memory) and P = lower(Gamma o QK) (split and written to the
            // chunk block from registers) with this head's gates.  Along a row,
            // Gamma[t][s] = exp(G_t - G_s) takes one exponential, at the last of
            // the 16 columns with s <= t; walking left, each next column is one
            // product with a decay, Gamma[t][s - 1] = Gamma[t][s] * a_s (every
            // factor is at most 1, so nothing overflows)
            const int r = quarter * 32 + lane;
            uint32_t v[16];
            tc::tmem_ld16_nowait(tmem_base + ((uint32_t)(quarter * 32) << 16) + part * 16, v);
            const bool isA = r < C;   // warp-uniform
            const int t = isA ? r : r - C;
            const int c0 = part * 16, top = min(t, c0 + 15);   // top < c0: the whole piece is masked
            const float Gt = Gc[t], bt = isA ? beta[t] : 1.0f;
            float gam = __expf(__fsub_rn(Gt, Gc[max(top, c0)]));
            tc::tmem_wait_ld();
            float x[2][8];
#pragma unroll
            for (int e = 15; e >= 0; --e) {
                const int sc = c0 + e;
                const bool keep = t < n && sc < n && (isA ? sc < t : sc <= t);
                x[e >> 3][e & 7] = keep ? __fmul_rn(__fmul_rn(bt, gam), __uint_as_float(v[e])) : 0.0f;
                if (sc <= top) gam = __fmul_rn(gam, dec[sc]);
            }
            if (isA) {
                float *dst = A + t * AS + part * 16;
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[e] = x[e >> 3][e & 7];
            } else {
                store_split8(blk + TcBlock::kPK, blk + TcBlock::kPK + TcBlock::kPKLo, t, part * 16, C, x[0]);
                store_split8(blk + TcBlock::kPK, blk + TcBlock::kPK + TcBlock::kPKLo, t, part * 16 + 8, C, x[1]);
            }
        }
        __syncthreads();
        // T = (I + M)^-1 by 16 x 16 blocks.  Threads < C solve the four diagonal
        // blocks (one column each), right-looking: once x_kk is final it is
        // folded into every later row, so each step is one FMA deep (the sums
        // run in the same order as a row-by-row substitution).
        if (tid < C) {
            const int b0 = (tid / 16) * 16, c = tid % 16;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.0f : 0.0f;
#pragma unroll
            for (int kk = 0; kk < 15; ++kk)
#pragma unroll
                for (int r = kk + 1; r < 16; ++r) x[r] = __fmaf_rn(-A[(b0 + r) * AS + b0 + kk], x[kk], x[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r) T[(b0 + r) * AS + b0 + c] = x[r];
        }
        __syncthreads();
        // Off-diagonal blocks by doubling: for a block lower-triangular
        // L = [L11 0; L21 L22], L^-1 has lower-left block -L22^-1 L21 L11^-1.
        // Level 1 (16-blocks): T10 = -T11 (M10 T00), T32 = -T33 (M32 T22);
        // level 2 (32-blocks): T[32:, :32] = -T[32:, 32:] (M[32:, :32] T[:32, :32]).
        // The diagonal blocks' zero upper halves let the level-1 sums run full
        // length.  Every sum runs on two or four independent partial sums.
        // The strictly upper 16-blocks of T are never written; the operands
        // below take them as zero.
        float *X = QK;   // scratch (P went straight to the chunk block)
        {
            const int pr = tid >> 8, rr = (tid >> 4) & 15, cc = tid & 15;
            const int bi = 2 * pr + 1, bj = 2 * pr;
            const float *m = A + (bi * 16 + rr) * AS + bj * 16;
            const float *tb = T + (bj * 16) * AS + bj * 16 + cc;
            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
            for (int kk = 0; kk < 16; kk += 2) {
                a0 = __fmaf_rn(m[kk], tb[kk * AS], a0);
                a1 = __fmaf_rn(m[kk + 1], tb[(kk + 1) * AS], a1);
            }
            X[(pr * 16 + rr) * AS + cc] = __fadd_rn(a0, a1);
            __syncthreads();
            const float *td = T + (bi * 16 + rr) * AS + bi * 16;
            const float *xc = X + (pr * 16) * AS + cc;
            a0 = 0.0f;
            a1 = 0.0f;
#pragma unroll
            for (int kk = 0; kk < 16; kk += 2) {
                a0 = __fmaf_rn(td[kk], xc[kk * AS], a0);
                a1 = __fmaf_rn(td[kk + 1], xc[(kk + 1) * AS], a1);
            }
            T[(bi * 16 + rr) * AS + bj * 16 + cc] = -__fadd_rn(a0, a1);
        }
        __syncthreads();
        constexpr int H = C / 2;
        constexpr int NU = H * H / kPrepTcThreads;
        {   // level 2, X = M[32:, :32] T[:32, :32]: lane row r, warp-uniform columns
            // c1 = w and c2 = 31 - w (balancing the threads); T[:32, :32] is lower
            // triangular, so column c's sum starts at kk = c, and from kk = c2 on
            // the two sums share their load of M[32 + r][kk]
            static_assert(NU == 2, "two level-2 outputs per thread");
            const int c1 = warp, c2 = H - 1 - warp, r = lane;
            const float *m = A + (H + r) * AS;
            float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
            int kk = c1;
            for (; kk + 1 < c2; kk += 2) {
                a0 = __fmaf_rn(m[kk], T[kk * AS + c1], a0);
                a1 = __fmaf_rn(m[kk + 1], T[(kk + 1) * AS + c1], a1);
            }
            if (kk < c2) {
                a0 = __fmaf_rn(m[kk], T[kk * AS + c1], a0);
                ++kk;
            }
            for (; kk < H; ++kk) {
                const float mv = m[kk];
                a1 = __fmaf_rn(mv, T[kk * AS + c1], a1);
                b0 = __fmaf_rn(mv, T[kk * AS + c2], b0);
            }
            X[r * AS + c1] = __fadd_rn(a0, a1);
            X[r * AS + c2] = __fadd_rn(b0, b1);
        }
        __syncthreads();
        {   // T[32:, :32] = -T[32:, 32:] X: lane column c, warp-uniform rows r1 = w
            // and r2 = 31 - w; T[32:, 32:] is lower triangular, so row r's sum
            // stops at kk = r, and up to kk = r1 the two sums share their load
            // of X[kk][c]
            const int r1 = warp, r2 = H - 1 - warp, c = lane;
            const float *t1 = T + (H + r1) * AS + H, *t2 = T + (H + r2) * AS + H;
            float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
            int kk = 0;
            for (; kk <= r1; ++kk) {
                const float xv = X[kk * AS + c];
                a0 = __fmaf_rn(t1[kk], xv, a0);
                b0 = __fmaf_rn(t2[kk], xv, b0);
            }
            for (; kk + 1 <= r2; kk += 2) {
                b0 = __fmaf_rn(t2[kk], X[kk * AS + c], b0);
                b1 = __fmaf_rn(t2[kk + 1], X[(kk + 1) * AS + c], b1);
            }
            if (kk <= r2) b0 = __fmaf_rn(t2[kk], X[kk * AS + c], b0);
            T[(H + r1) * AS + c] = -__fadd_rn(a0, a1);
            T[(H + r2) * AS + c] = -__fadd_rn(b0, b1);
        }
        __syncthreads();
        // operands, rows t, K = s: T (for U~) and T' = T diag(b gamma) (for W),
        // both from one read of T
        for (int it = tid; it < C * (C / 8); it += kPrepTcThreads) {
            const int t = it % C, s0 = (it / C) * 8;
            float x[8], xp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s2 = s0 + e;
                x[e] = (s2 >> 4) > (t >> 4) ? 0.0f : T[t * AS + s2];
                xp[e] = __fmul_rn(x[e], __fmul_rn(beta[s2], eG[s2]));
            }
            store_split8(t_hi, t_lo, t, s0, C, x);
            store_split8(tp_hi, tp_lo, t, s0, C, xp);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();

        // MMA 2: W^T = K^T T'^T (columns 64..127), U~^T = (b V)^T T^T (128..191)
        if (tid == 0) {
            constexpr uint32_t idn = tc::idesc_bf16(128, C);
            const uint32_t th = tc::smem_u32(t_hi), tl = tc::smem_u32(t_lo);
            const uint32_t ph_ = tc::smem_u32(tp_hi), pl = tc::smem_u32(tp_lo);
            const uint32_t kh_ = tc::smem_u32(kt_hi), kl = tc::smem_u32(kt_lo);
            const uint32_t vh = tc::smem_u32(v_hi), vl = tc::smem_u32(v_lo);
            tc::mma_bf16<C>(tmem_base + 64, kh_, ph_, idn, false);
            tc::mma_bf16<C>(tmem_base + 64, kh_, pl, idn, true);
            tc::mma_bf16<C>(tmem_base + 64, kl, ph_, idn, true);
            tc::mma_bf16<C>(tmem_base + 128, vh, th, idn, false);
            tc::mma_bf16<C>(tmem_base + 128, vh, tl, idn, true);
            tc::mma_bf16<C>(tmem_base + 128, vl, th, idn, true);
            tc::mma_commit(&bar_mma);
        }
        // while MMA 2 runs: K~^T = (diag(gamma_C / gamma) K)^T for the scan
        for (int it = tid; it < D * (C / 8); it += kPrepTcThreads) {   // K~^T rows j, 8 t
            const int j = it % D, t0 = (it / D) * 8;
            float kt[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) kt[e] = (t0 + e) < n ? __fmul_rn(eGC[t0 + e], k[(t0 + e) * LD + j]) : 0.0f;
            store_split8(blk + TcBlock::kPK, blk + TcBlock::kPK + TcBlock::kPKLo, C + j, t0, C, kt);
        }
        ok = tc::mbar_wait(&bar_mma, ph, kPrepWaitLimit) && ok;
        ph ^= 1;
        tc::fence_after_sync();
        {
            // lane j of W^T: W[t][j] for every t (warps 0-7); lane i of U~^T:
            // U~^T[i][t] (warps 8-15); two warps per lane quarter and matrix,
            // 32 columns each, into fp32 stages
            const int r = quarter * 32 + lane;
            const bool isU = part >= 2;
            const int c0 = (part & 1) * (C / 2);
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (isU ? 128 : 64) + c0;
            uint32_t v[C / 32][16];
#pragma unroll
            for (int q2 = 0; q2 < C / 32; ++q2) tc::tmem_ld16_nowait(taddr + q2 * 16, v[q2]);
            tc::tmem_wait_ld();
            if (!isU) {   // column r of W: the lanes' columns differ in their low five bits
#pragma unroll
                for (int q2 = 0; q2 < C / 32; ++q2)
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int t = c0 + q2 * 16 + e;
                        Wf[t * D + swz(t, r)] = __uint_as_float(v[q2][e]);
                    }
            } else {      // row r of U~^T as float4s (eight lanes cover the 32 banks)
#pragma unroll
                for (int q2 = 0; q2 < C / 32; ++q2)
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(Uf + r * C + swz(r, c0 + q2 * 16 + e)) =
                            make_float4(__uint_as_float(v[q2][e]), __uint_as_float(v[q2][e + 1]),
                                        __uint_as_float(v[q2][e + 2]), __uint_as_float(v[q2][e + 3]));
            }
        }
        if (gi + 1 < p.G) cp_async_wait_all();   // the next head's v inputs and weights
        __syncthreads();   // the W and U~^T stages are complete (and the next head's v inputs landed)
        // The stores leave at the SM's store rate, and a thread waits on its
        // own stores: with a next head, warps 0-7 store while warps 8-15 run
        // its v conv (which writes the v operand in region 1's first half and
        // touches neither stage); the next head's first barrier orders both
        // before M and T reuse the stages.  The last head stores on every warp.
        const bool more = gi + 1 < p.G;
        const int n_st = more ? kPrepTcThreads / 2 : kPrepTcThreads;
        if (tid < n_st) {
            float4 *dst = reinterpret_cast<float4 *>(blk + TcBlock::kUt);   // U~^T [128][64] fp32, row-major
            for (int it = tid; it < D * C / 4; it += n_st) {
                const int i = it / (C / 4), t4 = it % (C / 4);
                dst[it] = *reinterpret_cast<const float4 *>(Uf + i * C + swz(i, t4 * 4));
            }
            for (int it = tid; it < C * (D / 8); it += n_st) {   // -W hi | lo, rows t, 8 columns j
                const int t = it % C, j0 = (it / C) * 8;
                const float4 a4 = *reinterpret_cast<const float4 *>(Wf + t * D + swz(t, j0));
                const float4 b4 = *reinterpret_cast<const float4 *>(Wf + t * D + swz(t, j0 + 4));
                const float x[8] = {-a4.x, -a4.y, -a4.z, -a4.w, -b4.x, -b4.y, -b4.z, -b4.w};
                store_split8(blk + TcBlock::kWQ, blk + TcBlock::kWQ + TcBlock::kWQLo, t, j0, D, x);
            }
            if (tid == 0) *reinterpret_cast<float *>(blk + TcBlock::kMisc) = eG[n - 1];
            if (tid < C) reinterpret_cast<float *>(blk + TcBlock::kGam)[tid] = eG[tid];   // gamma_t for O
        } else {
            conv_v(gi + 1, n_st, kPrepTcThreads - n_st);
        }
    }
    }   // items
    if (tid == 0) {
        if (!ok) raise_error(p.err, GDN_DERR_TIMEOUT);
        tc::mma_commit(&bar_mma);   // no MMA may still write TMEM when it is freed
        tc::mbar_wait(&bar_mma, ph, kPrepWaitLimit);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

// ---------------------------------------------------------------------------
// scan on the tensor cores (d = 128): one CTA of 256 threads per (value
// head, sequence).  Threads i and i + 128 (warps w and w + 4) share TMEM lane
// i, i.e. state row i, and split its columns.  TMEM (512 columns) holds
//   0..127    [U^T | O1^T] fp32 [128 x 64] each
//   128..319  [O2^T | S]: O2^T [128 x 64] and the state S fp32 [128 x 128],
//             kept from chunk to chunk
//   320..383  S0 hi, 384..447 S0 lo   (bf16 pairs: A operand of group 1)
//   448..479  U^T hi, 480..511 U^T lo (bf16 pairs: A operand of group 2)
// A operands in TMEM put row m in lane m and elements (m, 2c), (m, 2c + 1)
// in the low and high half of column c.  Every product is three bf16 MMAs
// (hi*hi + hi*lo + lo*hi) accumulating in fp32.  Per chunk:
//   group 1: [U^T | O1^T] = [U~^T | 0] + S0 [-W; Q]^T   (N = 128, K = 128;
//            U~^T is stored into TMEM a chunk ahead, so U = U~ - S0 W^T
//            leaves the tensor core finished; Q is the key head's, shared
//            by its value heads, so the decay gamma_t is applied after)
//   U -> bf16 hi/lo A operand
//   group 2: [O2^T | S] += U^T [P; K~^T]^T        (N = 192, K = 64)
//   S -> bf16 hi/lo A operand of the next chunk; S <- gamma_C' S
//   O^T = diag(gamma) O1^T + O2^T -> the workspace (fp32) for the norm pass
// With both A operands in TMEM a 128 x 128 x 16 step reads only its B tile
// from shared memory.  The chunk operands are double-buffered in shared
// memory: chunk c+1's bulk copies (five for group 1 and gamma_t, one for
// group 2; a bulk-copy issue costs tens of cycles whatever its size) are
// issued by a thread of warp 1 when chunk c starts, so the MMA-issuing
// thread never waits on them.
// ---------------------------------------------------------------------------
constexpr int kScanTcThreads = 256;   // two threads per TMEM lane, splitting the columns
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kOpBuf = TcBlock::kOpBytes + 64 * 4;   // one chunk's operands, then its gamma_t
constexpr size_t kScanTcSmem = 2 * (size_t)kOpBuf;
constexpr uint32_t kTmemO2 = 128, kTmemS = 192, kTmemShi = 320, kTmemSlo = 384, kTmemUhi = 448, kTmemUlo = 480;

// The chunk's [-W; Q] operand (-W from the head's block, Q from the key
// head's lead block) and gamma_t, completing on bar1, and its [P; K~^T]
// operand on bar2, into one buffer.
__device__ __forceinline__ void issue_chunk_copies(unsigned char *ops, const unsigned char *blk,
                                                   const unsigned char *lead, uint64_t *bar1, uint64_t *bar2) {
    constexpr int H = TcBlock::kHalf, LO = TcBlock::kWQLo;
    tc::mbar_expect_tx(bar1, TcBlock::kGroup1 + 64 * 4);
    tc::bulk_g2s(ops, blk, H, bar1);                      // -W hi
    tc::bulk_g2s(ops + H, lead + H, H, bar1);             // Q hi
    tc::bulk_g2s(ops + LO, blk + LO, H, bar1);            // -W lo
    tc::bulk_g2s(ops + LO + H, lead + LO + H, H, bar1);   // Q lo
    tc::bulk_g2s(ops + TcBlock::kOpBytes, blk + TcBlock::kGam, 64 * 4, bar1);
    tc::mbar_expect_tx(bar2, TcBlock::kGroup2);
    tc::bulk_g2s(ops + TcBlock::kGroup1, blk + TcBlock::kGroup1, TcBlock::kGroup2, bar2);
}

// S (TMEM fp32) -> its bf16 hi/lo pair columns (the next group-1 A operand),
// and S <- gamma_C * S for the coming U^T K~ accumulation.  This thread
// handles its lane's columns [half * 64, half * 64 + 64).
__device__ __forceinline__ void split_and_scale_state(uint32_t tmem_lane, int half, float gC) {
    uint32_t r[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q) tc::tmem_ld16_nowait(tmem_lane + kTmemS + half * 64 + q * 16, r[q]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            tc::split_bf16x2(__uint_as_float(r[q][2 * e]), __uint_as_float(r[q][2 * e + 1]), hw[e], lw[e]);
        tc::tmem_st8_nowait(tmem_lane + kTmemShi + half * 32 + q * 8, hw);
        tc::tmem_st8_nowait(tmem_lane + kTmemSlo + half * 32 + q * 8, lw);
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fmul_rn(gC, __uint_as_float(r[q][e]));
        tc::tmem_st16_nowait(tmem_lane + kTmemS + half * 64 + q * 16, v);
    }
    tc::tmem_wait_st();
}

// Seed the accumulators of this thread's lane: its half of the chunk's U~^T
// row into the U columns, zeros into the O1 and O2 columns.
template <int C>
__device__ __forceinline__ void seed_group1(uint32_t tmem_lane, int half, const float4 (&ut)[C / 8]) {
#pragma unroll
    for (int q = 0; q < C / 32; ++q) {
        float v[16], z[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 u = ut[q * 4 + e];
            v[4 * e] = u.x; v[4 * e + 1] = u.y; v[4 * e + 2] = u.z; v[4 * e + 3] = u.w;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0.0f;
        tc::tmem_st16_nowait(tmem_lane + half * (C / 2) + q * 16, v);
        tc::tmem_st16_nowait(tmem_lane + 64 + half * (C / 2) + q * 16, z);
        tc::tmem_st16_nowait(tmem_lane + kTmemO2 + half * (C / 2) + q * 16, z);
    }
    tc::tmem_wait_st();
}

// This thread's half of row i of a chunk's U~^T (fp32 [128][C]).
template <int C>
__device__ __forceinline__ void load_ut(float4 (&ut)[C / 8], const unsigned char *blk, int i, int half) {
    const float4 *src = reinterpret_cast<const float4 *>(blk + TcBlock::kUt) + i * (C / 4) + half * (C / 8);
#pragma unroll
    for (int e = 0; e < C / 8; ++e) ut[e] = src[e];
}

template <int C>
__global__ void __launch_bounds__(kScanTcThreads, 1) gdn_prefill_scan_tc_kernel(const PrefillParams p) {
    constexpr int D = 128;
    static_assert(C == 64, "the TMEM column map is for C = 64");
    extern __shared__ __align__(1024) unsigned char tsm[];   // two operand buffers
    __shared__ __align__(8) uint64_t bar_g1[2], bar_g2[2], bar_u, bar_s, bar_end;
    __shared__ uint32_t tmem_base;
    __shared__ int fail;

    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int base = chunk_base(p, C, s);
    if (base < 0) {
        if (h == 0 && tid == 0) raise_error(p.err, GDN_DERR_SEQLENS);
        return;
    }
    const int lo = __ldg(p.cu_seqlens + s), hi = __ldg(p.cu_seqlens + s + 1);
    const int L_s = hi - lo;
    if (L_s == 0) return;
    const int sl = __ldg(p.slot + s);
    if (sl < 0 || sl >= p.n_slots) {
        if (h == 0 && tid == 0) raise_error(p.err, GDN_DERR_SLOT);
        return;
    }
    const int n_chunks = (L_s + C - 1) / C;
    // this launch's chunks of the sequence: [c_first, c_end); the state comes
    // from the slot and goes back to it, so launches over consecutive ranges
    // continue one another
    const int c_first = max(0, p.c_lo - base), c_end = min(n_chunks, p.c_hi - base);
    if (c_first >= c_end) return;
    const size_t blk_stride = (size_t)p.Hv * TcBlock::kBytes;
    const unsigned char *blk0 = reinterpret_cast<const unsigned char *>(p.ws_chunks) +
                                ((size_t)(base + c_first) * p.Hv + h) * TcBlock::kBytes;
    const size_t lead_off = (size_t)(h % p.G) * TcBlock::kBytes;   // blk - lead: Q is in the key head's first block

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bar_g1[b], 1);
            tc::mbar_init(&bar_g2[b], 1);
        }
        tc::mbar_init(&bar_u, 1);
        tc::mbar_init(&bar_s, 1);
        tc::mbar_init(&bar_end, 1);
        fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::fence_async_smem();
    if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t tl = tmem_base + ((uint32_t)(quarter * 32) << 16);   // this warp's lane quarter
    const int i = quarter * 32 + (tid & 31);   // state row (value channel); columns split by `half`
    constexpr uint32_t idN128 = tc::idesc_bf16(128, 128), idN192 = tc::idesc_bf16(128, 192);

    constexpr int kCopier = 32;   // lane 0 of warp 1 issues the bulk copies
    if (tid == kCopier) issue_chunk_copies(tsm, blk0, blk0 - lead_off, &bar_g1[0], &bar_g2[0]);
    // the committed state row i into TMEM
    float *srow = p.state + ((size_t)sl * p.Hv + h) * D * D + (size_t)i * D;
#pragma unroll 1
    for (int cb = half * 4; cb < half * 4 + 4; ++cb) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(srow + cb * 16 + e);
            v[e] = f.x; v[e + 1] = f.y; v[e + 2] = f.z; v[e + 3] = f.w;
        }
        tc::tmem_st16_nowait(tl + kTmemS + cb * 16, v);
    }
    tc::tmem_wait_st();

    // chunk 0's gamma_C and U~^T row; later chunks' are read one chunk ahead
    float gC = *reinterpret_cast<const float *>(blk0 + TcBlock::kMisc);
    float4 ut[C / 8];
    load_ut<C>(ut, blk0, i, half);
    split_and_scale_state(tl, half, gC);
    seed_group1<C>(tl, half, ut);

    bool ok = true;
    int issued = 1;   // chunks (counted from c_first) whose copies have been issued
    const int n_run = c_end - c_first;
    // A chunk's O^T row leaves TMEM at the chunk's end but goes to the
    // workspace only after the next chunk's group-1 MMAs are issued: the
    // stores (32 KB a chunk, bound by the SM's store rate) then drain while
    // the tensor core works instead of delaying the next issue.
    uint32_t o_r[C / 32][16];
    int o_start = 0, o_n = 0;
    auto store_o = [&]() {
        float *ocol = p.ws_out + ((size_t)o_start * p.Hv + h) * D + i;
#pragma unroll
        for (int q = 0; q < C / 32; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int t = half * (C / 2) + q * 16 + e;
                if (t < o_n) ocol[(size_t)t * p.Hv * D] = __uint_as_float(o_r[q][e]);
            }
        o_n = 0;
    };
#pragma unroll 1
    for (int c = 0; c < n_run && ok; ++c) {   // c counts from c_first
        const unsigned char *blk = blk0 + (size_t)c * blk_stride;
        unsigned char *ops = tsm + (c & 1) * kOpBuf;
        const uint32_t par = (c >> 1) & 1;   // fill count of this buffer, mod 2
        const bool more = c + 1 < n_run;
        const int start = lo + (c_first + c) * C;
        const int n = min(C, hi - start);
        tc::fence_before_sync();
        __syncthreads();   // S operand written; the previous chunk's O readout is done
        tc::fence_after_sync();
        if (fail) {   // read after a barrier: the same value in every thread
            ok = false;
            break;
        }
        // the other buffer was last read by chunk c-1's MMAs, all complete
        if (tid == kCopier && more)
            issue_chunk_copies(tsm + ((c + 1) & 1) * kOpBuf, blk + blk_stride, blk + blk_stride - lead_off,
                               &bar_g1[(c + 1) & 1],
                               &bar_g2[(c + 1) & 1]);
        if (more) issued = c + 2;

        // group 1: [U^T | O^T] = S0 [W; Q~]^T, one N = 128 product into TMEM columns 0..127
        if (tid == 0) {
            if (!tc::mbar_wait(&bar_g1[c & 1], par, kWaitLimit)) {
                fail = 1;
                tc::mma_commit(&bar_u);
            } else {
                const uint32_t b_hi = tc::smem_u32(ops + TcBlock::kWQ), b_lo = b_hi + TcBlock::kWQLo;
                tc::mma_bf16_ta<D>(tmem_base, tmem_base + kTmemShi, b_hi, idN128, true);
                tc::mma_bf16_ta<D>(tmem_base, tmem_base + kTmemShi, b_lo, idN128, true);
                tc::mma_bf16_ta<D>(tmem_base, tmem_base + kTmemSlo, b_hi, idN128, true);
                tc::mma_commit(&bar_u);
            }
        }
        // while the MMAs run: the previous chunk's O, the next chunk's gamma_C and U~^T row
        if (o_n > 0) store_o();
        float gC_nx = 0.0f;
        if (more) {
            gC_nx = *reinterpret_cast<const float *>(blk + blk_stride + TcBlock::kMisc);
            load_ut<C>(ut, blk + blk_stride, i, half);
        }
        if (!tc::mbar_wait(&bar_u, c & 1, kWaitLimit)) fail = 1;
        tc::fence_after_sync();

        // U (finished by the tensor core) -> its bf16 hi/lo pairs (row i, K = t) in TMEM
        {
            uint32_t r[C / 32][16];
#pragma unroll
            for (int q = 0; q < C / 32; ++q) tc::tmem_ld16_nowait(tl + half * (C / 2) + q * 16, r[q]);
            tc::tmem_wait_ld();
            uint32_t hw[C / 4], lw[C / 4];
#pragma unroll
            for (int e = 0; e < C / 4; ++e)
                tc::split_bf16x2(__uint_as_float(r[e / 8][(e % 8) * 2]), __uint_as_float(r[e / 8][(e % 8) * 2 + 1]),
                                 hw[e], lw[e]);
            tc::tmem_st16_nowait(tl + kTmemUhi + half * (C / 4), hw);
            tc::tmem_st16_nowait(tl + kTmemUlo + half * (C / 4), lw);
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (fail) {
            ok = false;
            break;
        }

        // group 2: [O^T | S] += U^T [P; K~^T]^T, one N = 192 product into TMEM columns 64..255
        if (tid == 0) {
            if (!tc::mbar_wait(&bar_g2[c & 1], par, kWaitLimit)) {
                fail = 1;
                tc::mma_commit(&bar_s);
            } else {
                const uint32_t b_hi = tc::smem_u32(ops + TcBlock::kPK), b_lo = b_hi + TcBlock::kPKLo;
                tc::mma_bf16_ta<C>(tmem_base + kTmemO2, tmem_base + kTmemUhi, b_hi, idN192, true);
                tc::mma_bf16_ta<C>(tmem_base + kTmemO2, tmem_base + kTmemUhi, b_lo, idN192, true);
                tc::mma_bf16_ta<C>(tmem_base + kTmemO2, tmem_base + kTmemUlo, b_hi, idN192, true);
                tc::mma_commit(&bar_s);
            }
        }
        if (!tc::mbar_wait(&bar_s, c & 1, kWaitLimit)) fail = 1;
        tc::fence_after_sync();
        if (more && !fail) {
            gC = gC_nx;
            split_and_scale_state(tl, half, gC);   // the next chunk's S operand
        }

        // O^T row i = gamma_t O1^T + O2^T out of TMEM (stored to O[t][i] during
        // the next chunk's group 1); gamma_t came with this chunk's group-1 copies
        {
            const float *gam = reinterpret_cast<const float *>(ops + TcBlock::kOpBytes) + half * (C / 2);
#pragma unroll
            for (int q = 0; q < C / 32; ++q) {
                uint32_t o2[16];
                tc::tmem_ld16_nowait(tl + 64 + half * (C / 2) + q * 16, o_r[q]);
                tc::tmem_ld16_nowait(tl + kTmemO2 + half * (C / 2) + q * 16, o2);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    o_r[q][e] = __float_as_uint(
                        __fmaf_rn(gam[q * 16 + e], __uint_as_float(o_r[q][e]), __uint_as_float(o2[e])));
            }
        }
        o_start = start;
        o_n = n;
        if (more && !fail) seed_group1<C>(tl, half, ut);   // after this lane's U and O columns are read
    }
    if (ok && o_n > 0) store_o();   // the last chunk's O
    __syncthreads();
    ok = fail == 0;

    if (ok) {
        // final state row i back to the slot
#pragma unroll 1
        for (int cb = half * 4; cb < half * 4 + 4; ++cb) {
            float v[16];
            tc::tmem_ld16(tl + kTmemS + cb * 16, v);
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(srow + cb * 16 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
        // the slot's new conv tail (as in the CUDA-core scan), by the launch
        // that ends the sequence
        const int kh = h / p.G;
        const bool lead = (h % p.G) == 0;
        const size_t CH = (size_t)p.CH;
        for (int cc = tid; cc < (c_end == n_chunks ? 3 * D : 0); cc += kScanTcThreads) {
            const int part = cc / D;
            if (part < 2 && !lead) continue;
            const int ch = pchannel<D>(part, cc - part * D, p.Hk, kh, h);
            uint16_t *tl16 = p.tail + (size_t)sl * 3 * CH + ch;
            const uint16_t old[3] = {tl16[0], tl16[CH], tl16[2 * CH]};
            uint16_t nw[3];
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const int pos = L_s - 3 + m;
                nw[m] = pos >= 0 ? p.mixed[(size_t)(lo + pos) * CH + ch] : old[3 + pos];
            }
            tl16[0] = nw[0];
            tl16[CH] = nw[1];
            tl16[2 * CH] = nw[2];
        }
    } else if (tid == 0) {
        raise_error(p.err, GDN_DERR_TIMEOUT);
    }
    if (tid == 0) {
        // no bulk copy may still land in this CTA's shared memory, and no MMA
        // may still write TMEM, when the CTA leaves (bounded waits)
        // the last fill of each buffer (an already completed phase returns at once)
        for (int c2 = max(0, issued - 2); c2 < issued; ++c2) {
            tc::mbar_wait(&bar_g1[c2 & 1], (c2 >> 1) & 1, kWaitLimit);
            tc::mbar_wait(&bar_g2[c2 & 1], (c2 >> 1) & 1, kWaitLimit);
        }
        tc::mma_commit(&bar_end);
        tc::mbar_wait(&bar_end, 0, kWaitLimit);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------------------
// norm: one warp per (token, value head): y = O / sqrt(mean O^2 + eps) * w * SiLU(z)
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void norm_item(const PrefillParams &p, size_t item, int lane) {
    constexpr int CPL = D / 32;
    static_assert(CPL == 1 || CPL == 2 || CPL == 4, "lane slices of 1, 2 or 4 elements");
    float ov[CPL];
    uint16_t zb[CPL], wb[CPL];
    const size_t at = item * D + lane * CPL;
    if constexpr (CPL == 4) {   // 16-byte O, 8-byte z and w per lane
        const float4 o4 = *reinterpret_cast<const float4 *>(p.ws_out + at);
        ov[0] = o4.x; ov[1] = o4.y; ov[2] = o4.z; ov[3] = o4.w;
        const uint2 z2 = *reinterpret_cast<const uint2 *>(p.z + at);
        const uint2 w2 = *reinterpret_cast<const uint2 *>(p.norm_w + lane * CPL);
        zb[0] = z2.x & 0xffffu; zb[1] = z2.x >> 16; zb[2] = z2.y & 0xffffu; zb[3] = z2.y >> 16;
        wb[0] = w2.x & 0xffffu; wb[1] = w2.x >> 16; wb[2] = w2.y & 0xffffu; wb[3] = w2.y >> 16;
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            ov[c] = p.ws_out[at + c];
            zb[c] = p.z[at + c];
            wb[c] = p.norm_w[lane * CPL + c];
        }
    }
    float ss = __fmul_rn(ov[0], ov[0]);
#pragma unroll
    for (int c = 1; c < CPL; ++c) ss = __fmaf_rn(ov[c], ov[c], ss);
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / D), p.eps_rms)));
    uint16_t yb[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const float yv = __fmul_rn(__fmul_rn(__fmul_rn(ov[c], inv), bf_bits(wb[c])), silu(bf_bits(zb[c])));
        yb[c] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
    }
    if constexpr (CPL == 4) {
        *reinterpret_cast<uint2 *>(p.y + at) =
            make_uint2((uint32_t)yb[0] | ((uint32_t)yb[1] << 16), (uint32_t)yb[2] | ((uint32_t)yb[3] << 16));
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) p.y[at + c] = yb[c];
    }
}

// The tokens of global chunks [c_lo, c_hi): one CTA per (value head, chunk),
// so a pipelined pass normalises each chunk group right after its scan.
// Only tokens of a sequence that the scan ran are normalised: tokens outside
// every sequence (before cu_seqlens[0] or after the last entry) and the
// tokens of a sequence skipped for a bad slot or bad cu_seqlens have no O,
// and their y is left as it was.
template <int D, int C>
__global__ void __launch_bounds__(kNormThreads) gdn_prefill_norm_chunks_kernel(const PrefillParams p) {
    __shared__ int info[2];
    // blockIdx.x = head * kNormSplit + part: each CTA takes C / kNormSplit of
    // its chunk's tokens, so that a CTA is short and hands its SM back soon
    const int h = blockIdx.x / kNormSplit, part = blockIdx.x % kNormSplit, gc = p.c_lo + blockIdx.y;
    if (threadIdx.x == 0) {
        int seq = -1, start = 0, n = 0, seq_start = 0, bad = 0;
        const bool ok = locate_chunk(p, C, gc, seq, start, n, seq_start, bad);
        const int sl = ok ? __ldg(p.slot + seq) : -1;
        info[0] = (ok && !bad && sl >= 0 && sl < p.n_slots) ? n : 0;
        info[1] = start;
    }
    __syncthreads();
    const int n = info[0], start = info[1];
    constexpr int TPC = C / kNormSplit;   // tokens of this CTA
    const int t_end = min(n, (part + 1) * TPC);
    for (int t = part * TPC + (threadIdx.x >> 5); t < t_end; t += kNormThreads / 32)
        norm_item<D>(p, (size_t)(start + t) * p.Hv + h, threadIdx.x & 31);
}

}  // namespace gdn
