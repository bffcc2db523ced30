// gdn_common.cuh -- device helpers shared by the GDN kernels (sm_103a).
//
// Rounding discipline: every floating-point step of the recurrence, the conv
// and the norms is written with explicit round-to-nearest intrinsics
// (__fmul_rn / __fadd_rn / __fmaf_rn / __fdiv_rn / __fsqrt_rn) or with one
// fixed fast intrinsic (SiLU's exponential and division, the RMSNorm's
// reciprocal square root), the same call in every kernel, so no compiler
// contraction can make two kernels that share these helpers round
// differently.  That is what makes every row of a window identical, bit for
// bit, to the same row run as a single step, and a tree node identical to
// the chain along its path (TensorFold #932, note on the Qwen3.5 CUDA
// engine, which asks exactly that of windows).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/gdn.h"

namespace gdn {

using bf16 = __nv_bfloat16;

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf(const bf16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float bf_bits(uint16_t u) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// SiLU(x) = x / (1 + e^-x), with the fast exponential and division (a few
// ulp; one function for every instantiation, so steps, windows and trees
// still agree bit for bit; beyond |x| ~ 88 the quotient's limit, x or 0, is
// what comes out)
__device__ __forceinline__ float silu(float x) {
    return __fdividef(x, __fadd_rn(1.0f, __expf(-x)));
}

// sigmoid(x) = 1 / (1 + e^-x)
__device__ __forceinline__ float sigmoidf_rn(float x) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

// softplus(x) = log(1 + e^x); above 20 the correction is below fp32's
// resolution of x and x itself is returned.
__device__ __forceinline__ float softplusf_rn(float x) {
    return x > 20.0f ? x : log1pf(expf(x));
}

// Sum over the 32 lanes of a warp with the xor butterfly 16, 8, 4, 2, 1.
// Every lane receives the same bits.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// Sum over the 32 lanes with the xor butterfly 1, 2, 4, 8, 16: after the
// first k levels every aligned group of 2^k lanes holds its own sum, so a
// sum split into aligned lane groups (and finished from the groups' sums in
// the same pairwise order) has the same bits as the whole.
__device__ __forceinline__ float warp_sum_up(float v) {
#pragma unroll
    for (int off = 1; off <= 16; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// Reduce-scatter of N partial sums (N a power of two, 2..32) across the 32
// lanes.  On return lane l holds the total of value (l >> (5 - log2 N)).
// The association is the same xor butterfly as warp_sum (partners l^16,
// then l^8, ...), so each total has the same bits as warp_sum would give.
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
    for (int level = 0; level < 5; ++level) {
        const int off = 16 >> level;
        const int cnt = N >> level;
        if (cnt > 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < cnt / 2; ++i) {
                const float send = upper ? v[i] : v[i + cnt / 2];
                const float keep = upper ? v[i + cnt / 2] : v[i];
                v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
            }
        } else {
            v[0] = __fadd_rn(v[0], __shfl_xor_sync(kFull, v[0], off));
        }
    }
    return v[0];
}

template <int N>
struct Log2 {
    static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

// 16-byte global -> shared copy that bypasses registers (and L1).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}

// Wait for every cp.async this thread issued.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *gmem) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(gmem));
}

// Ask L2 for `bytes` (a multiple of 16) at a 16-byte aligned global address:
// one bulk prefetch, nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void *gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

__device__ __forceinline__ void raise_error(int *err, int bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace gdn
