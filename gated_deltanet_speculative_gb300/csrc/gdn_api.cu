// gdn_api.cu -- the C ABI (include/gdn.h): host-side validation, launch
// configuration and status codes.  Nothing here allocates device memory;
// every buffer belongs to the caller (the d = 128 prefill also uses two side
// streams and four events of its own per device, made on first use).
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "gdn_commit.cuh"
#include "gdn_context.h"
#include "gdn_launch.h"
#include "gdn_prefill_launch.h"

namespace {

__device__ int g_device_error;   // OR of GDN_DERR_* bits raised by the kernels

constexpr int kMaxDevices = 64;

// Per-device address of g_device_error, looked up on a device's first call
// and again whenever the current context has changed since.
int *error_word() {
    static void *addr[kMaxDevices] = {};
    static unsigned long long ctx[kMaxDevices] = {};
    static std::mutex mu;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *a = nullptr;
    if (gdn::symbol_address(g_device_error, &a, &addr[dev], &ctx[dev], mu) != cudaSuccess) return nullptr;
    return static_cast<int *>(a);
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int check_dims(const gdn_dims *d) {
    if (!d) return GDN_ENULL;
    if (d->n_k_heads <= 0 || d->n_v_heads <= 0 || d->n_v_heads > 65535) return GDN_EINVAL;
    if (d->n_v_heads % d->n_k_heads != 0 || d->n_v_heads / d->n_k_heads > 8) return GDN_EINVAL;
    if (d->d_k != d->d_v || (d->d_k != 32 && d->d_k != 64 && d->d_k != 128)) return GDN_EINVAL;
    if (d->conv_width != 4) return GDN_EINVAL;
    if (!std::isfinite(d->q_scale)) return GDN_EINVAL;
    if (!(d->eps_l2 >= 0.0f) || !std::isfinite(d->eps_l2)) return GDN_EINVAL;
    if (!(d->eps_rms >= 0.0f) || !std::isfinite(d->eps_rms)) return GDN_EINVAL;
    return GDN_OK;
}

int check_weights(const gdn_weights *w) {
    if (!w || !w->conv_w || !w->A_log || !w->dt_bias || !w->norm_w) return GDN_ENULL;
    if (!aligned(w->conv_w, 16) || !aligned(w->norm_w, 16) || !aligned(w->A_log, 4) || !aligned(w->dt_bias, 4))
        return GDN_EALIGN;
    return GDN_OK;
}

int check_cache(const gdn_cache *c) {
    if (!c || !c->state || !c->tail) return GDN_ENULL;
    if (c->n_slots <= 0) return GDN_EINVAL;
    if (!aligned(c->state, 16) || !aligned(c->tail, 16)) return GDN_EALIGN;
    return GDN_OK;
}

int check_rows(const gdn_rows *r) {
    if (!r || !r->mixed || !r->z || !r->a || !r->b || !r->y) return GDN_ENULL;
    if (!aligned(r->mixed, 16) || !aligned(r->z, 16) || !aligned(r->y, 16) || !aligned(r->a, 2) ||
        !aligned(r->b, 2))
        return GDN_EALIGN;
    return GDN_OK;
}

#define GDN_TRY(expr)                 \
    do {                              \
        const int rc_ = (expr);       \
        if (rc_ != GDN_OK) return rc_; \
    } while (0)

gdn::RowParams row_params(const gdn_dims *d, const gdn_weights *w, const gdn_cache *c, const gdn_rows *r,
                          const int32_t *slot, int *err) {
    gdn::RowParams p = {};
    p.Hk = d->n_k_heads;
    p.Hv = d->n_v_heads;
    p.G = d->n_v_heads / d->n_k_heads;
    p.CH = 2 * d->n_k_heads * d->d_k + d->n_v_heads * d->d_v;
    p.q_scale = d->q_scale;
    p.eps_l2 = d->eps_l2;
    p.eps_rms = d->eps_rms;
    p.conv_w = static_cast<const uint16_t *>(w->conv_w);
    p.A_log = w->A_log;
    p.dt_bias = w->dt_bias;
    p.norm_w = static_cast<const uint16_t *>(w->norm_w);
    p.state = c->state;
    p.tail = static_cast<uint16_t *>(c->tail);
    p.n_slots = c->n_slots;
    p.mixed = static_cast<const uint16_t *>(r->mixed);
    p.z = static_cast<const uint16_t *>(r->z);
    p.a = static_cast<const uint16_t *>(r->a);
    p.b = static_cast<const uint16_t *>(r->b);
    p.y = static_cast<uint16_t *>(r->y);
    p.slot = slot;
    p.err = err;
    return p;
}

int launch_rows(int D, int mode, const gdn::RowParams &p, int n_streams, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
        case 32: e = gdn::launch_rows_d32(mode, p, n_streams, st); break;
        case 64: e = gdn::launch_rows_d64(mode, p, n_streams, st); break;
        default: e = gdn::launch_rows_d128(mode, p, n_streams, st); break;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ECUDA;
}

struct LogBuffers {
    float *a = nullptr, *u = nullptr, *k = nullptr;
};

// cuTensorMapEncodeTiled, fetched once through the runtime (the library does
// not link the driver library itself); nullptr if the driver lacks it.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Tensor map of a bf16 tensor of rank 2 or 3: dims and box innermost first,
// strides in elements for dims 1.. (the innermost is contiguous).  Zeros
// are read outside the tensor.
bool bf16_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
              const uint32_t *box) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i > 0) st[i - 1] = strides[i - 1] * 2;
    }
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The row kernel's TMA staging maps (windows and trees with d >= 64): the
// packed rows [R][CH], the committed tails [n_slots * 3][CH] and z
// [R][Hv][D], boxes of one head's D channels.
int encode_row_maps(gdn::RowParams &p, int D, int n_rows) {
    const uint64_t CH = (uint64_t)p.CH;
    p.box_rows = std::min(n_rows, (int)GDN_MAX_WINDOW);
    const uint64_t dm[2] = {CH, (uint64_t)n_rows}, sm_[1] = {CH};
    const uint32_t bm[2] = {(uint32_t)D, (uint32_t)p.box_rows};
    const uint64_t dt[2] = {CH, (uint64_t)p.n_slots * 3};
    const uint32_t bt[2] = {(uint32_t)D, 3u};
    const uint64_t dz[3] = {(uint64_t)D, (uint64_t)p.Hv, (uint64_t)n_rows}, sz[2] = {(uint64_t)D, (uint64_t)p.Hv * D};
    const uint32_t bz[3] = {(uint32_t)D, 1u, (uint32_t)p.box_rows};
    if (!bf16_map(&p.map_mixed, p.mixed, 2, dm, sm_, bm) || !bf16_map(&p.map_tail, p.tail, 2, dt, sm_, bt) ||
        !bf16_map(&p.map_z, p.z, 3, dz, sz, bz))
        return GDN_ECUDA;
    return GDN_OK;
}

int rows_entry(int mode, const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
               const int32_t *row_ptr, const int32_t *parent, int32_t n_streams, int32_t n_rows,
               const gdn_rows *rows, float *rec_state, void *rec_tail, void *stream, LogBuffers logs = {},
               const int32_t *rec_slot = nullptr, bool early_state = false) {
    GDN_TRY(check_dims(dims));
    GDN_TRY(check_weights(w));
    GDN_TRY(check_cache(cache));
    GDN_TRY(check_rows(rows));
    if (!slot) return GDN_ENULL;
    if (n_streams <= 0 || n_streams > 65535) return GDN_EINVAL;
    if (mode != gdn::kStep) {
        if (!row_ptr || !rec_tail) return GDN_ENULL;
        if (mode == gdn::kWindowLog || mode == gdn::kTreeLog) {
            if (!logs.a || !logs.u || !logs.k) return GDN_ENULL;
            if (!aligned(logs.a, 4) || !aligned(logs.u, 16) || !aligned(logs.k, 16)) return GDN_EALIGN;
        } else if (!rec_state) {
            return GDN_ENULL;
        }
        if ((mode == gdn::kTree || mode == gdn::kTreeLog) && !parent) return GDN_ENULL;
        if (n_rows <= 0) return GDN_EINVAL;
        if ((rec_state && !aligned(rec_state, 16)) || !aligned(rec_tail, 16)) return GDN_EALIGN;
    }
    if (!aligned(slot, 4) || (row_ptr && !aligned(row_ptr, 4)) || (parent && !aligned(parent, 4)))
        return GDN_EALIGN;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    gdn::RowParams p = row_params(dims, w, cache, rows, slot, err);
    p.row_ptr = row_ptr;
    p.parent = parent;
    p.n_rows = mode == gdn::kStep ? n_streams : n_rows;
    p.rec_state = rec_state;
    p.rec_tail = static_cast<uint16_t *>(rec_tail);
    p.rec_slot = rec_slot;
    p.log_a = logs.a;
    p.log_u = logs.u;
    p.log_k = logs.k;
    p.early_state = early_state ? 1 : 0;
    if (mode != gdn::kStep && dims->d_k >= 64) GDN_TRY(encode_row_maps(p, dims->d_k, n_rows));
    return launch_rows(dims->d_k, mode, p, n_streams, stream);
}

// Replay commit of chains (parent == nullptr) or trees.
int replay_entry(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot, const int32_t *row_ptr,
                 const int32_t *parent, const int32_t *keep_row, int32_t n_streams, int32_t n_rows,
                 const float *log_a, const float *log_u, const float *log_k, const void *rec_tail, void *stream) {
    GDN_TRY(check_dims(dims));
    GDN_TRY(check_cache(cache));
    if (!slot || !row_ptr || !keep_row || !log_a || !log_u || !log_k || !rec_tail) return GDN_ENULL;
    if (n_streams <= 0 || n_streams > 65535 || n_rows <= 0) return GDN_EINVAL;
    if (!aligned(slot, 4) || !aligned(row_ptr, 4) || !aligned(keep_row, 4) || !aligned(log_a, 4) ||
        !aligned(log_u, 16) || !aligned(log_k, 16) || !aligned(rec_tail, 16) || (parent && !aligned(parent, 4)))
        return GDN_EALIGN;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    gdn::ReplayParams p = {};
    p.Hk = dims->n_k_heads;
    p.Hv = dims->n_v_heads;
    p.G = dims->n_v_heads / dims->n_k_heads;
    p.CH = 2 * dims->n_k_heads * dims->d_k + dims->n_v_heads * dims->d_v;
    p.state = cache->state;
    p.tail = static_cast<uint16_t *>(cache->tail);
    p.n_slots = cache->n_slots;
    p.slot = slot;
    p.row_ptr = row_ptr;
    p.parent = parent;
    p.keep_row = keep_row;
    p.n_rows = n_rows;
    p.log_a = log_a;
    p.log_u = log_u;
    p.log_k = log_k;
    p.rec_tail = static_cast<const uint16_t *>(rec_tail);
    p.err = err;
    const dim3 grid(p.Hv, n_streams);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (parent) {
        switch (dims->d_k) {
            case 32: gdn::gdn_commit_replay_kernel<32, true><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
            case 64: gdn::gdn_commit_replay_kernel<64, true><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
            default: gdn::gdn_commit_replay_kernel<128, true><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
        }
    } else {
        switch (dims->d_k) {
            case 32: gdn::gdn_commit_replay_kernel<32><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
            case 64: gdn::gdn_commit_replay_kernel<64><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
            default: gdn::gdn_commit_replay_kernel<128><<<grid, gdn::kReplayThreads, 0, st>>>(p); break;
        }
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ECUDA;
}


}  // namespace

namespace gdn {
// gdn_prefill's host checks of everything but the workspace.
int prefill_validate(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                     const int32_t *cu_seqlens, int32_t n_seqs, int32_t n_tokens, const gdn_rows *rows,
                     int32_t chunk) {
    GDN_TRY(check_dims(dims));
    GDN_TRY(check_weights(w));
    GDN_TRY(check_cache(cache));
    GDN_TRY(check_rows(rows));
    if (!slot || !cu_seqlens) return GDN_ENULL;
    if (n_seqs <= 0 || n_seqs > 65535 || n_tokens <= 0 || n_tokens > (1 << 22) || chunk != gdn::kPrefillChunk)
        return GDN_EINVAL;
    if (!aligned(slot, 4) || !aligned(cu_seqlens, 4)) return GDN_EALIGN;
    if ((size_t)n_tokens / chunk + (size_t)n_seqs > 65535) return GDN_EINVAL;
    return GDN_OK;
}

// gdn_prefill with a choice of launch plan (see launch_prefill).
int prefill_entry(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                  const int32_t *cu_seqlens, int32_t n_seqs, int32_t n_tokens, const gdn_rows *rows, int32_t chunk,
                  void *workspace, size_t workspace_bytes, void *stream, bool pipelined) {
    GDN_TRY(prefill_validate(dims, w, cache, slot, cu_seqlens, n_seqs, n_tokens, rows, chunk));
    const size_t need = gdn_prefill_workspace_size(dims, n_seqs, n_tokens, chunk);
    if (!workspace || workspace_bytes < need) return GDN_EWORKSPACE;
    if (!aligned(workspace, 16)) return GDN_EALIGN;
    const size_t max_chunks = (size_t)n_tokens / chunk + (size_t)n_seqs;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    gdn::PrefillParams p = {};
    p.Hk = dims->n_k_heads;
    p.Hv = dims->n_v_heads;
    p.G = dims->n_v_heads / dims->n_k_heads;
    p.CH = 2 * dims->n_k_heads * dims->d_k + dims->n_v_heads * dims->d_v;
    p.q_scale = dims->q_scale;
    p.eps_l2 = dims->eps_l2;
    p.eps_rms = dims->eps_rms;
    p.conv_w = static_cast<const uint16_t *>(w->conv_w);
    p.A_log = w->A_log;
    p.dt_bias = w->dt_bias;
    p.norm_w = static_cast<const uint16_t *>(w->norm_w);
    p.state = cache->state;
    p.tail = static_cast<uint16_t *>(cache->tail);
    p.n_slots = cache->n_slots;
    p.mixed = static_cast<const uint16_t *>(rows->mixed);
    p.z = static_cast<const uint16_t *>(rows->z);
    p.a = static_cast<const uint16_t *>(rows->a);
    p.b = static_cast<const uint16_t *>(rows->b);
    p.y = static_cast<uint16_t *>(rows->y);
    p.slot = slot;
    p.cu_seqlens = cu_seqlens;
    p.n_seqs = n_seqs;
    p.n_tokens = n_tokens;
    p.max_chunks = (int)max_chunks;
    p.ws_chunks = static_cast<float *>(workspace);
    p.ws_out = p.ws_chunks + max_chunks * dims->n_v_heads * gdn::prefill_chunk_floats(dims->d_k);
    p.err = err;
    return gdn::launch_prefill(dims->d_k, p, static_cast<cudaStream_t>(stream), pipelined) == cudaSuccess
               ? GDN_OK
               : GDN_ECUDA;
}
}  // namespace gdn

extern "C" {

int gdn_step(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
             int32_t n_streams, const gdn_rows *rows, void *stream) {
    return rows_entry(gdn::kStep, dims, w, cache, slot, nullptr, nullptr, n_streams, n_streams, rows, nullptr,
                      nullptr, stream);
}

int gdn_step_ex(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                int32_t n_streams, const gdn_rows *rows, uint32_t flags, void *stream) {
    if (flags & ~(uint32_t)GDN_STEP_EARLY_STATE) return GDN_EINVAL;
    return rows_entry(gdn::kStep, dims, w, cache, slot, nullptr, nullptr, n_streams, n_streams, rows, nullptr,
                      nullptr, stream, LogBuffers{}, nullptr, (flags & GDN_STEP_EARLY_STATE) != 0);
}

int gdn_window(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
               const int32_t *row_ptr, int32_t n_streams, int32_t n_rows, const gdn_rows *rows, float *rec_state,
               void *rec_tail, void *stream) {
    return rows_entry(gdn::kWindow, dims, w, cache, slot, row_ptr, nullptr, n_streams, n_rows, rows, rec_state,
                      rec_tail, stream);
}

int gdn_tree(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
             const int32_t *row_ptr, const int32_t *parent, int32_t n_streams, int32_t n_rows,
             const gdn_rows *rows, float *rec_state, void *rec_tail, void *stream) {
    return rows_entry(gdn::kTree, dims, w, cache, slot, row_ptr, parent, n_streams, n_rows, rows, rec_state,
                      rec_tail, stream);
}

int gdn_window_pooled(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                      const int32_t *row_ptr, int32_t n_streams, int32_t n_rows, const gdn_rows *rows,
                      const int32_t *rec_slot, void *stream) {
    if (!cache) return GDN_ENULL;
    if (!rec_slot) return GDN_ENULL;
    if (!aligned(rec_slot, 4)) return GDN_EALIGN;
    return rows_entry(gdn::kWindow, dims, w, cache, slot, row_ptr, nullptr, n_streams, n_rows, rows, cache->state,
                      cache->tail, stream, LogBuffers{}, rec_slot);
}

int gdn_tree_pooled(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                    const int32_t *row_ptr, const int32_t *parent, int32_t n_streams, int32_t n_rows,
                    const gdn_rows *rows, const int32_t *rec_slot, void *stream) {
    if (!cache) return GDN_ENULL;
    if (!rec_slot) return GDN_ENULL;
    if (!aligned(rec_slot, 4)) return GDN_EALIGN;
    return rows_entry(gdn::kTree, dims, w, cache, slot, row_ptr, parent, n_streams, n_rows, rows, cache->state,
                      cache->tail, stream, LogBuffers{}, rec_slot);
}

int gdn_commit_swap(const gdn_dims *dims, const gdn_cache *cache, int32_t *slot, const int32_t *row_ptr,
                    const int32_t *keep_row, const int32_t *rec_slot, int32_t n_streams, int32_t n_rows,
                    int32_t *freed, void *stream) {
    GDN_TRY(check_dims(dims));
    GDN_TRY(check_cache(cache));
    if (!slot || !row_ptr || !keep_row || !rec_slot) return GDN_ENULL;
    if (n_streams <= 0 || n_streams > 65535 || n_rows <= 0) return GDN_EINVAL;
    if (!aligned(slot, 4) || !aligned(row_ptr, 4) || !aligned(keep_row, 4) || !aligned(rec_slot, 4) ||
        (freed && !aligned(freed, 4)))
        return GDN_EALIGN;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    gdn::SwapParams p = {};
    p.slot = slot;
    p.row_ptr = row_ptr;
    p.keep_row = keep_row;
    p.rec_slot = rec_slot;
    p.freed = freed;
    p.n_streams = n_streams;
    p.n_rows = n_rows;
    p.n_slots = cache->n_slots;
    p.err = err;
    // a programmatic dependent of the kernel before it: scheduled early, it
    // waits (griddepcontrol.wait) before reading anything that kernel writes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n_streams + gdn::kSwapThreads - 1) / gdn::kSwapThreads));
    cfg.blockDim = dim3(gdn::kSwapThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gdn::gdn_commit_swap_kernel, p) == cudaSuccess ? GDN_OK : GDN_ECUDA;
}

int gdn_commit(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot, const int32_t *row_ptr,
               const int32_t *keep_row, int32_t n_streams, int32_t n_rows, const float *rec_state,
               const void *rec_tail, void *stream) {
    GDN_TRY(check_dims(dims));
    GDN_TRY(check_cache(cache));
    if (!slot || !row_ptr || !keep_row || !rec_state || !rec_tail) return GDN_ENULL;
    if (n_streams <= 0 || n_streams > 65535 || n_rows <= 0) return GDN_EINVAL;
    if (!aligned(slot, 4) || !aligned(row_ptr, 4) || !aligned(keep_row, 4) || !aligned(rec_state, 16) ||
        !aligned(rec_tail, 16))
        return GDN_EALIGN;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    gdn::CommitParams p = {};
    p.Hv = dims->n_v_heads;
    p.D = dims->d_k;
    p.CH = 2 * dims->n_k_heads * dims->d_k + dims->n_v_heads * dims->d_v;
    p.state = cache->state;
    p.tail = static_cast<uint16_t *>(cache->tail);
    p.n_slots = cache->n_slots;
    p.slot = slot;
    p.row_ptr = row_ptr;
    p.keep_row = keep_row;
    p.n_rows = n_rows;
    p.rec_state = rec_state;
    p.rec_tail = static_cast<const uint16_t *>(rec_tail);
    p.err = err;
    const dim3 grid(p.Hv, n_streams);
    gdn::gdn_commit_kernel<<<grid, gdn::kCommitThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ECUDA;
}

size_t gdn_prefill_workspace_size(const gdn_dims *dims, int32_t n_seqs, int32_t n_tokens, int32_t chunk) {
    if (check_dims(dims) != GDN_OK || n_seqs <= 0 || n_tokens <= 0 || n_tokens > (1 << 22) ||
        chunk != gdn::kPrefillChunk)
        return 0;
    const size_t max_chunks = (size_t)n_tokens / chunk + (size_t)n_seqs;
    const size_t floats = max_chunks * dims->n_v_heads * gdn::prefill_chunk_floats(dims->d_k) +
                          (size_t)n_tokens * dims->n_v_heads * dims->d_v;
    return floats * sizeof(float);
}

size_t gdn_prefill_workspace(const gdn_dims *dims, int32_t n_seqs, int32_t n_tokens, int32_t chunk) {
    return gdn_prefill_workspace_size(dims, n_seqs, n_tokens, chunk);
}

int gdn_prefill(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                const int32_t *cu_seqlens, int32_t n_seqs, int32_t n_tokens, const gdn_rows *rows, int32_t chunk,
                void *workspace, size_t workspace_bytes, void *stream) {
    return gdn::prefill_entry(dims, w, cache, slot, cu_seqlens, n_seqs, n_tokens, rows, chunk, workspace,
                              workspace_bytes, stream, true);
}


int gdn_window_log(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                   const int32_t *row_ptr, int32_t n_streams, int32_t n_rows, const gdn_rows *rows, float *log_a,
                   float *log_u, float *log_k, void *rec_tail, void *stream) {
    LogBuffers logs;
    logs.a = log_a;
    logs.u = log_u;
    logs.k = log_k;
    return rows_entry(gdn::kWindowLog, dims, w, cache, slot, row_ptr, nullptr, n_streams, n_rows, rows, nullptr,
                      rec_tail, stream, logs);
}

int gdn_commit_replay(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot, const int32_t *row_ptr,
                      const int32_t *keep_row, int32_t n_streams, int32_t n_rows, const float *log_a,
                      const float *log_u, const float *log_k, const void *rec_tail, void *stream) {
    return replay_entry(dims, cache, slot, row_ptr, nullptr, keep_row, n_streams, n_rows, log_a, log_u, log_k,
                        rec_tail, stream);
}

int gdn_tree_log(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache, const int32_t *slot,
                 const int32_t *row_ptr, const int32_t *parent, int32_t n_streams, int32_t n_rows,
                 const gdn_rows *rows, float *log_a, float *log_u, float *log_k, void *rec_tail, void *stream) {
    LogBuffers logs;
    logs.a = log_a;
    logs.u = log_u;
    logs.k = log_k;
    return rows_entry(gdn::kTreeLog, dims, w, cache, slot, row_ptr, parent, n_streams, n_rows, rows, nullptr,
                      rec_tail, stream, logs);
}

int gdn_commit_replay_tree(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot,
                           const int32_t *row_ptr, const int32_t *parent, const int32_t *keep_row,
                           int32_t n_streams, int32_t n_rows, const float *log_a, const float *log_u,
                           const float *log_k, const void *rec_tail, void *stream) {
    if (!parent) return GDN_ENULL;
    return replay_entry(dims, cache, slot, row_ptr, parent, keep_row, n_streams, n_rows, log_a, log_u, log_k,
                        rec_tail, stream);
}

int gdn_debug_wait_timeout(uint32_t polls, void *stream) {
    if (polls > (1u << 22)) return GDN_EINVAL;
    int *err = error_word();
    if (!err) return GDN_ECUDA;
    return gdn::launch_wait_selftest(polls, err, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK
                                                                                                   : GDN_ECUDA;
}

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_EINVAL: return "invalid size or geometry";
        case GDN_ENULL: return "required pointer is NULL";
        case GDN_EALIGN: return "pointer misaligned";
        case GDN_ECUDA: return "CUDA runtime error";
        case GDN_EWORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int gdn_get_device_error(void *stream, int32_t *bits) {
    if (!bits) return GDN_ENULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int value = 0;
    static const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&value, g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GDN_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ECUDA;
    if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return GDN_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ECUDA;
    *bits = value;
    return GDN_OK;
}

}  // extern "C"
