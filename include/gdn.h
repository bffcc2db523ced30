/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated-DeltaNet verify path.
 *
 * One GDN linear-attention layer's core, after its input projection and
 * before its output projection: causal depthwise conv1d (width 4) with a
 * kept tail, SiLU, L2-normalised q and k, the gated delta rule
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t,
 *     a_t = exp(-exp(A_log) * softplus(a + dt_bias)),  b_t = sigmoid(b),
 * and the gated RMSNorm  y = RMSNorm(o) * w_norm * SiLU(z).
 *
 * Sources, by page:
 *  [P932]  TensorFold #932, titled "perf(qwen3_5 cuda): deliver the first
 *          token before drafting".  Its commit notes on the Qwen3.5 CUDA
 *          engine:
 *          - the note on the MLX affine 4-bit checkpoint: the layer's glue
 *            is a causal conv and the gated delta rule; a verify window of
 *            at most 16 rows keeps every row's state and conv tail, and
 *            each of its rows must match the same row run as a single step,
 *            bit for bit;
 *          - the note on the 2B engine's widths: fewer key heads than value
 *            heads, one A_log per value head;
 *          - the tree note: a window's rows can form a tree given by each
 *            row's parent, the conv taps and the recurrence following each
 *            row's own branch; single steps and prompts write the slot
 *            directly.
 *  [P747]  TensorFold #747, titled "perf(qwen27 cuda): reduce repeated-prompt
 *          TTFT", first commit note: one verify round serves the windows of
 *          all streams (at most 16 streams of 16 rows) and keeps only each
 *          stream's accepted rows; the engine has kernels for trees, for
 *          replays and for prompts, and prompts that come in together are
 *          prefilled in one pass.
 *  [P888]  TensorFold #888, titled "Qwen3.5/3.8 on CUDA: kept prompt states
 *          in host memory": a kept state is the full recurrent state of a
 *          stream together with its conv history.
 *
 * Conventions shared by every entry point
 *  - Every pointer argument named "device" is a CUDA device pointer owned by
 *    the caller; the library allocates no device memory at run time, frees
 *    nothing and keeps no state between calls except, per device: the
 *    address of its device error word and the SM count; the driver's
 *    tensor-map encoder (looked up once, for the TMA staging of windows and
 *    trees); the d = 128 prefill's two side streams and four events (see
 *    gdn_prefill); and gdn_prefill_noalloc's fixed scratch array, a
 *    module-scope device array reserved wherever the module is loaded, with
 *    its cached device address (see gdn_prefill_noalloc).  Cached device
 *    addresses are looked up again after the device's context is destroyed
 *    and made anew (cudaDeviceReset).
 *    All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and the call returns without synchronising.  Windows
 *    and trees of d >= 64 encode three tensor maps on the host per call
 *    (host work only, nothing is enqueued for it).
 *  - bf16 is IEEE bfloat16 (raw 16-bit storage); fp32 is IEEE binary32.
 *    Internally everything is fp32; y is rounded to bf16 (nearest even) once.
 *  - Geometry: Hk key heads, Hv value heads (Hv % Hk == 0, G = Hv/Hk <= 8),
 *    d_k == d_v in {32, 64, 128}, conv width 4.  CH = 2*Hk*d_k + Hv*d_v is
 *    the number of conv channels, laid out [q | k | v], head-major inside
 *    each block.  Value head h reads key head h / G.
 *  - State tiles are [d_v, d_k] fp32, row-major (row = value channel).
 *  - The conv tail of a slot is [3, CH] bf16: the three previous pre-conv
 *    inputs of its stream, oldest first.  Conv tap w[c][3] multiplies the
 *    current row, w[c][0] the input three rows back.  No conv bias.
 *  - Every pointer must be 16-byte aligned (GDN_EALIGN otherwise), except
 *    a, b, slot, row_ptr, parent, keep_row, cu_seqlens (4-byte / element
 *    alignment).
 *  - Errors: every size, geometry and pointer is validated on the host
 *    BEFORE anything is enqueued; an error return leaves every buffer
 *    untouched.  Device-resident indices (slot, row_ptr, parent, keep_row,
 *    cu_seqlens) are checked by the kernels: an out-of-range value sets a
 *    bit in the device error word (read with gdn_get_device_error) and the
 *    affected stream is skipped (its outputs are left unwritten).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GDN_OK          0
#define GDN_EINVAL     -1   /* a size or geometry outside the supported set */
#define GDN_ENULL      -2   /* a required pointer is NULL */
#define GDN_EALIGN     -3   /* a pointer misses its required alignment */
#define GDN_ECUDA      -4   /* the CUDA runtime refused the launch */
#define GDN_EWORKSPACE -5   /* workspace missing or smaller than required */

/* ---- device error word bits (gdn_get_device_error) --------------------- */
#define GDN_DERR_SLOT      1   /* slot[s] outside [0, n_slots) */
#define GDN_DERR_ROWS      2   /* row_ptr not monotone, > n_rows, or > 16 rows */
#define GDN_DERR_PARENT    4   /* parent[i] outside [-1, i) (window-local) */
#define GDN_DERR_KEEP      8   /* keep_row[s] not -1 and not one of stream s's rows */
#define GDN_DERR_SEQLENS  16   /* cu_seqlens not monotone or > n_tokens */
#define GDN_DERR_TIMEOUT  32   /* a bounded wait inside a kernel gave up */

#define GDN_MAX_WINDOW 16      /* rows per stream in one window or tree */

typedef struct {
    int32_t n_k_heads;  /* Hk */
    int32_t n_v_heads;  /* Hv, a multiple of Hk, Hv / Hk <= 8 */
    int32_t d_k;        /* key head width, equal to d_v, in {32, 64, 128} */
    int32_t d_v;        /* value head width */
    int32_t conv_width; /* must be 4 */
    float q_scale;      /* q is multiplied by this after its L2 norm */
    float eps_l2;       /* q, k <- x / sqrt(sum x^2 + eps_l2) */
    float eps_rms;      /* RMSNorm: o / sqrt(mean o^2 + eps_rms) */
} gdn_dims;

typedef struct {
    const void *conv_w;    /* device, bf16 [CH, 4] */
    const float *A_log;    /* device, fp32 [Hv] */
    const float *dt_bias;  /* device, fp32 [Hv] */
    const void *norm_w;    /* device, bf16 [d_v], shared by all heads */
} gdn_weights;

typedef struct {
    float *state;          /* device, fp32 [n_slots, Hv, d_v, d_k] committed states */
    void *tail;            /* device, bf16 [n_slots, 3, CH] committed conv tails */
    int32_t n_slots;
} gdn_cache;

typedef struct {
    const void *mixed;     /* device, bf16 [R, CH] conv inputs (in_proj q|k|v) */
    const void *z;         /* device, bf16 [R, Hv, d_v] output gate */
    const void *a;         /* device, bf16 [R, Hv] decay input */
    const void *b;         /* device, bf16 [R, Hv] beta input */
    void *y;               /* device, bf16 [R, Hv, d_v] output */
} gdn_rows;

/*
 * gdn_step -- one row per stream, in place ([P932] tree note: one-row steps
 * update in place).  Row s of `rows` belongs to stream s and advances the
 * committed state and tail of slot[s]; y[s] is written.
 *   slot      device int32 [n_streams], distinct values in [0, n_slots)
 *   n_streams >= 1 (<= 65535)
 * Launch: one CTA per (value head, stream), each head's state rows split
 * over up to 8 CTAs when few streams would leave SMs idle, clusters of the
 * key head's value heads.  The launch is a programmatic dependent of the
 * kernel before it on `stream`: its CTAs may be scheduled while that kernel
 * finishes, but touch no memory until it has completed, so ordering is that
 * of a plain launch (back-to-back steps, e.g. layer after layer in a graph,
 * overlap only their launch gaps).
 */
int gdn_step(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
             const int32_t *slot, int32_t n_streams, const gdn_rows *rows,
             void *stream);

/* Flags of gdn_step_ex. */
#define GDN_STEP_EARLY_STATE 1u

/*
 * gdn_step_ex -- gdn_step with launch flags (not in the pages: a latency
 * option of the layer loop that [P932]'s note on capturing a forward's
 * launches is about).
 *   flags  0: exactly gdn_step.
 *          GDN_STEP_EARLY_STATE: the caller promises that the kernel launched
 *          just before this one on `stream` writes none of slot[], the
 *          state and tail entries slot[] names, and the weights (true, for
 *          example, of a step of another layer: its own cache, or other
 *          entries of a shared one).  The step's CTAs
 *          then read the slot words, their rows of the state tile, the
 *          committed tail and the weights while that kernel finishes, and
 *          only the rows' inputs (mixed, z, a, b) after it; its writes (the
 *          state and tail in place, y) still wait for it.  The results are
 *          those of gdn_step, bit for bit.  A broken promise gives wrong
 *          results (stale state), never a fault.
 *          Any other bit: GDN_EINVAL.
 */
int gdn_step_ex(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                const int32_t *slot, int32_t n_streams, const gdn_rows *rows,
                uint32_t flags, void *stream);

/*
 * gdn_window -- chain verify windows (at most 16 rows a stream), recorded
 * row by row ([P932] MLX checkpoint note: every row's state and conv tail
 * are kept; [P747] one round for at most 16 streams x 16 rows).  Stream s owns packed rows [row_ptr[s], row_ptr[s+1]) of `rows`;
 * its first row follows the committed state and tail of slot[s], each later
 * row the row before it.  The committed slot is NOT modified.
 *   slot       device int32 [n_streams]
 *   row_ptr    device int32 [n_streams + 1], non-decreasing, row_ptr[s+1] -
 *              row_ptr[s] <= 16, row_ptr[n_streams] <= n_rows; a stream with
 *              no rows is skipped
 *   n_rows     R, rows in the packed buffers (>= 1)
 *   rec_state  device fp32 [R, Hv, d_v, d_k]: the state after each row
 *   rec_tail   device bf16 [R, 3, CH]: the tail after each row (the three
 *              newest conv inputs along the row's branch, oldest first)
 * Row r of y, rec_state and rec_tail equals, bit for bit, what gdn_step
 * would produce for that row from the state and tail it follows.
 * Launch: one CTA per (value head, stream); when those would leave SMs
 * idle (few streams), each head's state rows are split over a cluster of
 * 2 to 8 CTAs, with the same bits.  d >= 64 without that split stages the
 * inputs with TMA (three tensor maps encoded on the host per call).  Every
 * CTA signals programmatic dependents when it starts, so a kernel launched
 * after it as one (gdn_commit_swap) is scheduled early and waits for the
 * window's end; a plain launch after it is unaffected.
 */
int gdn_window(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
               const int32_t *slot, const int32_t *row_ptr, int32_t n_streams,
               int32_t n_rows, const gdn_rows *rows, float *rec_state,
               void *rec_tail, void *stream);

/*
 * gdn_tree -- tree verify windows ([P932] tree note: a row's parent is
 * given, and its conv taps and recurrence follow its own branch).  As
 * gdn_window, plus
 *   parent  device int32 [n_rows]: for packed row r of stream s, the
 *           window-local index (0-based within the stream's rows) of its
 *           parent, which must be smaller than its own index, or -1 for a
 *           row that follows the committed slot.
 * A row whose parent is the row before it continues from registers; any
 * other parent's state is re-read from rec_state.  A node's outputs equal
 * gdn_window's on the chain of rows along its root-to-node path.
 */
int gdn_tree(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
             const int32_t *slot, const int32_t *row_ptr, const int32_t *parent,
             int32_t n_streams, int32_t n_rows, const gdn_rows *rows,
             float *rec_state, void *rec_tail, void *stream);

/*
 * gdn_commit -- keep each stream's accepted path ([P747] first note: each
 * stream keeps only its accepted rows; [P932] MLX checkpoint note: the
 * recorded rows are what let a partially accepted window be kept).
 * For stream s with keep_row[s] = r >= 0 (a packed row index, normally the
 * last accepted row of the stream's window or the chosen tree node),
 * slot[s]'s state and tail become rec_state[r] and rec_tail[r].
 * keep_row[s] = -1 (nothing accepted) leaves the slot bit-unchanged.
 *   slot       device int32 [n_streams], distinct
 *   row_ptr    device int32 [n_streams + 1], the row_ptr the window or tree
 *              call took: stream s may keep only one of its own rows
 *   keep_row   device int32 [n_streams], each -1 or in
 *              [row_ptr[s], row_ptr[s+1]); anything else (a row of another
 *              stream's window, or past n_rows) sets GDN_DERR_KEEP and
 *              leaves that stream's slot bit-unchanged
 *   rec_state, rec_tail  as written by gdn_window / gdn_tree
 */
int gdn_commit(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot,
               const int32_t *row_ptr, const int32_t *keep_row, int32_t n_streams,
               int32_t n_rows, const float *rec_state, const void *rec_tail, void *stream);

/*
 * gdn_window_pooled, gdn_tree_pooled -- gdn_window / gdn_tree recording each
 * row in the cache itself, so that committing a row is a change of index
 * instead of a copy ([P747] first note: each stream keeps only its accepted
 * rows; [P932] MLX checkpoint note: only the accepted path is kept, so the
 * kept row's record can simply become the slot).  The cache is then a pool
 * of entries, some holding committed states (named by slot[]), the others
 * free.  Row r's state and tail go to entry rec_slot[r] of cache->state and
 * cache->tail, bit for bit what gdn_window / gdn_tree write to rec_state[r]
 * and rec_tail[r]; y is the same too.
 *   rec_slot  device int32 [n_rows]: pool entries in [0, n_slots), distinct
 *             from each other and from every slot[s] of the call (the
 *             library checks only that each is in range and is not its own
 *             stream's slot: otherwise GDN_DERR_SLOT and the stream is
 *             skipped).  Entries the caller no longer needs (the rows it does
 *             not keep) are free again after the commit.
 * Everything else as gdn_window / gdn_tree.
 */
int gdn_window_pooled(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                      const int32_t *slot, const int32_t *row_ptr, int32_t n_streams,
                      int32_t n_rows, const gdn_rows *rows, const int32_t *rec_slot, void *stream);
int gdn_tree_pooled(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                    const int32_t *slot, const int32_t *row_ptr, const int32_t *parent,
                    int32_t n_streams, int32_t n_rows, const gdn_rows *rows,
                    const int32_t *rec_slot, void *stream);

/*
 * gdn_commit_swap -- commit after gdn_window_pooled / gdn_tree_pooled: for
 * stream s with keep_row[s] = r in [row_ptr[s], row_ptr[s+1]), slot[s]
 * becomes rec_slot[r] (the entry that already holds row r's state and tail)
 * and freed[s] receives the stream's previous entry; keep_row[s] = -1 leaves
 * slot[s] as it is and sets freed[s] = -1.  One small kernel, no state or
 * tail is moved; it is launched as a programmatic dependent of the kernel
 * before it on `stream` (scheduled early, it reads nothing before that
 * kernel has completed).
 *   slot      device int32 [n_streams], read and written
 *   row_ptr, keep_row  as gdn_commit
 *   rec_slot  device int32 [n_rows], as given to the pooled window or tree
 *   freed     device int32 [n_streams] or NULL
 * A keep_row outside the stream's rows sets GDN_DERR_KEEP, a rec_slot[r]
 * outside [0, n_slots) or equal to slot[s] sets GDN_DERR_SLOT; either
 * leaves slot[s] as it is (freed[s] = -1).
 */
int gdn_commit_swap(const gdn_dims *dims, const gdn_cache *cache, int32_t *slot,
                    const int32_t *row_ptr, const int32_t *keep_row, const int32_t *rec_slot,
                    int32_t n_streams, int32_t n_rows, int32_t *freed, void *stream);

/*
 * gdn_prefill -- chunked prompt prefill ([P747] the engine's prompt kernel,
 * several prompts prefilled in one pass; [P932] tree note: a prompt writes
 * its slot directly).  Sequence s owns packed tokens
 * [cu_seqlens[s], cu_seqlens[s+1]) of `rows`; it starts from slot[s]'s
 * committed state and tail (zero them for a fresh prompt; a nonzero state
 * resumes a kept one) and leaves the state and tail after its last token
 * in the slot.  y is written for every token of a sequence; rows of the
 * packed buffers outside every sequence (before cu_seqlens[0] or from
 * cu_seqlens[n_seqs] on) are neither read nor written.  The result equals
 * running the tokens through gdn_step one by one, up to fp32 rounding (the
 * chunked form reorders the sums).
 *   cu_seqlens  device int32 [n_seqs + 1], non-decreasing, last <= n_tokens;
 *               empty sequences leave their slot untouched
 *   n_tokens    rows in the packed buffers (>= 1, <= 2^22)
 *   chunk       rows per chunk; must be 64
 *   workspace   device scratch of at least gdn_prefill_workspace_size()
 *               bytes, 16-byte aligned; its contents on entry do not
 *               matter and are garbage on return; GDN_EWORKSPACE if absent
 *               or too small
 * Launches: prep (chunk x head), scan (sequence x head; for d < 128 also
 * x d_v slice) and norm (token x head).  They run after the work enqueued
 * on `stream` before the call, and work enqueued on `stream` after the call
 * runs after them, so the call behaves as if all of it were on `stream`.
 * For d = 128 the chunks are taken in groups: prep of a group runs on
 * `stream`, its scan on a highest-priority side stream and its norm on a
 * third stream of the library (two streams and four events per device,
 * made by the first such call on that device), forked from and joined back
 * to `stream` by events, so they overlap the prep of later groups.  With
 * one sequence the groups are sized in whole prep rounds of the SMs and
 * every prep after the first leaves the scan's SMs free; with several they
 * shrink toward the end (about 75% of the chunks left each, at least 4).
 * The side streams are shared: calls made from several host threads at
 * once are serialised on them.  The fork and join are ordinary event
 * record / wait calls, so the call can be captured in a CUDA graph.
 */
int gdn_prefill(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                const int32_t *slot, const int32_t *cu_seqlens, int32_t n_seqs,
                int32_t n_tokens, const gdn_rows *rows, int32_t chunk,
                void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace gdn_prefill needs for these sizes (0 if invalid). */
size_t gdn_prefill_workspace_size(const gdn_dims *dims, int32_t n_seqs, int32_t n_tokens,
                                  int32_t chunk);
/* The same size under its shorter name (identical result). */
size_t gdn_prefill_workspace(const gdn_dims *dims, int32_t n_seqs, int32_t n_tokens, int32_t chunk);

/*
 * gdn_prefill_noalloc -- gdn_prefill without a workspace argument, for
 * callers that cannot allocate device memory (a host runtime whose pool owns
 * the device, a serving loop that must not pay cudaMalloc's device-wide
 * synchronisation, a plugin interface with no scratch argument).  The
 * source pages have no counterpart to this entry point.
 *   The scratch is a file-scope device array of
 *   GDN_PREFILL_NOALLOC_SCRATCH_BYTES (64 MiB), reserved on every GPU where
 *   the library's module is loaded until the process exits.  Sizes whose
 *   gdn_prefill_workspace_size() exceeds it return GDN_EWORKSPACE before
 *   anything is enqueued; other arguments are validated as in gdn_prefill.
 *   The first call on a device (and the first after that device's context
 *   was destroyed and made anew) looks up the array's device address once
 *   its arguments have passed the host checks; the lookup may load the
 *   module, so make that call before any stream capture.  All calls share
 *   the array: calls whose work overlaps on the GPU race and must be
 *   serialised by the caller.  Nothing in the array needs to start at zero:
 *   a call reads only what it wrote itself.  No cudaMalloc or cudaFree is
 *   made, and no stream or event is created: every launch goes on `stream`.
 */
#define GDN_PREFILL_NOALLOC_SCRATCH_BYTES (64u << 20)
int gdn_prefill_noalloc(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                        const int32_t *slot, const int32_t *cu_seqlens, int32_t n_seqs,
                        int32_t n_tokens, const gdn_rows *rows, int32_t chunk, void *stream);

/*
 * gdn_window_log -- chain verify windows that log instead of record
 * ([P932] tree note: keeping a state per row took 1.3 GB and limited the
 * 27B to 8-row windows, so each row now leaves a log of its decay, write
 * vector and key, and the commit replays the accepted rows).  As gdn_window (same y and rec_tail, bit for bit), but in
 * place of rec_state it writes, for every row r:
 *   log_a  device fp32 [R, Hv]         the decay a_r
 *   log_u  device fp32 [R, Hv, d_v]    the write u_r = b_r (v_r - a_r S_{r-1} k_r)
 *   log_k  device fp32 [R, Hk, d_k]    the normalised key k_r (per key head)
 * so that S_r = a_r S_{r-1} + u_r k_r^T.  About 1 KiB per row and head
 * instead of 64 KiB.
 */
int gdn_window_log(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                   const int32_t *slot, const int32_t *row_ptr, int32_t n_streams,
                   int32_t n_rows, const gdn_rows *rows, float *log_a, float *log_u,
                   float *log_k, void *rec_tail, void *stream);

/*
 * gdn_commit_replay -- commit after gdn_window_log: for stream s with
 * keep_row[s] = r in [row_ptr[s], row_ptr[s+1]), the slot's state is
 * advanced along rows row_ptr[s] .. r with S <- a S + u k^T, in the window's
 * own rounding, so it equals bit for bit what gdn_window would have recorded
 * for row r; the tail becomes rec_tail[r].  keep_row[s] = -1 leaves the
 * slot bit-unchanged.  Slots must be distinct.
 */
int gdn_commit_replay(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot,
                      const int32_t *row_ptr, const int32_t *keep_row, int32_t n_streams,
                      int32_t n_rows, const float *log_a, const float *log_u,
                      const float *log_k, const void *rec_tail, void *stream);

/*
 * gdn_tree_log -- tree verify windows that log instead of record ([P932]
 * tree note: the per-row logs of the decay, the write vector and the key,
 * and the replay of the kept path, serve trees as well as chains).  As
 * gdn_tree (same y and rec_tail, bit for bit), with gdn_window_log's logs
 * (log_a [R, Hv], log_u [R, Hv, d_v], log_k [R, Hk, d_k]) in place of
 * rec_state, so that S_r = a_r S_parent(r) + u_r k_r^T.  A node whose parent
 * is not the node visited just before it (nodes are visited depth first,
 * children in row order) rebuilds its parent's state from the committed
 * slot by re-applying the logged rows of the root-to-parent path with the
 * forward pass's rounding, so every state, and y, equals gdn_tree's bit for
 * bit.  parent is as in gdn_tree.
 */
int gdn_tree_log(const gdn_dims *dims, const gdn_weights *w, const gdn_cache *cache,
                 const int32_t *slot, const int32_t *row_ptr, const int32_t *parent,
                 int32_t n_streams, int32_t n_rows, const gdn_rows *rows, float *log_a,
                 float *log_u, float *log_k, void *rec_tail, void *stream);

/*
 * gdn_commit_replay_tree -- commit after gdn_tree_log: for stream s with
 * keep_row[s] = r in [row_ptr[s], row_ptr[s+1]) (the chosen node), the
 * slot's state is advanced along the node's root-to-node path (found
 * through `parent`, the same device array gdn_tree_log took), root first,
 * with S <- a S + u k^T in the window's own rounding, so it equals bit for
 * bit what gdn_tree would have recorded for node r; the tail becomes
 * rec_tail[r].  keep_row[s] = -1 leaves the slot bit-unchanged.  A parent
 * index on the path outside [-1, its own index) sets GDN_DERR_PARENT and
 * skips the stream.  Slots must be distinct.
 */
int gdn_commit_replay_tree(const gdn_dims *dims, const gdn_cache *cache, const int32_t *slot,
                           const int32_t *row_ptr, const int32_t *parent,
                           const int32_t *keep_row, int32_t n_streams, int32_t n_rows,
                           const float *log_a, const float *log_u, const float *log_k,
                           const void *rec_tail, void *stream);

/*
 * gdn_debug_wait_timeout -- a test hook for the failure path of the bounded
 * waits (no source passage; the pages name no such check).  Every wait of
 * the prefill kernels on an mbarrier polls a fixed number of times; if the
 * phase has not completed by then, the kernel sets GDN_DERR_TIMEOUT in the
 * device error word, waits (again bounded) for anything it has in flight,
 * and leaves, so a lost copy or MMA completion ends as an error status, not
 * a hang.  This call launches one CTA that runs that same wait on an
 * mbarrier nothing will ever complete, with nothing in flight: after
 * `polls` polls (at most 2^22; GDN_EINVAL above) it sets GDN_DERR_TIMEOUT
 * and returns, and the context stays usable.  Read the bit with
 * gdn_get_device_error.
 */
int gdn_debug_wait_timeout(uint32_t polls, void *stream);

/* Text for a status code (static storage). */
const char *gdn_status_string(int status);

/*
 * Reads and clears the calling device's error word on `stream` (this call
 * synchronises that stream).  *bits receives the OR of GDN_DERR_* flags
 * raised since the last read.  Returns GDN_OK or GDN_ECUDA.
 */
int gdn_get_device_error(void *stream, int32_t *bits);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
