/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential CPU reference for the gated-DeltaNet (GDN) layer
 * core used in speculative verification.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no source, header, table or constant with the CUDA library, and it never
 * reads anything the CUDA library produced.
 *
 * Sources of the operation (cited by page title and passage):
 *  - TensorFold #932 "deliver the first token before drafting", commit note
 *    on the MLX checkpoint for the CUDA engine: the layer's glue is a causal
 *    conv and the gated delta rule; a verify window (at most 16 rows) keeps
 *    every row's state and conv tail, and its rows must match single steps.
 *  - Same page, note on the 2B reading its widths from config.json: more
 *    linear value heads than key heads (grouped heads).
 *  - Same page, note on tree windows: each row has a parent, and the
 *    conv taps and the recurrence follow the row's own branch.
 *  - TensorFold #747 "reduce repeated-prompt TTFT", first commit note: one
 *    verify round serves at most 16 streams of 16 rows, and each stream
 *    keeps only its accepted rows.
 *  - The layer's arithmetic (the gated-DeltaNet layer of this model family):
 *      conv1d width 4 with a kept tail, SiLU, L2-normalised q and k,
 *      S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t,
 *      a_t = exp(-exp(A_log) * softplus(a + dt_bias)),  b_t = sigmoid(b),
 *      y = RMSNorm(o) * SiLU(z).
 *
 * Everything is computed in double precision from the bf16 / fp32 inputs,
 * with no rounding anywhere in between and no blocking or reordering beyond
 * the definition.  Readings of points the sources leave open (each one is a
 * stated choice, not something the sources fix):
 *  - state S is d_v x d_k (row i = value channel, column j = key channel),
 *    so that v k^T has the shape of S and o = S q has d_v entries;
 *  - value head h reads key head h / (Hv/Hk) (contiguous groups);
 *  - the mixed conv input is laid out [q (Hk*dk) | k (Hk*dk) | v (Hv*dv)],
 *    head-major inside each block;
 *  - the conv has no bias; tap w[c][3] multiplies the current row and
 *    w[c][0] the row three steps back; the kept tail holds the three
 *    previous pre-conv inputs, oldest first;
 *  - L2 norm: x / sqrt(sum x^2 + eps_l2); q is then multiplied by q_scale;
 *  - softplus(x) = log(1 + e^x); sigmoid(x) = 1 / (1 + e^-x);
 *    SiLU(x) = x * sigmoid(x);
 *  - gated RMSNorm per value head over d_v:
 *      y_i = o_i / sqrt(mean(o^2) + eps_rms) * w_norm[i] * SiLU(z_i),
 *    one w_norm[d_v] shared by all heads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t n_k_heads, n_v_heads, d_k, d_v;
    double q_scale, eps_l2, eps_rms;
} or_dims;

/* ---- scalar definitions ------------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }
/* log(1 + e^x), written as max(x,0) + log(1 + e^-|x|) so that it neither
 * overflows nor loses the small term; the two forms are equal. */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* Gate terms of one (row, value head):
 *   g = -exp(A_log) * softplus(a + dt_bias),  decay a_t = exp(g),
 *   beta b_t = sigmoid(b). */
void oracle_gates(double A_log, double dt_bias, double a_in, double b_in,
                  double *decay, double *beta)
{
    double g = -exp(A_log) * softplus(a_in + dt_bias);
    *decay = exp(g);
    *beta = sigmoid(b_in);
}

/* Gated delta rule, one row of one value head.  S is d_v x d_k row-major and
 * is replaced by
 *     S' = a S (I - b k k^T) + b v k^T
 * computed as S' = a (S - b (S k) k^T) + b v k^T, which is the same product
 * with the d_k x d_k matrix never formed.  Then o = S' q. */
void oracle_delta_rule(int dv, int dk, double *S, const double *q,
                       const double *k, const double *v, double decay,
                       double beta, double *o)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)dv);
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * k[j];
        p[i] = acc;
    }
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
            double s = S[(size_t)i * dk + j];
            S[(size_t)i * dk + j] = decay * (s - beta * p[i] * k[j]) + beta * v[i] * k[j];
        }
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
    free(p);
}

/* Gated RMSNorm of one value head: y_i = o_i / sqrt(mean(o^2) + eps) * w_i * SiLU(z_i). */
void oracle_gated_rmsnorm(int dv, const double *o, const double *z,
                          const double *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < dv; ++i) ss += o[i] * o[i];
    double inv = 1.0 / sqrt(ss / dv + eps);
    for (int i = 0; i < dv; ++i) y[i] = o[i] * inv * w[i] * silu(z[i]);
}

/* L2 normalisation of a vector, then a scale: x * scale / sqrt(sum x^2 + eps). */
void oracle_l2norm(int n, double *x, double eps, double scale)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) x[i] = x[i] * inv * scale;
}

/* ---- one stream's rows ------------------------------------------------- */

/* The four conv inputs of row t, oldest first: hist[3] is row t itself,
 * hist[2] its parent's input, hist[1] the grandparent's, hist[0] the one
 * before.  Once the branch reaches the committed slot (parent -1) the walk
 * continues into the kept tail, most recent entry (tail row 2) first. */
static void conv_history(int32_t t, const int32_t *parent, const uint16_t *mixed,
                         const uint16_t *tail0, int CH, const uint16_t *hist[4])
{
    int32_t node = t;
    int tail_next = 2;
    hist[3] = mixed + (size_t)t * CH;
    for (int m = 2; m >= 0; --m) {
        if (node >= 0) node = parent ? parent[node] : node - 1;
        if (node >= 0) {
            hist[m] = mixed + (size_t)node * CH;
        } else {
            hist[m] = tail0 + (size_t)tail_next * CH;
            --tail_next;
        }
    }
}

/* conv over the 4 taps, then SiLU, for channels [c0, c0 + n). */
static void conv_silu(const uint16_t *hist[4], const uint16_t *conv_w, int c0,
                      int n, double *out)
{
    for (int i = 0; i < n; ++i) {
        int c = c0 + i;
        double acc = 0.0;
        for (int j = 0; j < 4; ++j)
            acc += bf16_value(conv_w[(size_t)c * 4 + j]) * bf16_value(hist[j][c]);
        out[i] = silu(acc);
    }
}

/*
 * One stream's rows through the layer, for value heads [h_begin, h_end).
 *
 *   n        rows in the window (or prompt)
 *   parent   [n] window-local parent of each row, -1 = the committed slot;
 *            NULL means a chain (parent[t] = t - 1)
 *   state0   [Hv, dv, dk] fp32 committed state
 *   tail0    [3, CH] bf16 committed conv tail, oldest first
 *   mixed    [n, CH] bf16 conv inputs; z [n, Hv, dv]; a, b [n, Hv] (bf16)
 * Outputs (each may be NULL unless noted):
 *   y          [n, Hv, dv] gated RMSNorm output, unrounded (required)
 *   rec_state  [n, Hv, dv, dk] state after each row (required for trees)
 *   rec_tail   [n, 3, CH] bf16: the three newest conv inputs after each row,
 *              oldest first (the tail a commit of that row keeps); written
 *              for every channel
 *   final_state [Hv, dv, dk] state after row n-1 of a chain
 *   final_tail  [3, CH] tail after row n-1 of a chain
 *   q_out, k_out [n, Hv, dk] and v_out [n, Hv, dv]: the normalised q, k
 *              and the v each head used (for the tests' checks)
 *   decay_out, beta_out [n, Hv]
 * Returns 0, or -1 for an invalid argument.
 */
int oracle_gdn_rows(const or_dims *d, const uint16_t *conv_w, const float *A_log,
                    const float *dt_bias, const uint16_t *norm_w, int32_t n,
                    const int32_t *parent, const float *state0,
                    const uint16_t *tail0, const uint16_t *mixed,
                    const uint16_t *z, const uint16_t *a, const uint16_t *b,
                    int32_t h_begin, int32_t h_end, double *y,
                    double *rec_state, uint16_t *rec_tail, double *final_state,
                    uint16_t *final_tail, double *q_out, double *k_out,
                    double *v_out, double *decay_out, double *beta_out)
{
    const int Hk = d->n_k_heads, Hv = d->n_v_heads, dk = d->d_k, dv = d->d_v;
    if (Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk != 0 || n < 0) return -1;
    if (h_begin < 0 || h_end > Hv || h_begin > h_end) return -1;
    if (!y || (parent && !rec_state)) return -1;
    for (int32_t t = 0; parent && t < n; ++t)
        if (parent[t] < -1 || parent[t] >= t) return -1;

    const int G = Hv / Hk;
    const int CH = 2 * Hk * dk + Hv * dv;
    const size_t tile = (size_t)dv * dk;

    double *S = (double *)malloc(sizeof(double) * tile);
    double *q = (double *)malloc(sizeof(double) * dk);
    double *k = (double *)malloc(sizeof(double) * dk);
    double *v = (double *)malloc(sizeof(double) * dv);
    double *o = (double *)malloc(sizeof(double) * dv);
    double *zz = (double *)malloc(sizeof(double) * dv);
    double *wn = (double *)malloc(sizeof(double) * dv);
    for (int i = 0; i < dv; ++i) wn[i] = bf16_value(norm_w[i]);

    for (int32_t t = 0; t < n; ++t) {
        const uint16_t *hist[4];
        conv_history(t, parent, mixed, tail0, CH, hist);
        if (rec_tail)
            for (int m = 0; m < 3; ++m)
                memcpy(rec_tail + ((size_t)t * 3 + m) * CH, hist[m + 1], sizeof(uint16_t) * CH);
        if (final_tail && t == n - 1)
            for (int m = 0; m < 3; ++m)
                memcpy(final_tail + (size_t)m * CH, hist[m + 1], sizeof(uint16_t) * CH);
    }

    for (int32_t h = h_begin; h < h_end; ++h) {
        const int kh = h / G;
        for (size_t e = 0; e < tile; ++e) S[e] = (double)state0[(size_t)h * tile + e];
        for (int32_t t = 0; t < n; ++t) {
            int32_t par = parent ? parent[t] : t - 1;
            if (parent) {
                /* a tree row starts from its parent's state */
                if (par < 0)
                    for (size_t e = 0; e < tile; ++e) S[e] = (double)state0[(size_t)h * tile + e];
                else
                    memcpy(S, rec_state + ((size_t)par * Hv + h) * tile, sizeof(double) * tile);
            }
            const uint16_t *hist[4];
            conv_history(t, parent, mixed, tail0, CH, hist);
            conv_silu(hist, conv_w, kh * dk, dk, q);
            conv_silu(hist, conv_w, Hk * dk + kh * dk, dk, k);
            conv_silu(hist, conv_w, 2 * Hk * dk + h * dv, dv, v);
            oracle_l2norm(dk, q, d->eps_l2, d->q_scale);
            oracle_l2norm(dk, k, d->eps_l2, 1.0);

            double decay, beta;
            oracle_gates((double)A_log[h], (double)dt_bias[h],
                         bf16_value(a[(size_t)t * Hv + h]), bf16_value(b[(size_t)t * Hv + h]),
                         &decay, &beta);
            oracle_delta_rule(dv, dk, S, q, k, v, decay, beta, o);

            for (int i = 0; i < dv; ++i) zz[i] = bf16_value(z[((size_t)t * Hv + h) * dv + i]);
            oracle_gated_rmsnorm(dv, o, zz, wn, d->eps_rms, y + ((size_t)t * Hv + h) * dv);

            if (rec_state) memcpy(rec_state + ((size_t)t * Hv + h) * tile, S, sizeof(double) * tile);
            if (q_out) memcpy(q_out + ((size_t)t * Hv + h) * dk, q, sizeof(double) * dk);
            if (k_out) memcpy(k_out + ((size_t)t * Hv + h) * dk, k, sizeof(double) * dk);
            if (v_out) memcpy(v_out + ((size_t)t * Hv + h) * dv, v, sizeof(double) * dv);
            if (decay_out) decay_out[(size_t)t * Hv + h] = decay;
            if (beta_out) beta_out[(size_t)t * Hv + h] = beta;
        }
        if (final_state && !parent && n > 0) memcpy(final_state + (size_t)h * tile, S, sizeof(double) * tile);
        if (final_state && !parent && n == 0)
            for (size_t e = 0; e < tile; ++e) final_state[(size_t)h * tile + e] = (double)state0[(size_t)h * tile + e];
    }
    free(S); free(q); free(k); free(v); free(o); free(zz); free(wn);
    return 0;
}

/* Commit of the accepted path: a stream whose kept row is r >= 0 takes that
 * row's recorded state and tail as its new committed state and tail; r = -1
 * leaves it untouched.  (TensorFold #747, first note: only each stream's
 * accepted path is committed.) */
void oracle_commit(int32_t state_elems, int32_t tail_elems, int32_t keep_row,
                   const double *rec_state, const uint16_t *rec_tail,
                   double *state, uint16_t *tail)
{
    if (keep_row < 0) return;
    memcpy(state, rec_state + (size_t)keep_row * state_elems, sizeof(double) * state_elems);
    memcpy(tail, rec_tail + (size_t)keep_row * tail_elems, sizeof(uint16_t) * tail_elems);
}

/* ---- chunked form of the recurrence (for checking the chunk algebra) ---- */

/*
 * The chunked (WY / UT) form of the same recurrence for one head, on q, k, v
 * that are already normalised, with per-row log-decay g_t = log a_t and
 * beta b_t.  It is NOT the definition: the tests pin it to the sequential
 * recurrence above.  Chunks of C rows; inside a chunk, with
 * G_t = sum_{s<=t} g_s, gamma_t = exp(G_t), Gamma_ts = exp(G_t - G_s):
 *   A = K K^T
 *   (I + strict_lower(diag(b) (Gamma o A))) X = Y   solved for
 *     W  = X with Y = diag(b gamma) K
 *     U~ = X with Y = diag(b) V
 *   U = U~ - W S0^T
 *   O = diag(gamma) Q S0^T + lower(Gamma o (Q K^T)) U
 *   S = gamma_C S0 + U^T diag(gamma_C / gamma) K
 * S is d_v x d_k; Q, K are L x dk, V and O are L x dv (row-major).
 */
void oracle_chunked_rule(int dv, int dk, int L, int C, double *S,
                         const double *Q, const double *K, const double *V,
                         const double *g, const double *beta, double *O)
{
    double *Gc = (double *)malloc(sizeof(double) * C);
    double *A = (double *)malloc(sizeof(double) * C * C);
    double *W = (double *)malloc(sizeof(double) * C * dk);
    double *U = (double *)malloc(sizeof(double) * C * dv);
    double *Snew = (double *)malloc(sizeof(double) * dv * dk);
    for (int c0 = 0; c0 < L; c0 += C) {
        int n = (L - c0 < C) ? (L - c0) : C;
        const double *Qc = Q + (size_t)c0 * dk, *Kc = K + (size_t)c0 * dk, *Vc = V + (size_t)c0 * dv;
        const double *gc = g + c0, *bc = beta + c0;
        double run = 0.0;
        for (int t = 0; t < n; ++t) { run += gc[t]; Gc[t] = run; }
        for (int t = 0; t < n; ++t)
            for (int s = 0; s < n; ++s) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += Kc[(size_t)t * dk + j] * Kc[(size_t)s * dk + j];
                A[t * C + s] = acc;
            }
        /* forward substitution, row by row: x_t = y_t - b_t sum_{s<t} Gamma_ts A_ts x_s */
        for (int t = 0; t < n; ++t) {
            double gt = exp(Gc[t]);
            for (int j = 0; j < dk; ++j) W[(size_t)t * dk + j] = bc[t] * gt * Kc[(size_t)t * dk + j];
            for (int i = 0; i < dv; ++i) U[(size_t)t * dv + i] = bc[t] * Vc[(size_t)t * dv + i];
            for (int s = 0; s < t; ++s) {
                double m = bc[t] * exp(Gc[t] - Gc[s]) * A[t * C + s];
                for (int j = 0; j < dk; ++j) W[(size_t)t * dk + j] -= m * W[(size_t)s * dk + j];
                for (int i = 0; i < dv; ++i) U[(size_t)t * dv + i] -= m * U[(size_t)s * dv + i];
            }
        }
        /* U = U~ - W S0^T */
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += W[(size_t)t * dk + j] * S[(size_t)i * dk + j];
                U[(size_t)t * dv + i] -= acc;
            }
        /* O = diag(gamma) Q S0^T + lower(Gamma o Q K^T) U */
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += Qc[(size_t)t * dk + j] * S[(size_t)i * dk + j];
                acc *= exp(Gc[t]);
                for (int s = 0; s <= t; ++s) {
                    double qk = 0.0;
                    for (int j = 0; j < dk; ++j) qk += Qc[(size_t)t * dk + j] * Kc[(size_t)s * dk + j];
                    acc += exp(Gc[t] - Gc[s]) * qk * U[(size_t)s * dv + i];
                }
                O[(size_t)(c0 + t) * dv + i] = acc;
            }
        /* S = gamma_C S0 + U^T diag(gamma_C / gamma) K */
        double GC = Gc[n - 1];
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double acc = exp(GC) * S[(size_t)i * dk + j];
                for (int t = 0; t < n; ++t)
                    acc += U[(size_t)t * dv + i] * exp(GC - Gc[t]) * Kc[(size_t)t * dk + j];
                Snew[(size_t)i * dk + j] = acc;
            }
        memcpy(S, Snew, sizeof(double) * dv * dk);
    }
    free(Gc); free(A); free(W); free(U); free(Snew);
}
