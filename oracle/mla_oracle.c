/*
 * fp64 oracle for Multi-Head Latent Attention (MLA) and its variants.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow definition that the
 * CUDA path is checked against.  Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg may load it; the library itself never
 * does.  It shares no code, header, table or constant with the CUDA sources.
 *
 * Every quantity is computed in double precision straight from its definition:
 * the keys and values are materialised explicitly (the "definition" form).  A
 * second, weight-absorbed form is provided only so that tests can check that
 * the two agree; it is the same arithmetic regrouped by associativity.
 *
 * Sources (web pages on the subject, by title and section):
 *  [DS]  bird-of-paradise/deepseek-mla, src/mla.py: precompute_freqs_cis,
 *        apply_rotary_emb, MultiHeadLatentAttention.__init__/.forward.
 *  [SM]  frankenstein-transformer, latent/mla_attn.py: module docstring
 *        (formulation), _apply_rope, MLAAttention.forward.
 *  [LR]  frankenstein-transformer, latent/mlra_attn.py: module docstring,
 *        MLRAAttention.__init__/.forward.
 *  [GI]  gist "Multi-Head Latent Attention", mla.py (shape cross-check).
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes as well):
 *  - causal attention always: the query at absolute position p sees keys
 *    0..p; masked keys get weight exactly 0;
 *  - absolute 0-based positions for both queries and cached keys;
 *  - the rope-key cache holds k_R after rotation;
 *  - no biases, no dropout, no normalisation of c_Q or c_KV;
 *  - d_v equals d_nope and is independent of d_model.
 *
 * Layouts: row-major, weights in nn.Linear layout [out, in].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_MEM 2

int orc_version(void) { return 1; }

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* y[t, o] = sum_i W[o, i] * x[t, i]: nn.Linear without bias ([DS] __init__,
 * [SM] __init__ use bias=False; [GI] applies the same map as x @ w). */
void orc_linear(const double *x, long T, int n_in, const double *W, int n_out,
                double *y, int n_threads)
{
    long t;
    (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads > 0 ? n_threads : 1) schedule(static)
#endif
    for (t = 0; t < T; ++t) {
        const double *xr = x + t * (long)n_in;
        for (int o = 0; o < n_out; ++o) {
            const double *wr = W + (long)o * n_in;
            double s = 0.0;
            for (int i = 0; i < n_in; ++i) s += wr[i] * xr[i];
            y[t * (long)n_out + o] = s;
        }
    }
}

/* Rotary frequency of pair i in a d-wide rotated vector: theta_i = base^(-2i/d)
 * ([DS] precompute_freqs_cis; [SM] _apply_rope, inv_freq). */
static double rope_theta(int i, int d, double base)
{
    return pow(base, -2.0 * (double)i / (double)d);
}

/* Rotate the pair (a, b) by angle phi: (a cos - b sin, a sin + b cos).  This is
 * the complex product (a + ib) e^{i phi} of [DS] apply_rotary_emb and the
 * cat([x1 cos - x2 sin, x1 sin + x2 cos]) of [SM] _apply_rope. */
static void rotate_pair(double *a, double *b, double phi)
{
    double c = cos(phi), s = sin(phi);
    double x0 = *a, x1 = *b;
    *a = x0 * c - x1 * s;
    *b = x0 * s + x1 * c;
}

/* Interleaved RoPE ([DS] apply_rotary_emb: view_as_complex pairs the last
 * dimension as (x[2i], x[2i+1])).  x is [n_rows, n_groups, d]; row r is
 * rotated at position pos[r]. */
void orc_rope_interleaved(double *x, long n_rows, int n_groups, int d,
                          const int *pos, double base)
{
    for (long r = 0; r < n_rows; ++r)
        for (int g = 0; g < n_groups; ++g) {
            double *v = x + (r * n_groups + g) * (long)d;
            for (int i = 0; i < d / 2; ++i)
                rotate_pair(&v[2 * i], &v[2 * i + 1],
                            (double)pos[r] * rope_theta(i, d, base));
        }
}

/* Half-split RoPE ([SM] _apply_rope: x1 = x[:d/2], x2 = x[d/2:], pair i is
 * (x[i], x[i + d/2])). */
void orc_rope_half(double *x, long n_rows, int n_groups, int d, const int *pos,
                   double base)
{
    for (long r = 0; r < n_rows; ++r)
        for (int g = 0; g < n_groups; ++g) {
            double *v = x + (r * n_groups + g) * (long)d;
            for (int i = 0; i < d / 2; ++i)
                rotate_pair(&v[i], &v[i + d / 2],
                            (double)pos[r] * rope_theta(i, d, base));
        }
}

/* Softmax over s[0..n-1] in place: exp(s_j - max) / sum ([DS] forward,
 * F.softmax over the key axis; [SM] forward).  Only unmasked keys are passed
 * in, so masked keys never enter the sum and keep weight 0. */
static void softmax_inplace(double *s, long n)
{
    double m = -INFINITY, z = 0.0;
    for (long j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    for (long j = 0; j < n; ++j) { s[j] = exp(s[j] - m); z += s[j]; }
    for (long j = 0; j < n; ++j) s[j] /= z;
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* Per-sequence largest query position, so that keys are materialised once per
 * (sequence, head). */
static int *max_pos_per_seq(long n_q, const int *q_b, const int *q_pos,
                            int *n_seq_out)
{
    int nb = 0;
    for (long i = 0; i < n_q; ++i) if (q_b[i] + 1 > nb) nb = q_b[i] + 1;
    int *mp = (int *)malloc(sizeof(int) * (size_t)(nb > 0 ? nb : 1));
    if (!mp) return NULL;
    for (int b = 0; b < nb; ++b) mp[b] = -1;
    for (long i = 0; i < n_q; ++i) if (q_pos[i] > mp[q_b[i]]) mp[q_b[i]] = q_pos[i];
    *n_seq_out = nb;
    return mp;
}

/* ------------------------------------------------------------------------ */
/* Projections (the cache-append step and the query path)                    */
/* ------------------------------------------------------------------------ */

/* Decoupled MLA, per token at absolute position pos[t] ([DS] forward, query
 * path and use_cache branch; [GI] mla.py, its query and key-value steps):
 *   c_Q    = W_DQ x                       [r_q]
 *   q_nope = W_UQ c_Q                     [H, d_nope]
 *   q_rope = RoPE_pos(W_QR c_Q)  per head [H, d_rope]  (interleaved pairs)
 *   c_KV   = W_DKV x                      [r_kv]   (the cached latent)
 *   k_R    = RoPE_pos(W_KR x)             [d_rope] (cached, shared by heads)
 */
int orc_decoupled_project(int d_model, int H, int d_nope, int d_rope, int r_kv,
                          int r_q, double base, long T, const double *x,
                          const int *pos, const double *W_DQ, const double *W_UQ,
                          const double *W_QR, const double *W_DKV,
                          const double *W_KR, double *c_kv, double *k_r,
                          double *q_nope, double *q_rope, int n_threads)
{
    if (T < 0 || d_rope % 2) return ORC_ERR_ARG;
    double *c_q = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)r_q);
    if (!c_q) return ORC_ERR_MEM;
    orc_linear(x, T, d_model, W_DQ, r_q, c_q, n_threads);
    orc_linear(c_q, T, r_q, W_UQ, H * d_nope, q_nope, n_threads);
    orc_linear(c_q, T, r_q, W_QR, H * d_rope, q_rope, n_threads);
    orc_rope_interleaved(q_rope, T, H, d_rope, pos, base);
    orc_linear(x, T, d_model, W_DKV, r_kv, c_kv, n_threads);
    orc_linear(x, T, d_model, W_KR, d_rope, k_r, n_threads);
    orc_rope_interleaved(k_r, T, 1, d_rope, pos, base);
    free(c_q);
    return ORC_OK;
}

/* Small-model MLA ([SM] module docstring and forward): q = W_Q x, rotated
 * half-split per head when use_rope; c_KV = W_DKV x is all that is cached. */
int orc_small_project(int d_model, int H, int d, int r_kv, int use_rope,
                      double base, long T, const double *x, const int *pos,
                      const double *W_Q, const double *W_DKV, double *c_kv,
                      double *q, int n_threads)
{
    if (T < 0 || d % 2) return ORC_ERR_ARG;
    orc_linear(x, T, d_model, W_Q, H * d, q, n_threads);
    if (use_rope) orc_rope_half(q, T, H, d, pos, base);
    orc_linear(x, T, d_model, W_DKV, r_kv, c_kv, n_threads);
    return ORC_OK;
}

/* MLRA ([LR] forward): q = W_Q x (no rotary embedding), c_KV = W_DKV x. */
int orc_mlra_project(int d_model, int H, int d, int r_kv, long T, const double *x,
                     const double *W_Q, const double *W_DKV, double *c_kv,
                     double *q, int n_threads)
{
    if (T < 0) return ORC_ERR_ARG;
    orc_linear(x, T, d_model, W_Q, H * d, q, n_threads);
    orc_linear(x, T, d_model, W_DKV, r_kv, c_kv, n_threads);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention over the cache, definition form (keys and values materialised)  */
/* ------------------------------------------------------------------------ */

#define VAR_DECOUPLED 0
#define VAR_SMALL 1
#define VAR_MLRA 2

typedef struct {
    int variant;
    int H, d_nope, d_rope, d_v, r_kv, L, use_rope;
    double base;
    const double *cache_lat;  /* [B, S_max, r_kv] */
    const double *cache_rope; /* [B, S_max, d_rope] (decoupled only) */
    long S_max;
    const double *W_UK, *W_UV;
} kv_source;

/* Key and value of head h for cached token j of sequence b.
 *  decoupled ([DS] forward): k = [ (W_UK c_j)[h-slice] ‖ k_R,j ],
 *                            v = (W_UV c_j)[h-slice]
 *  small     ([SM] forward): k = RoPE_half,j((W_UK c_j)[h-slice]), v likewise
 *                            without rotation
 *  MLRA      ([LR] forward): k = view(cat_i(W_UK,i c_j,i))[h-slice]: element e
 *                            of head h is element (h*d + e) of the
 *                            concatenation of the L block outputs. */
static void materialize_kv(const kv_source *s, int b, int h, long j, double *k,
                           double *v)
{
    const double *c = s->cache_lat + ((long)b * s->S_max + j) * s->r_kv;
    if (s->variant == VAR_MLRA) {
        int sub_rank = s->r_kv / s->L;
        int sub_out_k = s->H * s->d_nope / s->L;
        int sub_out_v = s->H * s->d_v / s->L;
        for (int e = 0; e < s->d_nope; ++e) {
            int g = h * s->d_nope + e, blk = g / sub_out_k, row = g % sub_out_k;
            const double *w = s->W_UK + ((long)blk * sub_out_k + row) * sub_rank;
            k[e] = dot(w, c + (long)blk * sub_rank, sub_rank);
        }
        for (int e = 0; e < s->d_v; ++e) {
            int g = h * s->d_v + e, blk = g / sub_out_v, row = g % sub_out_v;
            const double *w = s->W_UV + ((long)blk * sub_out_v + row) * sub_rank;
            v[e] = dot(w, c + (long)blk * sub_rank, sub_rank);
        }
        return;
    }
    for (int e = 0; e < s->d_nope; ++e)
        k[e] = dot(s->W_UK + ((long)h * s->d_nope + e) * s->r_kv, c, s->r_kv);
    for (int e = 0; e < s->d_v; ++e)
        v[e] = dot(s->W_UV + ((long)h * s->d_v + e) * s->r_kv, c, s->r_kv);
    if (s->variant == VAR_DECOUPLED) {
        const double *kr = s->cache_rope + ((long)b * s->S_max + j) * s->d_rope;
        for (int e = 0; e < s->d_rope; ++e) k[s->d_nope + e] = kr[e];
    } else if (s->variant == VAR_SMALL && s->use_rope) {
        int p = (int)j;
        orc_rope_half(k, 1, 1, s->d_nope, &p, s->base);
    }
}

/* o[i, h] = sum_{j <= q_pos[i]} softmax_j(scale * <q[i, h], k_j>) v_j for every
 * query i (of sequence q_b[i]) and head h.  q is [n_q, H, dq] with dq the key
 * width.  probs, when given, receives the weights [n_q, H, S_max] with exact
 * zeros for masked keys. */
static int attend_materialized(const kv_source *s, int dq, long n_q,
                               const int *q_b, const int *q_pos, const double *q,
                               double scale, int n_threads, double *o,
                               double *probs)
{
    int nb = 0;
    int *mp = max_pos_per_seq(n_q, q_b, q_pos, &nb);
    if (!mp) return ORC_ERR_MEM;
    for (long i = 0; i < n_q; ++i)
        if (q_pos[i] < 0 || q_pos[i] >= s->S_max || q_b[i] < 0) { free(mp); return ORC_ERR_ARG; }
    int err = ORC_OK;
    int h;
    (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads > 0 ? n_threads : 1) schedule(dynamic)
#endif
    for (h = 0; h < s->H; ++h) {
        long cap = s->S_max;
        double *K = (double *)malloc(sizeof(double) * (size_t)cap * (size_t)dq);
        double *V = (double *)malloc(sizeof(double) * (size_t)cap * (size_t)s->d_v);
        double *sc = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!K || !V || !sc) {
            free(K); free(V); free(sc);
            err = ORC_ERR_MEM;
            continue;
        }
        for (int b = 0; b < nb; ++b) {
            if (mp[b] < 0) continue;
            for (long j = 0; j <= mp[b]; ++j)
                materialize_kv(s, b, h, j, K + j * dq, V + j * s->d_v);
            for (long i = 0; i < n_q; ++i) {
                if (q_b[i] != b) continue;
                long n_keys = (long)q_pos[i] + 1;          /* causal: keys 0..p */
                const double *qi = q + (i * s->H + h) * (long)dq;
                for (long j = 0; j < n_keys; ++j) sc[j] = scale * dot(qi, K + j * dq, dq);
                softmax_inplace(sc, n_keys);
                double *oi = o + (i * s->H + h) * (long)s->d_v;
                for (int e = 0; e < s->d_v; ++e) {
                    double acc = 0.0;
                    for (long j = 0; j < n_keys; ++j) acc += sc[j] * V[j * s->d_v + e];
                    oi[e] = acc;
                }
                if (probs) {
                    double *pi = probs + (i * s->H + h) * s->S_max;
                    for (long j = 0; j < s->S_max; ++j) pi[j] = j < n_keys ? sc[j] : 0.0;
                }
            }
        }
        free(K); free(V); free(sc);
    }
    free(mp);
    return err;
}

/* Decoupled MLA attention ([DS] forward): scores are
 * (q_C . k_C + q_R . k_R) / sqrt(d_nope + d_rope), causal softmax, weighted
 * sum of v.  q_nope [n_q, H, d_nope], q_rope [n_q, H, d_rope] (already
 * rotated at the query position), caches [B, S_max, *] with k_R rotated. */
int orc_decoupled_attend(int H, int d_nope, int d_rope, int d_v, int r_kv,
                         long n_q, const int *q_b, const int *q_pos,
                         const double *q_nope, const double *q_rope,
                         const double *cache_lat, const double *cache_rope,
                         long S_max, const double *W_UK, const double *W_UV,
                         int n_threads, double *o, double *probs)
{
    int dq = d_nope + d_rope;
    double *q = (double *)malloc(sizeof(double) * (size_t)(n_q > 0 ? n_q : 1) * (size_t)H * (size_t)dq);
    if (!q) return ORC_ERR_MEM;
    for (long i = 0; i < n_q; ++i)
        for (int h = 0; h < H; ++h) {
            double *qq = q + (i * H + h) * (long)dq;
            memcpy(qq, q_nope + (i * H + h) * (long)d_nope, sizeof(double) * (size_t)d_nope);
            memcpy(qq + d_nope, q_rope + (i * H + h) * (long)d_rope, sizeof(double) * (size_t)d_rope);
        }
    kv_source s = {VAR_DECOUPLED, H, d_nope, d_rope, d_v, r_kv, 1, 0, 0.0,
                   cache_lat, cache_rope, S_max, W_UK, W_UV};
    int rc = attend_materialized(&s, dq, n_q, q_b, q_pos, q,
                                 1.0 / sqrt((double)(d_nope + d_rope)), n_threads, o, probs);
    free(q);
    return rc;
}

/* Small-model MLA attention ([SM] forward): k = RoPE_half(W_UK c) per head at
 * the key's position (when use_rope), v = W_UV c, scale 1/sqrt(d). */
int orc_small_attend(int H, int d, int r_kv, int use_rope, double base, long n_q,
                     const int *q_b, const int *q_pos, const double *q,
                     const double *cache_lat, long S_max, const double *W_UK,
                     const double *W_UV, int n_threads, double *o, double *probs)
{
    kv_source s = {VAR_SMALL, H, d, 0, d, r_kv, 1, use_rope, base,
                   cache_lat, NULL, S_max, W_UK, W_UV};
    return attend_materialized(&s, d, n_q, q_b, q_pos, q, 1.0 / sqrt((double)d),
                               n_threads, o, probs);
}

/* MLRA attention ([LR] forward): block-wise up-projections of the L latent
 * sub-vectors, concatenated and viewed per head; no rotary embedding; scale
 * 1/sqrt(d). */
int orc_mlra_attend(int H, int d, int r_kv, int L, long n_q, const int *q_b,
                    const int *q_pos, const double *q, const double *cache_lat,
                    long S_max, const double *W_UK, const double *W_UV,
                    int n_threads, double *o, double *probs)
{
    if (L <= 0 || r_kv % L || (H * d) % L) return ORC_ERR_ARG;
    kv_source s = {VAR_MLRA, H, d, 0, d, r_kv, L, 0, 0.0,
                   cache_lat, NULL, S_max, W_UK, W_UV};
    return attend_materialized(&s, d, n_q, q_b, q_pos, q, 1.0 / sqrt((double)d),
                               n_threads, o, probs);
}

/* ------------------------------------------------------------------------ */
/* Weight-absorbed forms (same arithmetic regrouped; used to check the        */
/* absorption identity and to evaluate large decode cases quickly)           */
/* ------------------------------------------------------------------------ */

/* Decoupled: q_abs = W_UK,h^T q_C ; s_j = (q_abs . c_j + q_R . k_R,j) * scale ;
 * o_lat = sum_j p_j c_j ; o = W_UV,h o_lat.  Uses
 * q_C . (W_UK,h c_j) = (W_UK,h^T q_C) . c_j and
 * sum_j p_j W_UV,h c_j = W_UV,h sum_j p_j c_j. */
int orc_decoupled_attend_absorbed(int H, int d_nope, int d_rope, int d_v, int r_kv,
                                  long n_q, const int *q_b, const int *q_pos,
                                  const double *q_nope, const double *q_rope,
                                  const double *cache_lat, const double *cache_rope,
                                  long S_max, const double *W_UK,
                                  const double *W_UV, int n_threads, double *o)
{
    for (long i = 0; i < n_q; ++i)
        if (q_pos[i] < 0 || q_pos[i] >= S_max || q_b[i] < 0) return ORC_ERR_ARG;
    double scale = 1.0 / sqrt((double)(d_nope + d_rope));
    int err = ORC_OK;
    long ih;
    (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads > 0 ? n_threads : 1) schedule(dynamic)
#endif
    for (ih = 0; ih < n_q * H; ++ih) {
        long i = ih / H;
        int h = (int)(ih % H);
        int b = q_b[i];
        long n_keys = (long)q_pos[i] + 1;
        double *q_abs = (double *)calloc((size_t)r_kv, sizeof(double));
        double *o_lat = (double *)calloc((size_t)r_kv, sizeof(double));
        double *sc = (double *)malloc(sizeof(double) * (size_t)n_keys);
        if (!q_abs || !o_lat || !sc) {
            free(q_abs); free(o_lat); free(sc);
            err = ORC_ERR_MEM;
            continue;
        }
        const double *qn = q_nope + (i * H + h) * (long)d_nope;
        const double *qr = q_rope + (i * H + h) * (long)d_rope;
        for (int e = 0; e < d_nope; ++e) {
            const double *w = W_UK + ((long)h * d_nope + e) * r_kv;
            for (int c = 0; c < r_kv; ++c) q_abs[c] += w[c] * qn[e];
        }
        for (long j = 0; j < n_keys; ++j) {
            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;
            const double *kr = cache_rope + ((long)b * S_max + j) * d_rope;
            sc[j] = scale * (dot(q_abs, cj, r_kv) + dot(qr, kr, d_rope));
        }
        softmax_inplace(sc, n_keys);
        for (long j = 0; j < n_keys; ++j) {
            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;
            for (int c = 0; c < r_kv; ++c) o_lat[c] += sc[j] * cj[c];
        }
        double *oi = o + (i * H + h) * (long)d_v;
        for (int e = 0; e < d_v; ++e)
            oi[e] = dot(W_UV + ((long)h * d_v + e) * r_kv, o_lat, r_kv);
        free(q_abs); free(o_lat); free(sc);
    }
    return err;
}

/* MLRA, absorbed: element e of head h reads block blk = (h*d + e) / (H*d/L),
 * row (h*d + e) mod (H*d/L).  q_abs lives in the full rank-r latent space and
 * is zero outside the blocks the head touches. */
int orc_mlra_attend_absorbed(int H, int d, int r_kv, int L, long n_q,
                             const int *q_b, const int *q_pos, const double *q,
                             const double *cache_lat, long S_max,
                             const double *W_UK, const double *W_UV,
                             int n_threads, double *o)
{
    if (L <= 0 || r_kv % L || (H * d) % L) return ORC_ERR_ARG;
    for (long i = 0; i < n_q; ++i)
        if (q_pos[i] < 0 || q_pos[i] >= S_max || q_b[i] < 0) return ORC_ERR_ARG;
    int sub_rank = r_kv / L, sub_out = H * d / L;
    double scale = 1.0 / sqrt((double)d);
    int err = ORC_OK;
    long ih;
    (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads > 0 ? n_threads : 1) schedule(dynamic)
#endif
    for (ih = 0; ih < n_q * H; ++ih) {
        long i = ih / H;
        int h = (int)(ih % H);
        int b = q_b[i];
        long n_keys = (long)q_pos[i] + 1;
        double *q_abs = (double *)calloc((size_t)r_kv, sizeof(double));
        double *o_lat = (double *)calloc((size_t)r_kv, sizeof(double));
        double *sc = (double *)malloc(sizeof(double) * (size_t)n_keys);
        char *touched = (char *)calloc((size_t)L, 1);
        if (!q_abs || !o_lat || !sc || !touched) {
            free(q_abs); free(o_lat); free(sc); free(touched);
            err = ORC_ERR_MEM;
            continue;
        }
        const double *qi = q + (i * H + h) * (long)d;
        for (int e = 0; e < d; ++e) {
            int g = h * d + e, blk = g / sub_out, row = g % sub_out;
            const double *w = W_UK + ((long)blk * sub_out + row) * sub_rank;
            touched[blk] = 1;
            for (int c = 0; c < sub_rank; ++c) q_abs[blk * sub_rank + c] += w[c] * qi[e];
        }
        /* Blocks the head does not touch contribute exact zeros: skip them. */
        for (long j = 0; j < n_keys; ++j) {
            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;
            double acc = 0.0;
            for (int blk = 0; blk < L; ++blk)
                if (touched[blk])
                    acc += dot(q_abs + blk * sub_rank, cj + blk * sub_rank, sub_rank);
            sc[j] = scale * acc;
        }
        softmax_inplace(sc, n_keys);
        for (long j = 0; j < n_keys; ++j) {
            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;
            for (int blk = 0; blk < L; ++blk)
                if (touched[blk])
                    for (int c = 0; c < sub_rank; ++c)
                        o_lat[blk * sub_rank + c] += sc[j] * cj[blk * sub_rank + c];
        }
        double *oi = o + (i * H + h) * (long)d;
        for (int e = 0; e < d; ++e) {
            int g = h * d + e, blk = g / sub_out, row = g % sub_out;
            const double *w = W_UV + ((long)blk * sub_out + row) * sub_rank;
            oi[e] = dot(w, o_lat + blk * sub_rank, sub_rank);
        }
        free(q_abs); free(o_lat); free(sc); free(touched);
    }
    return err;
}
