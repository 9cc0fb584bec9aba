/*
 * fp64 CPU oracle for weight-absorbed Multi-head Latent Attention (MLA) decode.
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA path is checked against it; it is not the product: only the
 * test suite, the smoke check and the benchmark's CPU-baseline / reference legs
 * load it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Every activation is carried in double precision.  Cache, weights and query
 * inputs arrive as the exact bf16 bit patterns handed to the GPU and are widened
 * to double here (bf16 -> fp32 -> fp64 is exact).  There is no blocking, fusion
 * or reordering beyond what the definitions below state: plain loops, with an
 * OpenMP loop over independent output rows.
 *
 * Sources (page title, section):
 *  [MLA-dim]  "MLA, dim by dim" -- section "MLA Decode" (decode score order,
 *             decode value order), section "Why RoPE Gets in the Way"
 *             (decoupled content + positional score), "Notation and
 *             Preliminaries" (weight shapes W_UK:(h,d_c,d_k), W_UV:(h,d_c,d_v)).
 *  [AI]       "Why MLA and MTP Fight Each Other: Attention Through Arithmetic
 *             Intensity" -- sections 3.1 (K-side absorption), 3.2 (V-side
 *             absorption), 3.3 (un-absorbed re-expansion), 8 (S query positions
 *             against one cached history), Appendix A (decoupled RoPE segment
 *             shared by all heads, scoring only).
 *  [speedup]  "The MLA decode speedup hiding in your model card" -- sections
 *             "The naive form, written out", "The identity", "The absorbed form".
 *  [intens]   "Decode attention intensity is fixed at the query-to-KV head
 *             ratio..." -- "A strong answer" (576-wide latent: 512 c_kv + 64 RoPE
 *             key per token, shared by all heads; with an FP8 latent the same
 *             576 values take one byte each).
 *
 * Readings where the pages are silent:
 *  - the cached token row is [c_kv (d_c) | k_rope (d_rope)], contiguous;
 *  - q_rope and k_rope arrive already rotated; no rotation happens here;
 *  - seq_lens[b] counts the s_q new tokens, already appended; query i
 *    (0-based) sits at position L - s_q + i and sees cached tokens j <= L - s_q + i;
 *  - lse is the natural-log log-sum-exp of the *scaled* scores;
 *  - an invalid length (L < s_q, or L beyond the cache) yields NaN rows here:
 *    the oracle is never asked to agree with the GPU on invalid input;
 *  - an FP8 latent cache holds OCP FP8 E4M3 codes (1 sign, 4 exponent bits with
 *    bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN) and one fp32
 *    scale for the whole cache: a cached value is kv_scale * code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, H, s_q, d_c, d_rope, d_nope, d_v;
    double scale;
} orc_dims;

typedef struct {
    const void *kv;              /* bf16 bits or e4m3 codes; contiguous [B][seq_stride] or pool [P][page][W] */
    long long seq_stride;        /* contiguous layout: elements between two sequences */
    const int32_t *block_table;  /* NULL => contiguous; else [B][max_pages] page ids */
    int max_pages;
    int page_size;
    long long capacity;          /* tokens a sequence may hold (contiguous: T_max) */
    const int32_t *seq_lens;     /* [B] */
    int elem;                    /* 0: bf16 elements, 1: FP8 E4M3 codes */
    double kv_scale;             /* elem 1: a cached value is kv_scale * code */
} orc_cache;

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * (m/8)
 * for e = 0 (subnormal); e = 15 with m = 7 is NaN, there is no infinity. */
double orc_e4m3_to_f64(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* The E4M3 code nearest to v (ties to the code with an even mantissa, the
 * nearest-even rule), saturating: beyond the largest finite value 448 the code
 * of +-448; NaN gives the NaN code 0x7F.  Found by searching the 127 finite
 * non-negative codes, so it follows the format's definition directly. */
uint8_t orc_f64_to_e4m3(double v)
{
    if (v != v) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_to_f64((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

void orc_encode_e4m3(long long n, const double *v, uint8_t *codes)
{
    for (long long i = 0; i < n; ++i) codes[i] = orc_f64_to_e4m3(v[i]);
}

/* Element k of a cached row (bf16 widened, or the scaled FP8 value). */
static double row_elem(const orc_cache *c, const void *row, long long k)
{
    if (c->elem == 1) return c->kv_scale * orc_e4m3_to_f64(((const uint8_t *)row)[k]);
    return bf16_to_f64(((const uint16_t *)row)[k]);
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Token j of sequence b: contiguous rows, or page block_table[b][j / page]
 * row j % page of the shared pool. */
static const void *token_row(const orc_dims *d, const orc_cache *c, int b, long long j)
{
    long long w = (long long)d->d_c + d->d_rope;
    long long esize = c->elem == 1 ? 1 : 2;
    long long at;
    if (c->block_table == NULL) {
        at = (long long)b * c->seq_stride + j * w;
    } else {
        long long page = c->block_table[(long long)b * c->max_pages + j / c->page_size];
        at = (page * c->page_size + j % c->page_size) * w;
    }
    return (const uint8_t *)c->kv + at * esize;
}

/* Absorb W_UK into the query ([MLA-dim] "MLA Decode", decode score order;
 * [AI] 3.1; [speedup] "The identity"):
 *     q_abs[b,i,h,c] = sum_n q_nope[b,i,h,n] * W_UK[h,c,n]
 * and append the already-rotated RoPE query ([AI] Appendix A):
 *     q_cat[b,i,h,:] = [ q_abs[b,i,h,0:d_c] | q_rope[b,i,h,0:d_rope] ].
 * Layouts: q_nope [B][s_q][H][d_nope], q_rope [B][s_q][H][d_rope],
 * W_UK [H][d_c][d_nope], q_cat [B][s_q][H][d_c+d_rope]. */
void orc_absorb_q(const orc_dims *d, const uint16_t *q_nope, const uint16_t *q_rope,
                  const uint16_t *w_uk, double *q_cat)
{
    long long rows = (long long)d->B * d->s_q * d->H;
    long long wq = (long long)d->d_c + d->d_rope;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        int h = (int)(r % d->H);
        const uint16_t *qn = q_nope + r * d->d_nope;
        const uint16_t *qr = q_rope + r * d->d_rope;
        double *out = q_cat + r * wq;
        for (int c = 0; c < d->d_c; ++c) {
            const uint16_t *wrow = w_uk + ((long long)h * d->d_c + c) * d->d_nope;
            double acc = 0.0;
            for (int n = 0; n < d->d_nope; ++n)
                acc += bf16_to_f64(qn[n]) * bf16_to_f64(wrow[n]);
            out[c] = acc;
        }
        for (int k = 0; k < d->d_rope; ++k)
            out[d->d_c + k] = bf16_to_f64(qr[k]);
    }
}

static int row_is_valid(const orc_dims *d, const orc_cache *c, int b)
{
    long long L = c->seq_lens[b];
    return L >= d->s_q && L <= c->capacity;
}

/* Attention of one query row against the latent cache, in latent space.
 * Scores ([MLA-dim] "Why RoPE Gets in the Way", decoupled score;
 * [intens] "A strong answer": 576-wide score, 512-wide aggregate):
 *     s_j = scale * ( sum_{c<d_c} q_abs[c] c_kv[j,c] + sum_{k<d_rope} q_rope[k] k_rope[j,k] )
 * over the visible tokens j = 0 .. L - s_q + i.  Softmax by its plain
 * definition (two passes: maximum, then normalised exponentials):
 *     lse = m + ln sum_j exp(s_j - m),   p_j = exp(s_j - lse),
 * and the weighted sum stays in latent space ([AI] 3.2; [MLA-dim] decode value
 * order): o_lat[c] = sum_j p_j c_kv[j,c], c < d_c (the RoPE key has no value part,
 * [AI] Appendix A). */
static void attend_row(const orc_dims *d, const double *q_cat, const orc_cache *c,
                       long long r, double *scores, double *o_lat, double *lse)
{
    int h = (int)(r % d->H);
    long long bi = r / d->H;
    int i = (int)(bi % d->s_q);
    int b = (int)(bi / d->s_q);
    (void)h;
    long long wq = (long long)d->d_c + d->d_rope;
    const double *q = q_cat + r * wq;
    double *o = o_lat + r * d->d_c;
    if (!row_is_valid(d, c, b)) {
        for (int k = 0; k < d->d_c; ++k) o[k] = NAN;
        lse[r] = NAN;
        return;
    }
    long long L = c->seq_lens[b];
    long long n_vis = L - d->s_q + i + 1;
    double m = -INFINITY;
    for (long long j = 0; j < n_vis; ++j) {
        const void *t = token_row(d, c, b, j);
        double dot = 0.0;
        for (long long k = 0; k < wq; ++k)
            dot += q[k] * row_elem(c, t, k);
        scores[j] = d->scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    double sum = 0.0;
    for (long long j = 0; j < n_vis; ++j)
        sum += exp(scores[j] - m);
    double l = m + log(sum);
    for (int k = 0; k < d->d_c; ++k) o[k] = 0.0;
    for (long long j = 0; j < n_vis; ++j) {
        double p = exp(scores[j] - l);
        const void *t = token_row(d, c, b, j);
        for (int k = 0; k < d->d_c; ++k)
            o[k] += p * row_elem(c, t, k);
    }
    lse[r] = l;
}

static long long max_visible(const orc_dims *d, const orc_cache *c)
{
    long long mx = 1;
    for (int b = 0; b < d->B; ++b) {
        long long L = c->seq_lens[b];
        if (L > mx) mx = L;
    }
    return mx;
}

/* o_lat [B][s_q][H][d_c] and lse [B][s_q][H] for the listed flat rows
 * r = (b*s_q + i)*H + h (all rows when rows == NULL).  Unlisted rows are left
 * untouched. */
void orc_attend(const orc_dims *d, const double *q_cat, const orc_cache *c,
                const long long *rows, long long n_rows, double *o_lat, double *lse)
{
    long long total = rows ? n_rows : (long long)d->B * d->s_q * d->H;
    long long cap = max_visible(d, c);
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
#pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < total; ++t)
            attend_row(d, q_cat, c, rows ? rows[t] : t, scores, o_lat, lse);
        free(scores);
    }
}

/* Sparse top-k attention ([AI] 6: a selector keeps k cached tokens per query
 * token, they are gathered by index and the scoring and the weighted sum run
 * over them only): row r = (b*s_q + i)*H + h attends over the entries
 * idx[b][i][0 .. topk) that name a visible token (0 <= j <= L - s_q + i;
 * other entries, such as -1 padding, take no part), each entry as listed,
 * with the same score and latent-space sum as orc_attend.  A row with no
 * visible entry gets o_lat = 0 and lse = -inf. */
static void attend_row_sparse(const orc_dims *d, const double *q_cat, const orc_cache *c,
                              const int32_t *idx, int topk, long long r, double *scores,
                              double *o_lat, double *lse)
{
    long long bi = r / d->H;
    int i = (int)(bi % d->s_q);
    int b = (int)(bi / d->s_q);
    long long wq = (long long)d->d_c + d->d_rope;
    const double *q = q_cat + r * wq;
    double *o = o_lat + r * d->d_c;
    if (!row_is_valid(d, c, b)) {
        for (int k = 0; k < d->d_c; ++k) o[k] = NAN;
        lse[r] = NAN;
        return;
    }
    long long lim = c->seq_lens[b] - d->s_q + i;
    const int32_t *list = idx + bi * topk;
    double m = -INFINITY;
    for (int e = 0; e < topk; ++e) {
        long long j = list[e];
        scores[e] = -INFINITY;
        if (j < 0 || j > lim) continue;
        const void *t = token_row(d, c, b, j);
        double dot = 0.0;
        for (long long k = 0; k < wq; ++k)
            dot += q[k] * row_elem(c, t, k);
        scores[e] = d->scale * dot;
        if (scores[e] > m) m = scores[e];
    }
    for (int k = 0; k < d->d_c; ++k) o[k] = 0.0;
    if (m == -INFINITY) {
        lse[r] = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int e = 0; e < topk; ++e)
        if (scores[e] != -INFINITY) sum += exp(scores[e] - m);
    double l = m + log(sum);
    for (int e = 0; e < topk; ++e) {
        if (scores[e] == -INFINITY) continue;
        double p = exp(scores[e] - l);
        const void *t = token_row(d, c, b, list[e]);
        for (int k = 0; k < d->d_c; ++k)
            o[k] += p * row_elem(c, t, k);
    }
    lse[r] = l;
}

void orc_attend_sparse(const orc_dims *d, const double *q_cat, const orc_cache *c,
                       const int32_t *idx, int topk, const long long *rows, long long n_rows,
                       double *o_lat, double *lse)
{
    long long total = rows ? n_rows : (long long)d->B * d->s_q * d->H;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
#pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < total; ++t)
            attend_row_sparse(d, q_cat, c, idx, topk, rows ? rows[t] : t, scores, o_lat, lse);
        free(scores);
    }
}

/* Unnormalised partial over the visible tokens of row r that fall in [j0, j1):
 * m = max s_j (-inf if none), l = sum exp(s_j - m), acc[c] = sum exp(s_j - m) c_kv[j,c].
 * Used to pin the cross-split merge below. */
void orc_attend_partial(const orc_dims *d, const double *q_cat, const orc_cache *c,
                        long long r, long long j0, long long j1,
                        double *m_out, double *l_out, double *acc)
{
    long long bi = r / d->H;
    int i = (int)(bi % d->s_q);
    int b = (int)(bi / d->s_q);
    long long wq = (long long)d->d_c + d->d_rope;
    const double *q = q_cat + r * wq;
    long long L = c->seq_lens[b];
    long long lim = L - d->s_q + i + 1;
    if (j1 > lim) j1 = lim;
    double m = -INFINITY;
    for (int k = 0; k < d->d_c; ++k) acc[k] = 0.0;
    for (long long j = j0; j < j1; ++j) {
        const void *t = token_row(d, c, b, j);
        double dot = 0.0;
        for (long long k = 0; k < wq; ++k) dot += q[k] * row_elem(c, t, k);
        double s = d->scale * dot;
        if (s > m) m = s;
    }
    double l = 0.0;
    if (m != -INFINITY) {
        for (long long j = j0; j < j1; ++j) {
            const void *t = token_row(d, c, b, j);
            double dot = 0.0;
            for (long long k = 0; k < wq; ++k) dot += q[k] * row_elem(c, t, k);
            double e = exp(d->scale * dot - m);
            l += e;
            for (int k = 0; k < d->d_c; ++k) acc[k] += e * row_elem(c, t, k);
        }
    }
    *m_out = m;
    *l_out = l;
}

/* Merge of n partials (m_s, l_s, acc_s) of one row into the whole-row result:
 *     M = max_s m_s,  L = sum_s l_s exp(m_s - M),
 *     o = sum_s acc_s exp(m_s - M) / L,  lse = M + ln L.
 * A partial with no visible token (m = -inf, l = 0) carries weight 0; a row
 * with no visible token at all gives o = 0, lse = -inf. */
void orc_combine(int n, int width, const double *m, const double *l, const double *acc,
                 double *o, double *lse)
{
    double M = -INFINITY;
    for (int s = 0; s < n; ++s)
        if (m[s] > M) M = m[s];
    for (int k = 0; k < width; ++k) o[k] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double Lsum = 0.0;
    for (int s = 0; s < n; ++s) {
        if (m[s] == -INFINITY) continue;
        double w = exp(m[s] - M);
        Lsum += l[s] * w;
        for (int k = 0; k < width; ++k) o[k] += acc[(long long)s * width + k] * w;
    }
    for (int k = 0; k < width; ++k) o[k] /= Lsum;
    *lse = M + log(Lsum);
}

/* Project the latent-space output back to each head's value width
 * ([MLA-dim] "MLA Decode", decode value order; [AI] 3.2; [speedup] "The absorbed
 * form", final einsum):  out[b,i,h,v] = sum_c o_lat[b,i,h,c] * W_UV[h,c,v].
 * Layouts: o_lat [B][s_q][H][d_c], W_UV [H][d_c][d_v], out [B][s_q][H][d_v]. */
void orc_out_proj(const orc_dims *d, const double *o_lat, const uint16_t *w_uv, double *out)
{
    long long rows = (long long)d->B * d->s_q * d->H;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        int h = (int)(r % d->H);
        const double *ol = o_lat + r * d->d_c;
        double *o = out + r * d->d_v;
        for (int v = 0; v < d->d_v; ++v) o[v] = 0.0;
        for (int c = 0; c < d->d_c; ++c) {
            const uint16_t *wrow = w_uv + ((long long)h * d->d_c + c) * d->d_v;
            double a = ol[c];
            for (int v = 0; v < d->d_v; ++v) o[v] += a * bf16_to_f64(wrow[v]);
        }
    }
}

/* Latent down-projection of the new tokens ([MLA-dim] "MLA Decode": the
 * current token's hidden state is compressed, x . W_DKV -> c^KV of width d_c, and
 * appended to the cache; [AI] 4.1, the 2 d_model d_c FLOPs of F_fixed):
 *     c[m,k] = sum_i x[m,i] * W_DKV[i,k]
 * Layouts: x [M][d_model], W_DKV [d_model][d_c], c [M][d_c]. */
void orc_down_proj(long long M, int d_model, int d_c, const uint16_t *x, const uint16_t *w_dkv, double *c)
{
#pragma omp parallel for schedule(static)
    for (long long m = 0; m < M; ++m) {
        double *out = c + m * d_c;
        for (int k = 0; k < d_c; ++k) out[k] = 0.0;
        for (int i = 0; i < d_model; ++i) {
            double a = bf16_to_f64(x[m * d_model + i]);
            const uint16_t *wrow = w_dkv + (long long)i * d_c;
            for (int k = 0; k < d_c; ++k) out[k] += a * bf16_to_f64(wrow[k]);
        }
    }
}

/* Naive decompress-then-attend ([speedup] "The naive form, written out";
 * [AI] 3.3; [intens] decompression cost): every visible cached latent of the
 * sequence is up-projected per head,
 *     K[j,n] = sum_c c_kv[j,c] W_UK[h,c,n],   V[j,v] = sum_c c_kv[j,c] W_UV[h,c,v],
 * then standard attention with the decoupled RoPE key appended to the score:
 *     s_j = scale * ( sum_n q_nope[n] K[j,n] + sum_k q_rope[k] k_rope[j,k] ),
 *     out[v] = sum_j softmax(s)_j V[j,v].
 * Each listed row re-expands its own sequence's visible tokens for its head
 * (nothing is shared between rows: this is the slow form, on purpose).  Rows are
 * listed as in orc_attend (NULL = all); out [B][s_q][H][d_v], lse [B][s_q][H]. */
void orc_naive(const orc_dims *d, const uint16_t *q_nope, const uint16_t *q_rope,
               const orc_cache *c, const uint16_t *w_uk, const uint16_t *w_uv,
               const long long *rows, long long n_rows, double *out, double *lse)
{
    long long total = rows ? n_rows : (long long)d->B * d->s_q * d->H;
    long long cap = max_visible(d, c);
#pragma omp parallel
    {
        double *K = (double *)malloc(sizeof(double) * (size_t)(cap * d->d_nope));
        double *V = (double *)malloc(sizeof(double) * (size_t)(cap * d->d_v));
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
#pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < total; ++t) {
            long long r = rows ? rows[t] : t;
            int h = (int)(r % d->H);
            long long bi = r / d->H;
            int i = (int)(bi % d->s_q);
            int b = (int)(bi / d->s_q);
            double *o = out + r * d->d_v;
            if (!row_is_valid(d, c, b)) {
                for (int v = 0; v < d->d_v; ++v) o[v] = NAN;
                lse[r] = NAN;
                continue;
            }
            long long L = c->seq_lens[b];
            long long n_vis = L - d->s_q + i + 1;
            for (long long j = 0; j < n_vis; ++j) {
                const void *tok = token_row(d, c, b, j);
                for (int n = 0; n < d->d_nope; ++n) K[j * d->d_nope + n] = 0.0;
                for (int v = 0; v < d->d_v; ++v) V[j * d->d_v + v] = 0.0;
                for (int cc = 0; cc < d->d_c; ++cc) {
                    double x = row_elem(c, tok, cc);
                    const uint16_t *wk = w_uk + ((long long)h * d->d_c + cc) * d->d_nope;
                    const uint16_t *wv = w_uv + ((long long)h * d->d_c + cc) * d->d_v;
                    for (int n = 0; n < d->d_nope; ++n) K[j * d->d_nope + n] += x * bf16_to_f64(wk[n]);
                    for (int v = 0; v < d->d_v; ++v) V[j * d->d_v + v] += x * bf16_to_f64(wv[v]);
                }
            }
            const uint16_t *qn = q_nope + r * d->d_nope;
            const uint16_t *qr = q_rope + r * d->d_rope;
            double m = -INFINITY;
            for (long long j = 0; j < n_vis; ++j) {
                const void *tok = token_row(d, c, b, j);
                double dot = 0.0;
                for (int n = 0; n < d->d_nope; ++n) dot += bf16_to_f64(qn[n]) * K[j * d->d_nope + n];
                for (int k = 0; k < d->d_rope; ++k) dot += bf16_to_f64(qr[k]) * row_elem(c, tok, d->d_c + k);
                scores[j] = d->scale * dot;
                if (scores[j] > m) m = scores[j];
            }
            double sum = 0.0;
            for (long long j = 0; j < n_vis; ++j) sum += exp(scores[j] - m);
            double l = m + log(sum);
            for (int v = 0; v < d->d_v; ++v) o[v] = 0.0;
            for (long long j = 0; j < n_vis; ++j) {
                double p = exp(scores[j] - l);
                for (int v = 0; v < d->d_v; ++v) o[v] += p * V[j * d->d_v + v];
            }
            lse[r] = l;
        }
        free(K);
        free(V);
        free(scores);
    }
}
