/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, single-threaded CPU statement, in double precision, of what the
 * hybrid compressed attention (CSA + HCA) of DeepSeek-V4 computes.  It exists only
 * so that tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm can check and time the CUDA library against it.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (web pages on DeepSeek-V4, cited by address and section):
 *   [P1] gxgjx.lffhtl.com/lxrt/355279.html, section "混肃穆力机制" (hybrid attention):
 *        CSA steps one to four, the HCA paragraph, and the tricks list
 *        (Q/KV normalization, Partial RoPE with the output RoPE at -i,
 *        sliding-window branch, attention sink).
 *   [P4] zhinnengdao.top, "DeepSeek-V4开源解读", section 3.1 "Hybrid Attention: CSA + HCA"
 *        (Flash hyper-parameters: m=4, 64 indexer heads of dim 128, top-k 512,
 *        m'=128, RoPE on the last 64 dims, one sink logit per head, SWA branch).
 * Where the pages leave a step open the plainest reading is taken; each such
 * reading is named at the function that encodes it.
 *
 * Conventions: bf16 values arrive as their raw 16-bit patterns (uint16_t) and are
 * widened exactly to double.  Every sum is a left-to-right loop in double.
 * Functions return 0 on success and a negative code when the inputs do not hold
 * what the definition needs (a missing token, an index out of range).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE fp32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Partial RoPE ([P1] "Partial RoPE"; [P4] 3.1 "最后64维加RoPE").
 * Rotates only the trailing R dims of x[0..c).  Reading taken (pages silent):
 * half-split pairing -- pair d (0 <= d < R/2) is (x[c-R+d], x[c-R+d+R/2]) --
 * frequency theta_d = base^(-2d/R), rotation angle pos * theta_d, and the
 * rotation (a, b) -> (a cos - b sin, a sin + b cos).
 */
static void rope_rotate(double *x, int c, int R, double base, double pos)
{
    int half = R / 2;
    for (int d = 0; d < half; ++d) {
        double theta = pow(base, -2.0 * (double)d / (double)R);
        double angle = pos * theta;
        double cs = cos(angle), sn = sin(angle);
        double a = x[c - R + d];
        double b = x[c - R + d + half];
        x[c - R + d] = a * cs - b * sn;
        x[c - R + d + half] = a * sn + b * cs;
    }
}

/*
 * RMSNorm ([P1] "Q/KV normalization": queries and KV entries are RMS-normalised
 * before core attention).  y_i = x_i / sqrt(mean(x^2) + eps) * gamma_i.
 */
static void rms_normalize(double *x, int c, const float *gamma, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < c; ++i)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)c + eps);
    for (int i = 0; i < c; ++i)
        x[i] = x[i] * inv * (double)gamma[i];
}

/*
 * KV compression, CSA step one and the HCA compressor ([P1] "步，KV 压缩" and the
 * HCA paragraph; [P4] 3.1: m=4 for CSA, m'=128 for HCA).
 *
 * Entry j pools the tokens t in [stride*(j+1) - span, stride*(j+1)), clipped at 0:
 *   CSA: span = 2m, stride = m  (overlapping windows of 2m, one entry per m tokens)
 *   HCA: span = stride = m'     (no overlap)
 * Learned softmax pooling, reading taken: a scalar logit z_t per token plus a
 * learned bias b[r] per offset r = t - (stride*(j+1) - span) inside the nominal
 * window (so a window clipped at position 0 keeps the offsets of its surviving
 * tokens); weights a_t = softmax over the surviving tokens of (z_t + b[r]);
 * u_j = sum_t a_t v_t.  Then, when gamma is given, RMSNorm with gamma, and when
 * rope_dims > 0, RoPE at the entry's position p_j = stride*(j+1) - 1 (its last token).
 *
 * tok_v[t_local*width + i], tok_z[t_local] hold token tok_pos0 + t_local.
 * out[(e*width) + i] receives entry first_entry + e, e < n_new.
 */
int orc_compress(int span, int stride, int width,
                 const uint16_t *tok_v, const float *tok_z, long tok_pos0, long n_tok,
                 const float *bias, const float *gamma, double eps,
                 int rope_dims, double rope_base,
                 long first_entry, long n_new, double *out)
{
    double *u = (double *)malloc(sizeof(double) * (size_t)width);
    if (!u)
        return -3;
    for (long e = 0; e < n_new; ++e) {
        long j = first_entry + e;
        long end = (long)stride * (j + 1);      /* one past the entry's last token */
        long nominal_begin = end - span;
        long begin = nominal_begin < 0 ? 0 : nominal_begin;
        if (begin < tok_pos0 || end > tok_pos0 + n_tok) {
            free(u);
            return -1;
        }
        double zmax = -INFINITY;
        for (long t = begin; t < end; ++t) {
            double s = (double)tok_z[t - tok_pos0] + (double)bias[t - nominal_begin];
            if (s > zmax)
                zmax = s;
        }
        double den = 0.0;
        for (long t = begin; t < end; ++t) {
            double s = (double)tok_z[t - tok_pos0] + (double)bias[t - nominal_begin];
            den += exp(s - zmax);
        }
        for (int i = 0; i < width; ++i)
            u[i] = 0.0;
        for (long t = begin; t < end; ++t) {
            double s = (double)tok_z[t - tok_pos0] + (double)bias[t - nominal_begin];
            double a = exp(s - zmax) / den;
            const uint16_t *v = tok_v + (size_t)(t - tok_pos0) * (size_t)width;
            for (int i = 0; i < width; ++i)
                u[i] += a * bf16_bits_to_double(v[i]);
        }
        if (gamma)
            rms_normalize(u, width, gamma, eps);
        if (rope_dims > 0)
            rope_rotate(u, width, rope_dims, rope_base, (double)(end - 1));
        memcpy(out + (size_t)e * (size_t)width, u, sizeof(double) * (size_t)width);
    }
    free(u);
    return 0;
}

/*
 * One row of the sliding-window branch ([P1] "Sliding window attention": each query
 * also sees the uncompressed KV of the most recent tokens).  Reading taken: the
 * uncompressed row of token t is that token's own KV vector, RMS-normalised with
 * the KV gamma and rotated by RoPE at position t, like every other key.
 */
void orc_window_row(int c, const uint16_t *v, const float *gamma, double eps,
                    int rope_dims, double rope_base, long pos, double *out)
{
    for (int i = 0; i < c; ++i)
        out[i] = bf16_bits_to_double(v[i]);
    rms_normalize(out, c, gamma, eps);
    if (rope_dims > 0)
        rope_rotate(out, c, rope_dims, rope_base, (double)pos);
}

/*
 * Lightning indexer, CSA step two ([P1] "二步，lightning indexer + top-k";
 * [P4] 3.1: 64 indexer query heads of dim 128).  The pages give no formula; the
 * one taken is the DeepSeek-V3.2 indexer score
 *     s_j = sum_h w_h * ReLU(q_h . k_j),   j < n_vis,
 * with no RoPE and no normalisation inside the indexer.
 * q[h*dim + d], w[h], keys[j*dim + d]; out[j] for j < n_vis.
 */
void orc_indexer_scores(int n_heads, int dim, const uint16_t *q, const float *w,
                        const uint16_t *keys, long n_vis, double *out)
{
    for (long j = 0; j < n_vis; ++j) {
        const uint16_t *k = keys + (size_t)j * (size_t)dim;
        double s = 0.0;
        for (int h = 0; h < n_heads; ++h) {
            double dot = 0.0;
            for (int d = 0; d < dim; ++d)
                dot += bf16_bits_to_double(q[h * dim + d]) * bf16_bits_to_double(k[d]);
            double relu = dot > 0.0 ? dot : 0.0;
            s += (double)w[h] * relu;
        }
        out[j] = s;
    }
}

/* Visible entries for a query at position pos ([P1]: compressed attention is strictly
 * causal, a query does not see the block it is in): entry j is visible iff its last
 * token m*(j+1)-1 is at or before pos, i.e. n_vis = floor((pos+1)/m). */
long orc_visible_entries(long pos, int ratio)
{
    return (pos + 1) / ratio;
}

typedef struct {
    double score;
    int32_t index;
} scored_entry;

/* (score descending, index ascending): the lower index wins a tie. */
static int by_score_then_index(const void *pa, const void *pb)
{
    const scored_entry *a = (const scored_entry *)pa, *b = (const scored_entry *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    return (a->index > b->index) - (a->index < b->index);
}

static int by_index(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * Top-k selection ([P1] CSA step two and "n/m 造成 top-k"; [P4] 3.1 top-k=512).
 * The first min(k, n) entries of the total order (score descending, index
 * ascending), written in ascending index order, the rest of out[0..k) set to -1.
 */
int orc_topk(const double *scores, long n, int k, int32_t *out)
{
    scored_entry *all = (scored_entry *)malloc(sizeof(scored_entry) * (size_t)(n > 0 ? n : 1));
    if (!all)
        return -3;
    for (long j = 0; j < n; ++j) {
        all[j].score = scores[j];
        all[j].index = (int32_t)j;
    }
    qsort(all, (size_t)n, sizeof(scored_entry), by_score_then_index);
    long take = n < k ? n : k;
    for (long i = 0; i < take; ++i)
        out[i] = all[i].index;
    qsort(out, (size_t)take, sizeof(int32_t), by_index);
    for (long i = take; i < k; ++i)
        out[i] = -1;
    free(all);
    return 0;
}

/*
 * Core attention for one query, CSA step three and HCA's dense attention, with the
 * tricks of [P1] (Q/KV normalisation, partial RoPE, output RoPE at -i,
 * sliding-window branch, attention sink) and [P4] 3.1.
 *
 * Key set (each row is both key and value, Multi-Query: one set shared by all heads):
 *   - compressed rows: comp[idx[i]] for every idx[i] >= 0 (CSA, idx != NULL), or
 *     comp[0 .. n_dense) (HCA, idx == NULL);
 *   - window rows: tokens t in [max(0, pos-W+1), pos] read from the ring at row
 *     t mod win_cap.  A token present both in the window and inside a chosen
 *     entry is counted in both (reading taken: no de-duplication).
 * Per head h:
 *   q_h = RoPE(RMSNorm(q_h) * gamma_q, pos);  l_r = scale * (q_h . row_r);
 *   p_r = exp(l_r) / (exp(sink_h) + sum_r exp(l_r));   (sink: denominator only)
 *   o_h = RoPE(sum_r p_r row_r, -pos);   lse_h = log(exp(sink_h) + sum_r exp(l_r)).
 * Rows already carry RMSNorm and RoPE at their own positions.
 */
/* One key/value row of the attention: bf16 bit patterns, or (variant) e4m3 codes with the
 * row's scale, read back as scale * value(code). */
typedef struct {
    const uint16_t *bf;
    const uint8_t *e8;
    double scale;
} key_row;

double orc_e4m3_decode(uint8_t c);

static double key_row_value(const key_row *r, int i)
{
    return r->bf ? bf16_bits_to_double(r->bf[i]) : r->scale * orc_e4m3_decode(r->e8[i]);
}

/* The per-head part of orc_attend over an assembled row list. */
static int attend_rows(int H, int c, int rope_dims, double rope_base, double eps, double scale,
                       const uint16_t *q, const float *gamma_q, long pos, const key_row *rows, long n_rows,
                       const float *sink, double *out, double *lse)
{
    double *qh = (double *)malloc(sizeof(double) * (size_t)c);
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)c);
    if (!qh || !logit || !acc) {
        free(qh); free(logit); free(acc);
        return -3;
    }
    for (int h = 0; h < H; ++h) {
        for (int i = 0; i < c; ++i)
            qh[i] = bf16_bits_to_double(q[(size_t)h * (size_t)c + i]);
        rms_normalize(qh, c, gamma_q, eps);
        if (rope_dims > 0)
            rope_rotate(qh, c, rope_dims, rope_base, (double)pos);

        double mx = (double)sink[h];
        for (long r = 0; r < n_rows; ++r) {
            double dot = 0.0;
            for (int i = 0; i < c; ++i)
                dot += qh[i] * key_row_value(&rows[r], i);
            logit[r] = scale * dot;
            if (logit[r] > mx)
                mx = logit[r];
        }
        double den = exp((double)sink[h] - mx);
        for (long r = 0; r < n_rows; ++r)
            den += exp(logit[r] - mx);
        for (int i = 0; i < c; ++i)
            acc[i] = 0.0;
        for (long r = 0; r < n_rows; ++r) {
            double p = exp(logit[r] - mx) / den;
            for (int i = 0; i < c; ++i)
                acc[i] += p * key_row_value(&rows[r], i);
        }
        if (rope_dims > 0)
            rope_rotate(acc, c, rope_dims, rope_base, -(double)pos);
        memcpy(out + (size_t)h * (size_t)c, acc, sizeof(double) * (size_t)c);
        if (lse)
            lse[h] = mx + log(den);
    }
    free(qh); free(logit); free(acc);
    return 0;
}

/* The row list of one query: the compressed rows (comp bf16, or comp8 with comp_scale) then the
 * window rows.  Returns the count, or -2 for an index outside the cache, -3 for no memory. */
static long gather_key_rows(int c, long pos, const uint16_t *comp, const uint8_t *comp8, const float *comp_scale,
                            long comp_rows, const int32_t *idx, long n_idx, long n_dense,
                            const uint16_t *win, long win_cap, long W, key_row **out_rows)
{
    long win_begin = pos - W + 1;
    if (win_begin < 0)
        win_begin = 0;
    long n_win = pos - win_begin + 1;
    long n_comp = idx ? n_idx : n_dense;
    long max_rows = n_comp + n_win;
    key_row *rows = (key_row *)malloc(sizeof(key_row) * (size_t)(max_rows > 0 ? max_rows : 1));
    if (!rows)
        return -3;
    long n_rows = 0;
    for (long i = 0; i < n_comp; ++i) {
        long j = idx ? (long)idx[i] : i;
        if (j < 0)
            continue;
        if (j >= comp_rows) {
            free(rows);
            return -2;
        }
        key_row kr = {0, 0, 0.0};
        if (comp8) {
            kr.e8 = comp8 + (size_t)j * (size_t)c;
            kr.scale = (double)comp_scale[j];
        } else {
            kr.bf = comp + (size_t)j * (size_t)c;
        }
        rows[n_rows++] = kr;
    }
    for (long t = win_begin; t <= pos; ++t) {
        key_row kr = {win + (size_t)(t % win_cap) * (size_t)c, 0, 0.0};
        rows[n_rows++] = kr;
    }
    *out_rows = rows;
    return n_rows;
}

int orc_attend(int H, int c, int rope_dims, double rope_base, double eps, double scale,
               const uint16_t *q, const float *gamma_q, long pos,
               const uint16_t *comp, long comp_rows,
               const int32_t *idx, long n_idx, long n_dense,
               const uint16_t *win, long win_cap, long W,
               const float *sink, double *out, double *lse)
{
    key_row *rows = 0;
    long n_rows = gather_key_rows(c, pos, comp, 0, 0, comp_rows, idx, n_idx, n_dense, win, win_cap, W, &rows);
    if (n_rows < 0)
        return (int)n_rows;
    int rc = attend_rows(H, c, rope_dims, rope_base, eps, scale, q, gamma_q, pos, rows, n_rows, sink, out, lse);
    free(rows);
    return rc;
}

/*
 * The same attention over an e4m3 compressed cache (the FP8 variant): compressed row j is
 * comp_scale[j] * e4m3(comp8[j][.]); the window rows stay bf16.
 */
int orc_attend_e4m3(int H, int c, int rope_dims, double rope_base, double eps, double scale,
                    const uint16_t *q, const float *gamma_q, long pos,
                    const uint8_t *comp8, const float *comp_scale, long comp_rows,
                    const int32_t *idx, long n_idx, long n_dense,
                    const uint16_t *win, long win_cap, long W,
                    const float *sink, double *out, double *lse)
{
    key_row *rows = 0;
    long n_rows = gather_key_rows(c, pos, 0, comp8, comp_scale, comp_rows, idx, n_idx, n_dense, win, win_cap, W,
                                  &rows);
    if (n_rows < 0)
        return (int)n_rows;
    int rc = attend_rows(H, c, rope_dims, rope_base, eps, scale, q, gamma_q, pos, rows, n_rows, sink, out, lse);
    free(rows);
    return rc;
}

/* Plain matrix product out[m*N + n] = sum_k A[m*K + k] * B[n*K + k] (bf16 inputs). */
void orc_gemm_bf16(long M, long N, long K, const uint16_t *A, const uint16_t *B, double *out)
{
    for (long m = 0; m < M; ++m)
        for (long n = 0; n < N; ++n) {
            double s = 0.0;
            for (long k = 0; k < K; ++k)
                s += bf16_bits_to_double(A[m * K + k]) * bf16_bits_to_double(B[n * K + k]);
            out[m * N + n] = s;
        }
}

/*
 * Grouped output projection, CSA step four ([P1] "四步，grouped output projection"):
 * the H heads' outputs (each of dim c) are split into G groups of H/G heads; group g
 * is projected by its own matrix Wg[g] (d_g x (H/G)*c) to d_g; the G results are
 * concatenated and projected by Wm (d_model x G*d_g).  Reading taken: two linear maps,
 * no bias, no activation in between.
 * o[h*c + i] (bf16), Wg[(g*d_g + r)*(H/G*c) + k], Wm[(n)*(G*d_g) + k]; y[n].
 */
int orc_grouped_oproj(int H, int c, int G, int d_g, int d_model,
                      const uint16_t *o, const uint16_t *Wg, const uint16_t *Wm, double *y)
{
    if (G <= 0 || H % G != 0)
        return -2;
    long in_g = (long)(H / G) * c;
    double *mid = (double *)malloc(sizeof(double) * (size_t)G * (size_t)d_g);
    if (!mid)
        return -3;
    for (int g = 0; g < G; ++g)
        for (int r = 0; r < d_g; ++r) {
            const uint16_t *wrow = Wg + ((size_t)g * d_g + r) * (size_t)in_g;
            const uint16_t *og = o + (size_t)g * (size_t)in_g;
            double s = 0.0;
            for (long k = 0; k < in_g; ++k)
                s += bf16_bits_to_double(wrow[k]) * bf16_bits_to_double(og[k]);
            mid[(size_t)g * d_g + r] = s;
        }
    for (int n = 0; n < d_model; ++n) {
        const uint16_t *wrow = Wm + (size_t)n * (size_t)G * (size_t)d_g;
        double s = 0.0;
        for (long k = 0; k < (long)G * d_g; ++k)
            s += bf16_bits_to_double(wrow[k]) * mid[k];
        y[n] = s;
    }
    free(mid);
    return 0;
}

/*
 * Manifold-constrained hyper-connections ([P1] section "mHC，给残差集结加层连续"; [P4] section
 * 3.2 "mHC"): the residual stream is widened to n parallel streams x[i] (i < n, width d) and
 * each layer mixes them with three maps: A (n weights that form the layer's input), B (an n x n
 * mixing of the streams) and C (n weights that spread the layer's output back over the
 * streams).  The maps are generated per token from the input (an input-dependent linear part
 * plus an input-independent bias); A and C pass through a sigmoid (non-negative, bounded); B is
 * projected onto the doubly stochastic matrices (rows and columns summing to 1) by the
 * Sinkhorn-Knopp iteration, row and column normalisations taken in turn, 20 times on the page.
 * Readings (the pages give no formula): z = flatten(x) . Phi^T + bias with Phi holding one row
 * of n*d weights per generated value, in the order a (n values), c (n values), B (n*n, row-major);
 * B starts from exp(z) (a positive matrix, as Sinkhorn-Knopp requires); one iteration is a row
 * normalisation followed by a column normalisation; the layer input is h = sum_i a_i x[i]; after
 * the layer, x'[i] = sum_j B[i][j] x[j] + c_i y with y the layer's output.
 */

/* The generated coefficients of one token: a[n], c[n] (sigmoids) and B[n*n] (Sinkhorn-Knopp). */
void orc_mhc_coeffs(int n, long d, int iters, const uint16_t *x, const uint16_t *phi, const float *bias,
                    double *a, double *c, double *B)
{
    const long nd = (long)n * d;
    const int K = 2 * n + n * n;
    double *z = (double *)malloc(sizeof(double) * (size_t)K);
    if (!z)
        return;
    for (int k = 0; k < K; ++k) {
        double s = 0.0;
        for (long f = 0; f < nd; ++f)
            s += bf16_bits_to_double(x[f]) * bf16_bits_to_double(phi[(size_t)k * (size_t)nd + (size_t)f]);
        z[k] = s + (double)bias[k];
    }
    for (int i = 0; i < n; ++i) {
        a[i] = 1.0 / (1.0 + exp(-z[i]));
        c[i] = 1.0 / (1.0 + exp(-z[n + i]));
    }
    for (int e = 0; e < n * n; ++e)
        B[e] = exp(z[2 * n + e]);
    for (int it = 0; it < iters; ++it) {
        for (int i = 0; i < n; ++i) {           /* rows */
            double s = 0.0;
            for (int j = 0; j < n; ++j)
                s += B[i * n + j];
            for (int j = 0; j < n; ++j)
                B[i * n + j] /= s;
        }
        for (int j = 0; j < n; ++j) {           /* columns */
            double s = 0.0;
            for (int i = 0; i < n; ++i)
                s += B[i * n + j];
            for (int i = 0; i < n; ++i)
                B[i * n + j] /= s;
        }
    }
    free(z);
}

/* The layer input of one token: h[e] = sum_i a[i] x[i][e]. */
void orc_mhc_pre(int n, long d, const uint16_t *x, const double *a, double *h)
{
    for (long e = 0; e < d; ++e) {
        double s = 0.0;
        for (int i = 0; i < n; ++i)
            s += a[i] * bf16_bits_to_double(x[(size_t)i * (size_t)d + (size_t)e]);
        h[e] = s;
    }
}

/* The streams after the layer: xo[i][e] = sum_j B[i][j] x[j][e] + c[i] y[e]. */
void orc_mhc_post(int n, long d, const uint16_t *x, const double *B, const double *c, const uint16_t *y, double *xo)
{
    for (int i = 0; i < n; ++i)
        for (long e = 0; e < d; ++e) {
            double s = c[i] * bf16_bits_to_double(y[e]);
            for (int j = 0; j < n; ++j)
                s += B[i * n + j] * bf16_bits_to_double(x[(size_t)j * (size_t)d + (size_t)e]);
            xo[(size_t)i * (size_t)d + (size_t)e] = s;
        }
}

/*
 * ----------------------------------------------------------------------------------
 * FP8 caches and the per-channel compressor (variants of the path, not fixed by the
 * pages: the news summary ynrysl.com, paragraph on HCA, mentions FP8 storage only in
 * passing, and [P1] CSA step one calls the compressor's weighting "learned" without
 * giving its shape).
 *
 * e4m3 (the 8-bit float with 1 sign, 4 exponent and 3 mantissa bits, exponent bias 7,
 * no infinities, S.1111.111 NaN): a code c >= 0x08 (magnitude bits) is normal,
 * (-1)^s 2^(e-7) (1 + m/8); e = 0 is subnormal, (-1)^s 2^-6 (m/8).  The largest finite
 * magnitude is 2^8 * 1.75 = 448.
 */
double orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * e4m3 code of a float: the nearest finite e4m3 value, a tie going to the code with an
 * even mantissa (round to nearest even), magnitudes beyond 448 saturating to 448 (the
 * "satfinite" conversion).  Found by comparing against every finite magnitude code,
 * so that no step of a bit-level conversion can be wrong.  NaN gives 0x7F.
 */
uint8_t orc_e4m3_encode(float x)
{
    if (x != x)
        return 0x7F;
    uint8_t sign = (signbit(x) ? 0x80 : 0);
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/*
 * Per-row e4m3 quantisation of bf16 rows (reading taken for "FP8 caches": one fp32
 * scale per row, the row's largest magnitude mapped to 448):
 *     amax = max_i |x_i|,  scale = amax / 448 (fp32),  code_i = e4m3(x_i / scale) (fp32
 *     division), and x_i is read back as scale * e4m3_value(code_i).
 * An all-zero row gets scale 0 and zero codes.  The divisions are single-precision
 * because they decide the codes: both sides round them the same way.
 */
void orc_quantize_rows_e4m3(long rows, int width, const uint16_t *x, uint8_t *q, float *scale)
{
    for (long r = 0; r < rows; ++r) {
        const uint16_t *xr = x + (size_t)r * (size_t)width;
        float amax = 0.0f;
        for (int i = 0; i < width; ++i) {
            float v = (float)fabs(bf16_bits_to_double(xr[i]));
            if (v > amax)
                amax = v;
        }
        volatile float s = amax / 448.0f;
        scale[r] = s;
        for (int i = 0; i < width; ++i) {
            if (amax == 0.0f) {
                q[(size_t)r * (size_t)width + (size_t)i] = 0;
                continue;
            }
            volatile float y = (float)bf16_bits_to_double(xr[i]) / s;
            q[(size_t)r * (size_t)width + (size_t)i] = orc_e4m3_encode(y);
        }
    }
}

/* The value of row r, channel i of a per-row-scaled e4m3 array. */
static double e4m3_value(const uint8_t *q, const float *scale, long r, int width, int i)
{
    return (double)scale[r] * orc_e4m3_decode(q[(size_t)r * (size_t)width + (size_t)i]);
}

/*
 * The compressor with per-channel weights (reading taken for the open shape of [P1] CSA
 * step one's "learned" weighting): each channel i has its own logit per token,
 * z[t][i], and its own learned offset bias, bias[r][i]; the softmax over the window is
 * taken per channel:
 *     a_{t,i} = exp(z[t][i] + bias[t - nominal][i]) / sum_{t'} exp(z[t'][i] + bias[...][i]),
 *     u_i = sum_t a_{t,i} v[t][i];
 * then RMSNorm and RoPE as in orc_compress.  With every channel's logits and biases
 * equal it is orc_compress.
 */
int orc_compress_pc(int span, int stride, int width,
                    const uint16_t *tok_v, const float *tok_z, long tok_pos0, long n_tok,
                    const float *bias, const float *gamma, double eps,
                    int rope_dims, double rope_base,
                    long first_entry, long n_new, double *out)
{
    double *u = (double *)malloc(sizeof(double) * (size_t)width);
    if (!u)
        return -3;
    for (long e = 0; e < n_new; ++e) {
        long j = first_entry + e;
        long end = (long)stride * (j + 1);
        long nominal_begin = end - span;
        long begin = nominal_begin < 0 ? 0 : nominal_begin;
        if (begin < tok_pos0 || end > tok_pos0 + n_tok) {
            free(u);
            return -1;
        }
        for (int i = 0; i < width; ++i) {
            double zmax = -INFINITY;
            for (long t = begin; t < end; ++t) {
                double s = (double)tok_z[(size_t)(t - tok_pos0) * (size_t)width + (size_t)i] +
                           (double)bias[(size_t)(t - nominal_begin) * (size_t)width + (size_t)i];
                if (s > zmax)
                    zmax = s;
            }
            double den = 0.0, num = 0.0;
            for (long t = begin; t < end; ++t) {
                double s = (double)tok_z[(size_t)(t - tok_pos0) * (size_t)width + (size_t)i] +
                           (double)bias[(size_t)(t - nominal_begin) * (size_t)width + (size_t)i];
                double wgt = exp(s - zmax);
                den += wgt;
                num += wgt * bf16_bits_to_double(tok_v[(size_t)(t - tok_pos0) * (size_t)width + (size_t)i]);
            }
            u[i] = num / den;
        }
        if (gamma)
            rms_normalize(u, width, gamma, eps);
        if (rope_dims > 0)
            rope_rotate(u, width, rope_dims, rope_base, (double)(end - 1));
        memcpy(out + (size_t)e * (size_t)width, u, sizeof(double) * (size_t)width);
    }
    free(u);
    return 0;
}

/*
 * Lightning-indexer scores over e4m3 rows: the same score as orc_indexer_scores,
 *     s_j = sum_h w_h ReLU(q_h . k_j),
 * with q_h = qscale[h] * e4m3(q8[h][.]) and k_j = kscale[j] * e4m3(k8[j][.]) read back from
 * their codes and scales.
 */
void orc_indexer_scores_e4m3(int n_heads, int dim, const uint8_t *q8, const float *qscale, const float *w,
                             const uint8_t *k8, const float *kscale, long n_vis, double *out)
{
    for (long j = 0; j < n_vis; ++j) {
        double s = 0.0;
        for (int h = 0; h < n_heads; ++h) {
            double dot = 0.0;
            for (int d = 0; d < dim; ++d)
                dot += e4m3_value(q8, qscale, h, dim, d) * e4m3_value(k8, kscale, j, dim, d);
            double relu = dot > 0.0 ? dot : 0.0;
            s += (double)w[h] * relu;
        }
        out[j] = s;
    }
}

/* Rows r of a per-row-scaled e4m3 array read back as doubles (out[r][i]). */
void orc_dequantize_rows_e4m3(long rows, int width, const uint8_t *q, const float *scale, double *out)
{
    for (long r = 0; r < rows; ++r)
        for (int i = 0; i < width; ++i)
            out[(size_t)r * (size_t)width + (size_t)i] = e4m3_value(q, scale, r, width, i);
}
