/*
 * Float64 CPU oracle for latent causal attention and the latent projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Everything is plain double-precision loops, written from the definitions on
 * two pages:
 *   [ATTN] page "FW-GLM-5-1 l2_p31" (fused MLA-style attention from
 *          compressed KV latents), its "The algorithm" passage: for every
 *          batch b, head h and query t, and every s from 0 to t inclusive,
 *          k = latent[b,s] @ w_up_k[:,h], v = latent[b,s] @ w_up_v[:,h],
 *          logit = (q[b,t,h] * k).sum() * scale; softmax over the logits;
 *          weighted sum of the values.  Shapes: q (B,T,H,d), kv_latent
 *          (B,T,rank), w_up_k / w_up_v (rank,H,d).
 *   [PROJ] page "FW-GLM-5-1 l2_p1" (fused latent projection), its problem
 *          statement: latent = hidden @ w_down, k = latent @ w_up_k,
 *          v = latent @ w_up_v with w_up_* of shape (rank, kv_dim).
 *   [MSA]  page "Kimi-K2.6 l2_p29" (MSA row-wise gated attention), its
 *          online-softmax derivation (running max m, running sum d, running
 *          weighted sum o, rescaled by exp(m - m_new)) and its treatment of
 *          -inf scores (initialise from the first element; the worked
 *          example [-inf, 0, 0] gives (v1 + v2) / 2).
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *   - the mask is inclusive (s <= t), as [ATTN] states;
 *   - when there are fewer queries than keys (Tq < Tkv) the queries are the
 *     LAST Tq positions: query i sits at t = Tkv - Tq + i;
 *   - causal = 0 lets every query see all Tkv keys;
 *   - the softmax is the max-subtracted two-pass form [ATTN] describes
 *     (max of the logits, then exp(x - max), then divide by the sum);
 *   - exp is the C library's double exp.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC mla_oracle.c -o libmla_oracle.so -lm
 * (no -ffast-math: the oracle keeps IEEE double semantics).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ORACLE_MUTANT (0 in every real build) plants one known mistake so that a
 * CPU test can show the pins catch it:
 *   1 exclusive mask (s < t)        2 neighbouring head's weights
 *   3 scale dropped                 4 w_up_k used for the values
 *   5 query taken at t instead of i 6 w_down read transposed
 *   7 softmax not normalised */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ----------------------------------------------------------------------- */
/* [PROJ] latent = hidden @ w_down; k = latent @ w_up_k; v = latent @ w_up_v. */
/* hidden (M, Dm), w_down (Dm, R), w_up_k / w_up_v (R, C), all row-major.     */
/* k and v may be NULL (then w_up_k / w_up_v are not read).                   */
/* ----------------------------------------------------------------------- */
void mla_oracle_project(const double *hidden, const double *w_down,
                        const double *w_up_k, const double *w_up_v,
                        double *latent, double *k, double *v,
                        int64_t M, int Dm, int R, int C)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int j = 0; j < Dm; ++j)
#if ORACLE_MUTANT == 6
                acc += hidden[m * Dm + j] * w_down[((int64_t)r * Dm + j) % ((int64_t)Dm * R)];
#else
                acc += hidden[m * Dm + j] * w_down[(int64_t)j * R + r];
#endif
            latent[m * R + r] = acc;
        }
        for (int c = 0; c < C && (k || v); ++c) {
            double ak = 0.0, av = 0.0;
            for (int r = 0; r < R; ++r) {
                const double l = latent[m * R + r];
                if (k) ak += l * w_up_k[(int64_t)r * C + c];
                if (v) av += l * w_up_v[(int64_t)r * C + c];
            }
            if (k) k[m * C + c] = ak;
            if (v) v[m * C + c] = av;
        }
    }
}

/* ----------------------------------------------------------------------- */
/* [ATTN] literal form.  One (b, h, i) row; k_s and v_s are rebuilt from the */
/* latent for every key s they are used with.                               */
/* ----------------------------------------------------------------------- */
static int last_key(int i, int Tq, int Tkv, int causal)
{
#if ORACLE_MUTANT == 1
    if (causal) { int t = Tkv - Tq + i; return t > 0 ? t - 1 : 0; }
#endif
    return causal ? (Tkv - Tq + i) : (Tkv - 1);
}

/* k_s[e] = sum_r latent[b,s,r] * w[r,h,e]  (w is w_up_k or w_up_v) */
static void rebuild(const double *lat_bs, const double *w, int h, int H, int d, int R,
                    double *vec)
{
#if ORACLE_MUTANT == 2
    h = (h + 1) % H;
#endif
    for (int e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int r = 0; r < R; ++r)
            acc += lat_bs[r] * w[((int64_t)r * H + h) * d + e];
        vec[e] = acc;
    }
}

/* Logits of one row, x_s = scale * sum_e q[b,i,h,e] * k_s[e], for s = 0..S-1. */
static void row_logits(const double *q, const double *lat, const double *wk,
                       int b, int h, int i, int Tq, int Tkv, int H, int d, int R,
                       double scale, int S, double *x, double *kbuf)
{
#if ORACLE_MUTANT == 5
    const int iq = (Tkv - Tq + i) < Tq ? (Tkv - Tq + i) : Tq - 1;
    const double *qv = q + (((int64_t)b * Tq + iq) * H + h) * d;
#else
    const double *qv = q + (((int64_t)b * Tq + i) * H + h) * d;
#endif
#if ORACLE_MUTANT == 3
    scale = 1.0;
#endif
    for (int s = 0; s < S; ++s) {
        rebuild(lat + ((int64_t)b * Tkv + s) * R, wk, h, H, d, R, kbuf);
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += qv[e] * kbuf[e];
        x[s] = dot * scale;
    }
}

static void attend_row(const double *q, const double *lat, const double *wk, const double *wv,
                       int b, int h, int i, int Tq, int Tkv, int H, int d, int R,
                       double scale, int causal, double *out_row)
{
    const int S = last_key(i, Tq, Tkv, causal) + 1;
    double *x = (double *)malloc(sizeof(double) * (size_t)S);
    double *buf = (double *)malloc(sizeof(double) * (size_t)d);
    row_logits(q, lat, wk, b, h, i, Tq, Tkv, H, d, R, scale, S, x, buf);
    /* max-subtracted softmax: m = max x, w_s = exp(x_s - m), Z = sum w_s */
    double m = x[0];
    for (int s = 1; s < S; ++s) if (x[s] > m) m = x[s];
    double Z = 0.0;
    for (int s = 0; s < S; ++s) { x[s] = exp(x[s] - m); Z += x[s]; }
    for (int e = 0; e < d; ++e) out_row[e] = 0.0;
    for (int s = 0; s < S; ++s) {
#if ORACLE_MUTANT == 4
        rebuild(lat + ((int64_t)b * Tkv + s) * R, wk, h, H, d, R, buf);
#else
        rebuild(lat + ((int64_t)b * Tkv + s) * R, wv, h, H, d, R, buf);
#endif
#if ORACLE_MUTANT == 7
        const double p = x[s];
#else
        const double p = x[s] / Z;
#endif
        for (int e = 0; e < d; ++e) out_row[e] += p * buf[e];
    }
    free(buf);
    free(x);
}

/* out (B,Tq,H,d) for q (B,Tq,H,d), kv_latent (B,Tkv,R), w_up_k / w_up_v (R,H,d). */
void mla_oracle_attention(const double *q, const double *lat, const double *wk, const double *wv,
                          double *out, int B, int Tq, int Tkv, int H, int d, int R,
                          double scale, int causal)
{
    const int64_t rows = (int64_t)B * Tq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = rows - 1; n >= 0; --n) {          /* longest rows first */
        const int h = (int)(n % H);
        const int i = (int)((n / H) % Tq);
        const int b = (int)(n / ((int64_t)H * Tq));
        attend_row(q, lat, wk, wv, b, h, i, Tq, Tkv, H, d, R, scale, causal,
                   out + n * d);
    }
}

/* Selected rows only: bi holds n pairs (b, i); out_rows (n, H, d). */
void mla_oracle_attention_rows(const double *q, const double *lat, const double *wk,
                               const double *wv, const int32_t *bi, int n, double *out_rows,
                               int B, int Tq, int Tkv, int H, int d, int R,
                               double scale, int causal)
{
    (void)B;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int j = 0; j < n; ++j)
        for (int h = 0; h < H; ++h)
            attend_row(q, lat, wk, wv, bi[2 * j], h, bi[2 * j + 1], Tq, Tkv, H, d, R, scale,
                       causal, out_rows + ((int64_t)j * H + h) * d);
}

/* Normalised softmax weights of one row (length last_key + 1); returns it. */
int mla_oracle_attention_weights(const double *q, const double *lat, const double *wk,
                                 int b, int h, int i, int B, int Tq, int Tkv, int H, int d,
                                 int R, double scale, int causal, double *w)
{
    (void)B;
    const int S = last_key(i, Tq, Tkv, causal) + 1;
    double *buf = (double *)malloc(sizeof(double) * (size_t)d);
    row_logits(q, lat, wk, b, h, i, Tq, Tkv, H, d, R, scale, S, w, buf);
    double m = w[0];
    for (int s = 1; s < S; ++s) if (w[s] > m) m = w[s];
    double Z = 0.0;
    for (int s = 0; s < S; ++s) { w[s] = exp(w[s] - m); Z += w[s]; }
    for (int s = 0; s < S; ++s) w[s] /= Z;
    free(buf);
    return S;
}

/* ----------------------------------------------------------------------- */
/* Absorbed form (the identity (latent_s W_k) . q = latent_s . (W_k q)):     */
/*   q'_r = sum_e w_up_k[r,h,e] q[e];  x_s = scale * q' . latent_s;           */
/*   o_r = sum_s p_s latent_s[r];      out_e = sum_r o_r w_up_v[r,h,e].       */
/* Used only to check that the identity the GPU path relies on holds.         */
/* ----------------------------------------------------------------------- */
static void absorbed_row(const double *q, const double *lat, const double *wk,
                         const double *wv, int b, int h, int i, int Tq, int Tkv, int H, int d,
                         int R, double scale, int causal, double *out_row)
{
    const int S = last_key(i, Tq, Tkv, causal) + 1;
    const double *qv = q + (((int64_t)b * Tq + i) * H + h) * d;
    double *qa = (double *)malloc(sizeof(double) * (size_t)R);
    double *o = (double *)calloc((size_t)R, sizeof(double));
    double *x = (double *)malloc(sizeof(double) * (size_t)S);
    for (int r = 0; r < R; ++r) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += wk[((int64_t)r * H + h) * d + e] * qv[e];
        qa[r] = acc;
    }
    double m = -INFINITY;
    for (int s = 0; s < S; ++s) {
        const double *ls = lat + ((int64_t)b * Tkv + s) * R;
        double acc = 0.0;
        for (int r = 0; r < R; ++r) acc += qa[r] * ls[r];
        x[s] = acc * scale;
        if (x[s] > m) m = x[s];
    }
    double Z = 0.0;
    for (int s = 0; s < S; ++s) { x[s] = exp(x[s] - m); Z += x[s]; }
    for (int s = 0; s < S; ++s) {
        const double *ls = lat + ((int64_t)b * Tkv + s) * R;
        const double p = x[s] / Z;
        for (int r = 0; r < R; ++r) o[r] += p * ls[r];
    }
    for (int e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int r = 0; r < R; ++r) acc += o[r] * wv[((int64_t)r * H + h) * d + e];
        out_row[e] = acc;
    }
    free(x); free(o); free(qa);
}

void mla_oracle_attention_absorbed(const double *q, const double *lat, const double *wk,
                                   const double *wv, double *out, int B, int Tq, int Tkv,
                                   int H, int d, int R, double scale, int causal)
{
    const int64_t rows = (int64_t)B * Tq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < rows; ++n) {
        const int h = (int)(n % H);
        const int i = (int)((n / H) % Tq);
        const int b = (int)(n / ((int64_t)H * Tq));
        absorbed_row(q, lat, wk, wv, b, h, i, Tq, Tkv, H, d, R, scale, causal, out + n * d);
    }
}

/* Absorbed form for selected (b, i) rows; same layout as the literal rows call. */
void mla_oracle_attention_absorbed_rows(const double *q, const double *lat, const double *wk,
                                        const double *wv, const int32_t *bi, int n,
                                        double *out_rows, int B, int Tq, int Tkv, int H, int d,
                                        int R, double scale, int causal)
{
    (void)B;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int j = 0; j < n; ++j)
        for (int h = 0; h < H; ++h)
            absorbed_row(q, lat, wk, wv, bi[2 * j], h, bi[2 * j + 1], Tq, Tkv, H, d, R, scale,
                         causal, out_rows + ((int64_t)j * H + h) * d);
}

/* ----------------------------------------------------------------------- */
/* [MSA] online softmax with a weighted sum, initialised from the first     */
/* element: m = x_0, den = 1, o = v_0; then for each later j                 */
/*   m_new = max(m, x_j); den = den*exp(m - m_new) + exp(x_j - m_new);       */
/*   o = o*exp(m - m_new) + v_j*exp(x_j - m_new);  out = o / den.            */
/* x (n), v (n, dv) row-major, out (dv).                                     */
/* ----------------------------------------------------------------------- */
void mla_oracle_online_softmax(const double *x, const double *v, int n, int dv, double *out)
{
    double m = x[0], den = 1.0;
    for (int e = 0; e < dv; ++e) out[e] = v[e];
    for (int j = 1; j < n; ++j) {
        const double m_new = x[j] > m ? x[j] : m;
        const double a = exp(m - m_new), c = exp(x[j] - m_new);
        den = den * a + c;
        for (int e = 0; e < dv; ++e) out[e] = out[e] * a + v[(int64_t)j * dv + e] * c;
        m = m_new;
    }
    for (int e = 0; e < dv; ++e) out[e] /= den;
}

/* Merge of partial online-softmax states, the same recurrence applied to   */
/* whole partitions: part i carries its max m_i, its sum l_i (relative to   */
/* m_i) and its unnormalised weighted sum o_i (dv).  An empty or fully      */
/* masked part has m_i = -inf and contributes nothing.  out = o / l.        */
void mla_oracle_merge_partials(const double *m_i, const double *l_i, const double *o_i,
                               int parts, int dv, double *out)
{
    double m = -INFINITY;
    for (int i = 0; i < parts; ++i) if (m_i[i] > m) m = m_i[i];
    double l = 0.0;
    for (int e = 0; e < dv; ++e) out[e] = 0.0;
    for (int i = 0; i < parts; ++i) {
        if (m_i[i] == -INFINITY) continue;              /* exp(-inf - m) = 0 */
        const double a = exp(m_i[i] - m);
        l += a * l_i[i];
        for (int e = 0; e < dv; ++e) out[e] += a * o_i[(int64_t)i * dv + e];
    }
    for (int e = 0; e < dv; ++e) out[e] /= l;
}
