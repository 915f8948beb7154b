/*
 * ssa_oracle.c -- fp64 CPU oracle for the spatial self-attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (tensortonic "diffusion-l03-spatial-self-attention",
 * problem statement and its block equation):
 *
 *     Z   = tokens(GN(x))                       x: (B, C, H, W)
 *     Q   = Z Wq^T + bq,  K = Z Wk^T + bk,  V = Z Wv^T + bv
 *     O_j = softmax(Q_j K_j^T / sqrt(d)) V_j    head j = channels [j d, (j+1) d)
 *     out = x + image([O_1 .. O_n] Wo^T + bo)
 *
 *   * GN is a group norm with G contiguous channel groups, statistics per
 *     sample over the (C/G) * H * W values of a group, the biased (population)
 *     variance, eps = 1e-5 inside the square root, then the per-channel affine
 *     norm_weight / norm_bias (problem statement, GN sentence).
 *   * tokens(): pixel (i, j) of sample b becomes row i*W + j of a (HW, C)
 *     matrix; image() is its inverse (problem statement, tokens sentence and
 *     the flatten(2).transpose(1, 2) hint).
 *   * "used as in a linear layer": y = z W^T + b with W stored (out, in).
 *   * d = C / num_heads; the softmax runs over keys and is scaled by 1/sqrt(d)
 *     (the worked example 1 explanation divides by sqrt(2) for d = 2).
 *   * The result takes the dtype of x (problem statement, return sentence):
 *     ssa_oracle_round() rounds the exact fp64 value once, to nearest-even.
 *
 * Every input is taken as fp64 (the caller up-converts stored values, which is
 * exact for fp32 and bf16).  All arithmetic is fp64 with plain loops in the
 * order the definition gives; GN statistics use two passes (mean, then the
 * sum of squared deviations).  Parallelism is OpenMP over independent
 * (sample, row) work items only; no loop is blocked, fused or reordered.
 *
 * Query-sampled mode: when qidx != NULL only the nq listed pixels of every
 * sample get Q, O and the branch output; Z, K and V are still formed for all
 * H*W pixels, because every query attends to every key.
 *
 * Variants (HNDL "attention" operator page, parameter table and its Biases,
 * Masking, Relative position bias and Rotary embeddings paragraphs), applied
 * to the block's token sequence (T = H*W tokens in row-major pixel order):
 *   * bias flags: a NULL bq / bk / bv / bo means that projection has no bias;
 *   * causal: key m is masked (score -inf) for query position t when m > t;
 *   * rope: Q and K rows are rotated by their token position t per head with
 *     the rotate-half convention over the full head dim, base 10000:
 *     theta_i = 10000^(-2i/d), angle = t * theta_i (i < d/2),
 *     x' = x * cos(angle) + rotate_half(x) * sin(angle), rotate_half([a, b])
 *     = [-b, a]; the rotation is evaluated exactly in fp64 here;
 *   * relative position bias: a table [(2H-1)(2W-1)][heads]; for query token
 *     (rq, cq) and key token (rk, ck) of the row-major grid, head j adds
 *     table[((rq - rk + H - 1) * (2W - 1) + (cq - ck + W - 1)) * heads + j]
 *     to the scaled logit before the softmax.
 *   * query-key RMS normalisation (vit-pytorch simple_vit_with_qk_norm.py,
 *     RMSNorm class): each head's Q and K rows become
 *     x / max(||x||_2, 1e-12) * sqrt(d) * gamma[head][:], gamma [h][d] per
 *     projection; applied before the rotation when both are on.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GN_EPS 1e-5

/* ---- GroupNorm statistics: two-pass mean and biased variance --------------
 * x: [B][C][N] (N = H*W), mean/rstd: [B][G].  Returns 0, or -1 when C % G. */
int ssa_oracle_gn_stats(const double *x, int B, int C, int N, int G,
                        double *mean, double *rstd)
{
    if (B <= 0 || C <= 0 || N <= 0 || G <= 0 || C % G) return -1;
    const int cg = C / G;
    const long long cnt = (long long)cg * N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < G; ++g) {
            const double *xg = x + ((long long)b * C + (long long)g * cg) * N;
            double s = 0.0;
            for (long long i = 0; i < cnt; ++i) s += xg[i];
            const double mu = s / (double)cnt;
            double ss = 0.0;
            for (long long i = 0; i < cnt; ++i) {
                const double dlt = xg[i] - mu;
                ss += dlt * dlt;
            }
            const double var = ss / (double)cnt; /* biased (population) */
            mean[b * G + g] = mu;
            rstd[b * G + g] = 1.0 / sqrt(var + GN_EPS);
        }
    return 0;
}

/* ---- Step 3: attention from given Q, K, V --------------------------------
 * q [B][nq][C] (the query rows), k, v [B][N][C], o [B][nq][C],
 * p (optional) [B][h][nq][N].  Per head j: scores over all keys scaled by
 * 1/sqrt(d), a softmax over the key axis (the maximum is subtracted only to
 * keep exp() in range), then P V; head outputs side by side in head order. */
static void attention_core(const double *q, const double *k, const double *v, int B, int N, int nq, int C,
                           int nh, const int *qpos, int causal, const double *rel, int H, int W,
                           double *o, double *p_out)
{
    const int d = C / nh;
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * N);
#pragma omp for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < nq; ++t) {
                const double *qr = q + ((long long)b * nq + t) * C;
                double *orow = o + ((long long)b * nq + t) * C;
                const int tq = qpos ? qpos[t] : t; /* token position of this query */
                for (int j = 0; j < nh; ++j) {
                    const int c0 = j * d;
                    double smax = -INFINITY;
                    for (int m = 0; m < N; ++m) {
                        const double *kr = k + ((long long)b * N + m) * C;
                        double acc = 0.0;
                        for (int e = 0; e < d; ++e) acc += qr[c0 + e] * kr[c0 + e];
                        s[m] = acc * scale;
                        if (rel) {
                            const int dy = tq / W - m / W + (H - 1);
                            const int dx = tq % W - m % W + (W - 1);
                            s[m] += rel[((long long)dy * (2 * W - 1) + dx) * nh + j];
                        }
                        if (causal && m > tq) s[m] = -INFINITY;
                        if (s[m] > smax) smax = s[m];
                    }
                    double den = 0.0;
                    for (int m = 0; m < N; ++m) {
                        s[m] = exp(s[m] - smax);
                        den += s[m];
                    }
                    for (int m = 0; m < N; ++m) s[m] /= den;
                    if (p_out) {
                        double *pr = p_out + (((long long)b * nh + j) * nq + t) * N;
                        for (int m = 0; m < N; ++m) pr[m] = s[m];
                    }
                    for (int e = 0; e < d; ++e) {
                        double acc = 0.0;
                        for (int m = 0; m < N; ++m)
                            acc += s[m] * v[((long long)b * N + m) * C + c0 + e];
                        orow[c0 + e] = acc;
                    }
                }
            }
        free(s);
    }
}

void ssa_oracle_attention(const double *q, const double *k, const double *v, int B, int N, int nq, int C,
                          int nh, double *o, double *p_out)
{
    attention_core(q, k, v, B, N, nq, C, nh, NULL, 0, NULL, 1, 1, o, p_out);
}

/* Attention with the variants: qpos [nq] token position of each query row
 * (NULL: row t is position t), causal mask, relative-position table (NULL:
 * none) over an H x W grid with H * W == N. */
void ssa_oracle_attention_ex(const double *q, const double *k, const double *v, int B, int N, int nq, int C,
                             int nh, const int *qpos, int causal, const double *rel, int H, int W,
                             double *o, double *p_out)
{
    attention_core(q, k, v, B, N, nq, C, nh, qpos, causal, rel, H, W, o, p_out);
}

/* ---- Rotary embedding of one (rows x C) matrix, in place ------------------
 * Row r sits at token position pos[r] (or r when pos is NULL); each head's
 * d features are rotated pairwise (i, i + d/2) by angle pos * 10000^(-2i/d). */
void ssa_oracle_rope(double *m, int rows, int C, int nh, const int *pos)
{
    const int d = C / nh, hd = d / 2;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const double t = (double)(pos ? pos[r] : r);
        double *row = m + (long long)r * C;
        for (int j = 0; j < nh; ++j)
            for (int i = 0; i < hd; ++i) {
                const double theta = pow(10000.0, -2.0 * (double)i / (double)d);
                const double a = row[j * d + i], bb = row[j * d + hd + i];
                const double cs = cos(t * theta), sn = sin(t * theta);
                row[j * d + i] = a * cs - bb * sn;       /* a cos + (-b) sin */
                row[j * d + hd + i] = bb * cs + a * sn;  /* b cos + a sin */
            }
    }
}

/* ---- Query-key RMS normalisation of one (rows x C) matrix, in place ------
 * Per row and head j: x_j / max(||x_j||_2, 1e-12) * sqrt(d) * gamma[j][:]. */
void ssa_oracle_qk_norm(double *m, int rows, int C, int nh, const double *gamma)
{
    const int d = C / nh;
    const double sd = sqrt((double)d);
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double *row = m + (long long)r * C;
        for (int j = 0; j < nh; ++j) {
            double ss = 0.0;
            for (int e = 0; e < d; ++e) ss += row[j * d + e] * row[j * d + e];
            double nrm = sqrt(ss);
            if (nrm < 1e-12) nrm = 1e-12;
            for (int e = 0; e < d; ++e) row[j * d + e] = row[j * d + e] / nrm * sd * gamma[j * d + e];
        }
    }
}

/* ---- Step 4: output projection and image() --------------------------------
 * o [B][nq][C] -> y [B][C][nq] = (o Wo^T + bo) with the pixel axis last. */
void ssa_oracle_out_proj(const double *o, const double *wo, const double *bo, int B, int nq, int C, double *y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < nq; ++t) {
            const double *orow = o + ((long long)b * nq + t) * C;
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int e = 0; e < C; ++e) acc += orow[e] * wo[(long long)c * C + e];
                y[((long long)b * C + c) * nq + t] = acc + (bo ? bo[c] : 0.0);
            }
        }
}

/* ---- The whole block ------------------------------------------------------
 * Inputs (all fp64, contiguous):
 *   x [B][C][H*W]; gw, gb, bq, bk, bv, bo [C]; wq, wk, wv, wo [C][C] (out, in).
 *   qidx: NULL for every pixel, else nq pixel indices in [0, H*W) shared by
 *   every sample and every head.
 * Outputs (each may be NULL unless stated):
 *   y    [B][C][nq]  REQUIRED: the branch image([O] Wo^T + bo) at the chosen
 *                    pixels (out = x + y before rounding).
 *   mean, rstd [B][G]
 *   z    [B][N][C]   tokens(GN(x))
 *   q    [B][nq][C]  k, v [B][N][C]
 *   o    [B][nq][C]  concatenated head outputs
 *   p    [B][h][nq][N] softmax probabilities (only for small problems)
 * ssa_oracle_forward_ex also takes causal, rope (both 0/1), rel (NULL or
 * the table [(2H-1)(2W-1)][h]) and q_gamma / k_gamma (both NULL, or the
 * query-key RMS-norm weights [h][d]); any bias pointer may be NULL (no bias);
 * q and k are returned after the normalisation and rotation.
 * Returns 0; -1 on a bad shape (C % G, C % h, non-positive sizes, an odd head
 * dim with rope). */
int ssa_oracle_forward_ex(const double *x, int B, int C, int H, int W, int G, int nh,
                          const double *gw, const double *gb,
                          const double *wq, const double *bq,
                          const double *wk, const double *bk,
                          const double *wv, const double *bv,
                          const double *wo, const double *bo,
                          int causal, int rope, const double *rel,
                          const double *q_gamma, const double *k_gamma,
                          const int *qidx, int nq,
                          double *y, double *mean_out, double *rstd_out,
                          double *z_out, double *q_out, double *k_out,
                          double *v_out, double *o_out, double *p_out)
{
    if (B <= 0 || C <= 0 || H <= 0 || W <= 0 || G <= 0 || nh <= 0) return -1;
    if (C % G || C % nh) return -1;
    if (rope && (C / nh) % 2) return -1; /* rotate-half needs an even head dim */
    const int N = H * W;
    if (!qidx) nq = N;
    if (nq <= 0) return -1;
    const int cg = C / G;

    double *mean = (double *)malloc(sizeof(double) * B * G);
    double *rstd = (double *)malloc(sizeof(double) * B * G);
    double *z = (double *)malloc(sizeof(double) * (size_t)B * N * C);
    double *k = (double *)malloc(sizeof(double) * (size_t)B * N * C);
    double *v = (double *)malloc(sizeof(double) * (size_t)B * N * C);
    double *q = (double *)malloc(sizeof(double) * (size_t)B * nq * C);
    double *o = (double *)malloc(sizeof(double) * (size_t)B * nq * C);
    if (!mean || !rstd || !z || !k || !v || !q || !o) {
        free(mean); free(rstd); free(z); free(k); free(v); free(q); free(o);
        return -2;
    }

    /* 1. GroupNorm statistics, then Z = tokens(GN(x)): z[b][iW+j][c]. */
    ssa_oracle_gn_stats(x, B, C, N, G, mean, rstd);
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int n = 0; n < N; ++n)
            for (int c = 0; c < C; ++c) {
                const int g = c / cg;
                const double xh = (x[((long long)b * C + c) * N + n] - mean[b * G + g]) * rstd[b * G + g];
                z[((long long)b * N + n) * C + c] = xh * gw[c] + gb[c];
            }

    /* 2. Projections "as in a linear layer": K, V for every pixel, Q for the
     *    chosen pixels. */
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int n = 0; n < N; ++n) {
            const double *zr = z + ((long long)b * N + n) * C;
            double *kr = k + ((long long)b * N + n) * C;
            double *vr = v + ((long long)b * N + n) * C;
            for (int f = 0; f < C; ++f) {
                double sk = 0.0, sv = 0.0;
                for (int c = 0; c < C; ++c) {
                    sk += zr[c] * wk[(long long)f * C + c];
                    sv += zr[c] * wv[(long long)f * C + c];
                }
                kr[f] = sk + (bk ? bk[f] : 0.0);
                vr[f] = sv + (bv ? bv[f] : 0.0);
            }
        }
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < nq; ++t) {
            const int n = qidx ? qidx[t] : t;
            const double *zr = z + ((long long)b * N + n) * C;
            double *qr = q + ((long long)b * nq + t) * C;
            for (int f = 0; f < C; ++f) {
                double s = 0.0;
                for (int c = 0; c < C; ++c) s += zr[c] * wq[(long long)f * C + c];
                qr[f] = s + (bq ? bq[f] : 0.0);
            }
        }

    /* 2b. Query-key RMS normalisation, then the rotary embedding of Q and K
     *     by token position. */
    if (q_gamma && k_gamma)
        for (int b = 0; b < B; ++b) {
            ssa_oracle_qk_norm(q + (long long)b * nq * C, nq, C, nh, q_gamma);
            ssa_oracle_qk_norm(k + (long long)b * N * C, N, C, nh, k_gamma);
        }
    if (rope)
        for (int b = 0; b < B; ++b) {
            ssa_oracle_rope(q + (long long)b * nq * C, nq, C, nh, qidx);
            ssa_oracle_rope(k + (long long)b * N * C, N, C, nh, NULL);
        }

    /* 3. Attention per head, then 4. the output projection and image(). */
    attention_core(q, k, v, B, N, nq, C, nh, qidx, causal, rel, H, W, o, p_out);
    ssa_oracle_out_proj(o, wo, bo, B, nq, C, y);

    if (mean_out) memcpy(mean_out, mean, sizeof(double) * B * G);
    if (rstd_out) memcpy(rstd_out, rstd, sizeof(double) * B * G);
    if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)B * N * C);
    if (q_out) memcpy(q_out, q, sizeof(double) * (size_t)B * nq * C);
    if (k_out) memcpy(k_out, k, sizeof(double) * (size_t)B * N * C);
    if (v_out) memcpy(v_out, v, sizeof(double) * (size_t)B * N * C);
    if (o_out) memcpy(o_out, o, sizeof(double) * (size_t)B * nq * C);
    free(mean); free(rstd); free(z); free(k); free(v); free(q); free(o);
    return 0;
}

int ssa_oracle_forward(const double *x, int B, int C, int H, int W, int G, int nh,
                       const double *gw, const double *gb,
                       const double *wq, const double *bq,
                       const double *wk, const double *bk,
                       const double *wv, const double *bv,
                       const double *wo, const double *bo,
                       const int *qidx, int nq,
                       double *y, double *mean_out, double *rstd_out,
                       double *z_out, double *q_out, double *k_out,
                       double *v_out, double *o_out, double *p_out)
{
    return ssa_oracle_forward_ex(x, B, C, H, W, G, nh, gw, gb, wq, bq, wk, bk, wv, bv, wo, bo, 0, 0, NULL, NULL,
                                 NULL, qidx, nq, y, mean_out, rstd_out, z_out, q_out, k_out, v_out, o_out, p_out);
}

/* ---- Rounding to the dtype of x -------------------------------------------
 * The block returns x's dtype.  The exact fp64 value is rounded once,
 * to nearest with ties to even.
 *   dtype 0: fp32 -> out is float[n]
 *   dtype 1: bf16 -> out is uint16_t[n] (the bf16 bit pattern)
 * bf16 rounding is done directly from fp64 (no intermediate fp32 rounding):
 * the value is snapped to the bf16 grid spacing of its binade (8 significant
 * bits), nearbyint() in the default round-to-nearest-even mode breaking ties. */
static uint16_t round_bf16(double v)
{
    union { float f; uint32_t u; } cv;
    if (isnan(v)) return 0x7fc0;
    if (v == 0.0) { cv.f = (float)v; return (uint16_t)(cv.u >> 16); }
    int e;
    (void)frexp(fabs(v), &e);           /* |v| in [2^(e-1), 2^e) */
    int e_min = -125;                   /* normal bf16 binade floor: 2^-126 = 2^(e-1) with e = -125 */
    if (e < e_min) e = e_min;           /* subnormal range keeps a fixed spacing */
    const double ulp = ldexp(1.0, e - 8); /* 8 significant bits per binade */
    double r = nearbyint(v / ulp) * ulp;
    if (fabs(r) >= ldexp(1.0, 128)) {   /* beyond the largest finite bf16 */
        cv.f = (v > 0) ? INFINITY : -INFINITY;
        return (uint16_t)(cv.u >> 16);
    }
    cv.f = (float)r;                    /* exact: r has <= 8 significant bits */
    return (uint16_t)(cv.u >> 16);
}

void ssa_oracle_round(const double *v, long long n, int dtype, void *out)
{
    if (dtype == 0) {
        float *o = (float *)out;
        for (long long i = 0; i < n; ++i) o[i] = (float)v[i]; /* IEEE RNE */
    } else {
        uint16_t *o = (uint16_t *)out;
        for (long long i = 0; i < n; ++i) o[i] = round_bf16(v[i]);
    }
}

#ifdef _OPENMP
extern int omp_get_max_threads(void);
extern void omp_set_num_threads(int);
#endif

int ssa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ssa_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
