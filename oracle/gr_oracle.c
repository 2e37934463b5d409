/*
 * Gated Residual (GR) oracle: the plain definition, in fp64, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or load this file;
 * only the tests, the smoke check and the bench's CPU-baseline leg use it. It shares no code
 * with the CUDA library.
 *
 * Sources (page, section, equation):
 *   "【论文解读】 Qwen3.8 Flash Next" (wkq9411.github.io), §二.4 Gated Residual:
 *     eq rms      R̂_i = RMSNorm(R_i; γ_i)
 *     eq gate     G = unvec σ(W_u SiLU((1/n_r) W_d vec R̂)),  W_d: r×n_r·d,  W_u: n_r·d×r
 *     eq use_gate x = (1/n_r) Σ_i G_i ⊙ R̂_i
 *     eq s        s = 2σ((1/n_r) W_w vec R̂),  W_w: n_r×n_r·d
 *     eq write    R'_i = R_i + s_i y
 *   "Qwen3.8-Flash-Next 架构笔记 · 06 / RESIDUAL" (cbphcr.github.io), §2 and §3 (same
 *   formulas at n_r = 4).
 * Where the pages leave a point open this file reads it as follows: eps inside the square
 * root (1/sqrt(mean + eps)), a multiplicative gain γ, vec stacking the branches branch-major
 * (index i·D + c); eps is a parameter here.
 *
 * Layouts, all row-major:
 *   R, R_out  [n][nb][D]      token, branch, channel
 *   y, x      [n][D]
 *   s         [n][nb]
 *   gamma     [nb][D]
 *   Wd        [r][nb*D]       vec index j = i*D + c (branches stacked)
 *   Wu        [nb*D][r]
 *   Ww        [nb][nb*D]
 *   G (opt.)  [n][nb][D]      the read gates, for tests of eq auv
 *   inv (opt.)[n][nb]         1/sqrt(mean(R_i^2) + eps)
 *
 * Every function loops over tokens independently (OpenMP over tokens when available).
 * Return value: 0, or -1 on a bad argument, or -2 when scratch memory could not be had.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Logistic function 1/(1+e^{-a}), written so that neither branch overflows. */
static double sigmoid(double a)
{
    if (a >= 0.0)
        return 1.0 / (1.0 + exp(-a));
    double e = exp(a);
    return e / (1.0 + e);
}

/* SiLU(a) = a·σ(a) (the activation inside eq gate). */
static double silu(double a) { return a * sigmoid(a); }

/* Group RMSNorm of one token, eq rms: per branch i, inv_i = 1/sqrt(mean_c R_i[c]^2 + eps),
 * Rh[i*D+c] = R_i[c] · inv_i · gamma_i[c]. */
static void group_rmsnorm(int nb, int D, double eps, const double *R, const double *gamma,
                          double *Rh, double *inv)
{
    for (int i = 0; i < nb; ++i) {
        const double *Ri = R + (size_t)i * D;
        double ss = 0.0;
        for (int c = 0; c < D; ++c)
            ss += Ri[c] * Ri[c];
        double ms = ss / (double)D;
        inv[i] = 1.0 / sqrt(ms + eps);
        for (int c = 0; c < D; ++c)
            Rh[(size_t)i * D + c] = Ri[c] * inv[i] * gamma[(size_t)i * D + c];
    }
}

/* The read of one token given its normalised state Rh (= vec R̂, length nb*D):
 * eq gate, eq use_gate and eq s. h (length r) and g (length nb*D) are scratch. */
static void read_from_normalised(int nb, int D, int r, const double *Rh, const double *Wd,
                                 const double *Wu, const double *Ww, double *h, double *g,
                                 double *x, double *s, double *G_out)
{
    const size_t K = (size_t)nb * D;
    const double inv_nb = 1.0 / (double)nb;

    /* z = (1/n_r) W_d vec R̂ ; h = SiLU(z) */
    for (int k = 0; k < r; ++k) {
        const double *w = Wd + (size_t)k * K;
        double acc = 0.0;
        for (size_t j = 0; j < K; ++j)
            acc += w[j] * Rh[j];
        h[k] = silu(inv_nb * acc);
    }
    /* G = unvec σ(W_u h) */
    for (size_t j = 0; j < K; ++j) {
        const double *w = Wu + j * (size_t)r;
        double acc = 0.0;
        for (int k = 0; k < r; ++k)
            acc += w[k] * h[k];
        g[j] = sigmoid(acc);
    }
    /* x = (1/n_r) Σ_i G_i ⊙ R̂_i */
    for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int i = 0; i < nb; ++i)
            acc += g[(size_t)i * D + c] * Rh[(size_t)i * D + c];
        x[c] = inv_nb * acc;
    }
    /* s = 2σ((1/n_r) W_w vec R̂) */
    for (int i = 0; i < nb; ++i) {
        const double *w = Ww + (size_t)i * K;
        double acc = 0.0;
        for (size_t j = 0; j < K; ++j)
            acc += w[j] * Rh[j];
        s[i] = 2.0 * sigmoid(inv_nb * acc);
    }
    if (G_out)
        memcpy(G_out, g, K * sizeof(double));
}

static int bad_dims(int64_t n, int nb, int D, int r)
{
    return n < 0 || nb < 1 || D < 1 || r < 1;
}

/* gr_read: eq rms → eq gate → eq use_gate, and eq s, for n tokens. */
int gro_read(int64_t n, int nb, int D, int r, double eps, const double *R, const double *gamma,
             const double *Wd, const double *Wu, const double *Ww, double *x, double *s,
             double *G_out, double *inv_out)
{
    if (bad_dims(n, nb, D, r) || !R || !gamma || !Wd || !Wu || !Ww || !x || !s)
        return -1;
    const size_t K = (size_t)nb * D;
    int failed = 0;
#pragma omp parallel
    {
        double *Rh = malloc(K * sizeof(double));
        double *g = malloc(K * sizeof(double));
        double *h = malloc((size_t)r * sizeof(double));
        double *inv = malloc((size_t)nb * sizeof(double));
        if (!Rh || !g || !h || !inv) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t) {
                group_rmsnorm(nb, D, eps, R + (size_t)t * K, gamma, Rh, inv);
                read_from_normalised(nb, D, r, Rh, Wd, Wu, Ww, h, g, x + (size_t)t * D,
                                     s + (size_t)t * nb, G_out ? G_out + (size_t)t * K : NULL);
                if (inv_out)
                    memcpy(inv_out + (size_t)t * nb, inv, (size_t)nb * sizeof(double));
            }
        }
        free(Rh);
        free(g);
        free(h);
        free(inv);
    }
    return failed ? -2 : 0;
}

/* ---- backward (the chain rule through eq rms … eq s and eq write) ----------------------------
 * Gradients of a scalar loss L given dL/dx [n][D] and dL/ds [n][nb] (the read's outputs).
 * Per token, with a = W_d vec R̂ / n_r, u = W_w vec R̂ / n_r, g = W_u h (the read's own
 * intermediates, recomputed in fp64):
 *   dG_i[c]  = dx[c] · R̂_i[c] / n_r                dR̂_i[c] += dx[c] · G_i[c] / n_r
 *   dg       = dG ⊙ G ⊙ (1 − G)                     (σ' = σ(1 − σ))
 *   dh       = W_uᵀ dg,        dW_u += dg ⊗ h
 *   dz       = dh ⊙ SiLU'(z),  SiLU'(z) = σ(z)(1 + z(1 − σ(z)))
 *   du       = ds ⊙ 2σ(u)(1 − σ(u))
 *   dvec R̂ += (W_dᵀ dz + W_wᵀ du) / n_r,  dW_d += dz ⊗ vec R̂ / n_r,  dW_w += du ⊗ vec R̂ / n_r
 *   dγ_i[c] += dR̂_i[c] · R_i[c] · inv_i
 *   with p_i[c] = dR̂_i[c] γ_i[c]:  dR_i[c] = inv_i p_i[c] − inv_i³ R_i[c] Σ_c' p_i[c'] R_i[c'] / D
 * (the last line differentiates R̂_i = γ_i R_i (mean R_i² + eps)^-1/2). The weight gradients
 * are sums over the n tokens (outputs overwritten). */
int gro_read_backward(int64_t n, int nb, int D, int r, double eps, const double *R,
                      const double *gamma, const double *Wd, const double *Wu, const double *Ww,
                      const double *dx, const double *ds, double *dR, double *dgamma,
                      double *dWd, double *dWu, double *dWw)
{
    if (bad_dims(n, nb, D, r) || !R || !gamma || !Wd || !Wu || !Ww || !dx || !ds || !dR ||
        !dgamma || !dWd || !dWu || !dWw)
        return -1;
    const size_t K = (size_t)nb * D;
    const double inv_nb = 1.0 / (double)nb;
    memset(dgamma, 0, K * sizeof(double));
    memset(dWd, 0, (size_t)r * K * sizeof(double));
    memset(dWu, 0, K * (size_t)r * sizeof(double));
    memset(dWw, 0, (size_t)nb * K * sizeof(double));
    int failed = 0;
#pragma omp parallel
    {
        double *Rh = malloc(K * sizeof(double)), *inv = malloc((size_t)nb * sizeof(double));
        double *z = malloc((size_t)r * sizeof(double)), *h = malloc((size_t)r * sizeof(double));
        double *u = malloc((size_t)nb * sizeof(double)), *G = malloc(K * sizeof(double));
        double *dRh = malloc(K * sizeof(double)), *dg = malloc(K * sizeof(double));
        double *dz = malloc((size_t)r * sizeof(double)), *du = malloc((size_t)nb * sizeof(double));
        /* per-thread partial sums of the parameter gradients */
        double *pg = calloc(K, sizeof(double)), *pWd = calloc((size_t)r * K, sizeof(double));
        double *pWu = calloc(K * (size_t)r, sizeof(double));
        double *pWw = calloc((size_t)nb * K, sizeof(double));
        if (!Rh || !inv || !z || !h || !u || !G || !dRh || !dg || !dz || !du || !pg || !pWd ||
            !pWu || !pWw) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t) {
                const double *Rt = R + (size_t)t * K;
                const double *dxt = dx + (size_t)t * D, *dst = ds + (size_t)t * nb;
                group_rmsnorm(nb, D, eps, Rt, gamma, Rh, inv);
                for (int k = 0; k < r; ++k) {          /* z, h */
                    double acc = 0.0;
                    for (size_t j = 0; j < K; ++j)
                        acc += Wd[(size_t)k * K + j] * Rh[j];
                    z[k] = inv_nb * acc;
                    h[k] = silu(z[k]);
                }
                for (size_t j = 0; j < K; ++j) {       /* G */
                    double acc = 0.0;
                    for (int k = 0; k < r; ++k)
                        acc += Wu[j * (size_t)r + k] * h[k];
                    G[j] = sigmoid(acc);
                }
                for (int i = 0; i < nb; ++i) {          /* u */
                    double acc = 0.0;
                    for (size_t j = 0; j < K; ++j)
                        acc += Ww[(size_t)i * K + j] * Rh[j];
                    u[i] = inv_nb * acc;
                }
                /* eq use_gate: x[c] = (1/n_r) Σ_i G_i[c] R̂_i[c] */
                for (int i = 0; i < nb; ++i)
                    for (int c = 0; c < D; ++c) {
                        const size_t j = (size_t)i * D + c;
                        const double dG = inv_nb * dxt[c] * Rh[j];
                        dRh[j] = inv_nb * dxt[c] * G[j];
                        dg[j] = dG * G[j] * (1.0 - G[j]);
                    }
                /* eq gate: g = W_u h, h = SiLU(z) */
                for (int k = 0; k < r; ++k) {
                    double acc = 0.0;
                    for (size_t j = 0; j < K; ++j)
                        acc += Wu[j * (size_t)r + k] * dg[j];
                    const double sg = sigmoid(z[k]);
                    dz[k] = acc * sg * (1.0 + z[k] * (1.0 - sg));
                }
                for (size_t j = 0; j < K; ++j)
                    for (int k = 0; k < r; ++k)
                        pWu[j * (size_t)r + k] += dg[j] * h[k];
                /* eq s: s = 2σ(u) */
                for (int i = 0; i < nb; ++i) {
                    const double sg = sigmoid(u[i]);
                    du[i] = dst[i] * 2.0 * sg * (1.0 - sg);
                }
                /* z = W_d vec R̂ / n_r and u = W_w vec R̂ / n_r */
                for (size_t j = 0; j < K; ++j) {
                    double acc = 0.0;
                    for (int k = 0; k < r; ++k)
                        acc += Wd[(size_t)k * K + j] * dz[k];
                    for (int i = 0; i < nb; ++i)
                        acc += Ww[(size_t)i * K + j] * du[i];
                    dRh[j] += inv_nb * acc;
                }
                for (int k = 0; k < r; ++k)
                    for (size_t j = 0; j < K; ++j)
                        pWd[(size_t)k * K + j] += inv_nb * dz[k] * Rh[j];
                for (int i = 0; i < nb; ++i)
                    for (size_t j = 0; j < K; ++j)
                        pWw[(size_t)i * K + j] += inv_nb * du[i] * Rh[j];
                /* eq rms: R̂_i = γ_i R_i inv_i */
                for (int i = 0; i < nb; ++i) {
                    const double *Ri = Rt + (size_t)i * D;
                    double pr = 0.0;
                    for (int c = 0; c < D; ++c) {
                        const size_t j = (size_t)i * D + c;
                        pg[j] += dRh[j] * Ri[c] * inv[i];
                        pr += dRh[j] * gamma[j] * Ri[c];
                    }
                    const double i3 = inv[i] * inv[i] * inv[i];
                    for (int c = 0; c < D; ++c) {
                        const size_t j = (size_t)i * D + c;
                        dR[(size_t)t * K + j] =
                            inv[i] * dRh[j] * gamma[j] - i3 * Ri[c] * pr / (double)D;
                    }
                }
            }
#pragma omp critical
            {
                for (size_t j = 0; j < K; ++j)
                    dgamma[j] += pg[j];
                for (size_t j = 0; j < (size_t)r * K; ++j) {
                    dWd[j] += pWd[j];
                    dWu[j] += pWu[j];
                }
                for (size_t j = 0; j < (size_t)nb * K; ++j)
                    dWw[j] += pWw[j];
            }
        }
        free(Rh); free(inv); free(z); free(h); free(u); free(G); free(dRh); free(dg); free(dz);
        free(du); free(pg); free(pWd); free(pWu); free(pWw);
    }
    return failed ? -2 : 0;
}

/* Backward of eq write R' = R + s_i y: dR = dR', ds_i = Σ_c dR'_i[c] y[c], dy = Σ_i s_i dR'_i.
 * dR may equal dRp. */
int gro_write_backward(int64_t n, int nb, int D, const double *dRp, const double *y,
                       const double *s, double *dR, double *dy, double *ds)
{
    if (n < 0 || nb < 1 || D < 1 || !dRp || !y || !s || !dR || !dy || !ds)
        return -1;
    const size_t K = (size_t)nb * D;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int c = 0; c < D; ++c) {
            double acc = 0.0;
            for (int i = 0; i < nb; ++i)
                acc += s[(size_t)t * nb + i] * dRp[(size_t)t * K + (size_t)i * D + c];
            dy[(size_t)t * D + c] = acc;
        }
        for (int i = 0; i < nb; ++i) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += dRp[(size_t)t * K + (size_t)i * D + c] * y[(size_t)t * D + c];
            ds[(size_t)t * nb + i] = acc;
        }
        for (size_t j = 0; j < K; ++j)
            dR[(size_t)t * K + j] = dRp[(size_t)t * K + j];
    }
    return 0;
}

/* ---- contribution decomposition (eq auv and π, §二.6) -----------------------------------------
 * GR never mixes branches, so each branch of the state block v reads is the initial state plus
 * the writes of the blocks before it, and the read splits exactly into per-writer terms. Reader v
 * reads R (= R^(v)) with its parameters; writers u = 0..U-1 wrote y^(u) with strengths s^(u).
 * Per token, with G the read's gates and inv_i = 1/rms(R_i):
 *   a_{u→v,i}[c] = (1/n_r) G_i[c] γ_i[c] inv_i s_i^(u) y^(u)[c]     (branch i's share)
 *   a_{u→v}[c]   = Σ_i a_{u→v,i}[c]                                    (eq auv)
 *   norm[u]      = ‖a_{u→v}‖₂ over the D channels,  bnorm[u][i] = ‖a_{u→v,i}‖₂
 *   pi[u]        = norm[u] / Σ_u' norm[u']  (0 when that sum is 0)
 *   a_{0→v}[c]   = (1/n_r) Σ_i G_i[c] γ_i[c] inv_i R0_i[c],  a0_norm = ‖a_{0→v}‖₂  (R0 given)
 * Layouts: Y [U][n][D], S [U][n][nb], R0 [n][nb][D] (or NULL); outputs norm [n][U],
 * bnorm [n][U][nb], pi [n][U], a0_norm [n] (with R0); optional vectors A [n][U][D], A0 [n][D]. */
int gro_decompose(int64_t n, int nb, int D, int r, double eps, const double *R,
                  const double *gamma, const double *Wd, const double *Wu, const double *Ww,
                  int U, const double *Y, const double *S, const double *R0, double *norm,
                  double *bnorm, double *pi, double *a0_norm, double *A, double *A0)
{
    if (bad_dims(n, nb, D, r) || U < 0 || !R || !gamma || !Wd || !Wu || !Ww || !norm ||
        !bnorm || !pi || (U > 0 && (!Y || !S)) || (R0 && !a0_norm))
        return -1;
    const size_t K = (size_t)nb * D;
    const double inv_nb = 1.0 / (double)nb;
    int failed = 0;
#pragma omp parallel
    {
        double *Rh = malloc(K * sizeof(double));
        double *G = malloc(K * sizeof(double));
        double *h = malloc((size_t)r * sizeof(double));
        double *inv = malloc((size_t)nb * sizeof(double));
        double *xs = malloc(((size_t)D + nb) * sizeof(double));
        double *bq = malloc((size_t)nb * sizeof(double));
        if (!Rh || !G || !h || !inv || !xs || !bq) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t) {
                const double *Rt = R + (size_t)t * K;
                group_rmsnorm(nb, D, eps, Rt, gamma, Rh, inv);
                read_from_normalised(nb, D, r, Rh, Wd, Wu, Ww, h, G, xs, xs + D, NULL);
                double total = 0.0;
                for (int u = 0; u < U; ++u) {
                    const double *yu = Y + ((size_t)u * n + t) * D;
                    const double *su = S + ((size_t)u * n + t) * nb;
                    double sq = 0.0;
                    for (int i = 0; i < nb; ++i)
                        bq[i] = 0.0;
                    for (int c = 0; c < D; ++c) {
                        double a = 0.0;
                        for (int i = 0; i < nb; ++i) {
                            const size_t j = (size_t)i * D + c;
                            const double ai = inv_nb * G[j] * gamma[j] * inv[i] * su[i] * yu[c];
                            bq[i] += ai * ai;
                            a += ai;
                        }
                        sq += a * a;
                        if (A)
                            A[((size_t)t * U + u) * D + c] = a;
                    }
                    norm[(size_t)t * U + u] = sqrt(sq);
                    for (int i = 0; i < nb; ++i)
                        bnorm[((size_t)t * U + u) * nb + i] = sqrt(bq[i]);
                    total += sqrt(sq);
                }
                for (int u = 0; u < U; ++u)
                    pi[(size_t)t * U + u] = total > 0.0 ? norm[(size_t)t * U + u] / total : 0.0;
                if (R0) {
                    const double *R0t = R0 + (size_t)t * K;
                    double sq = 0.0;
                    for (int c = 0; c < D; ++c) {
                        double a = 0.0;
                        for (int i = 0; i < nb; ++i) {
                            const size_t j = (size_t)i * D + c;
                            a += inv_nb * G[j] * gamma[j] * inv[i] * R0t[j];
                        }
                        sq += a * a;
                        if (A0)
                            A0[(size_t)t * D + c] = a;
                    }
                    a0_norm[t] = sqrt(sq);
                }
            }
        }
        free(Rh); free(G); free(h); free(inv); free(xs); free(bq);
    }
    return failed ? -2 : 0;
}

/* gr_write: eq write, R'_i = R_i + s_i y, for n tokens. R_out may equal R. */
int gro_write(int64_t n, int nb, int D, const double *R, const double *y, const double *s,
              double *R_out)
{
    if (n < 0 || nb < 1 || D < 1 || !R || !y || !s || !R_out)
        return -1;
    const size_t K = (size_t)nb * D;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int i = 0; i < nb; ++i) {
            const double si = s[(size_t)t * nb + i];
            for (int c = 0; c < D; ++c) {
                size_t e = (size_t)t * K + (size_t)i * D + c;
                R_out[e] = R[e] + si * y[(size_t)t * D + c];
            }
        }
    }
    return 0;
}

/* gr_write_then_read: eq write with the previous sublayer's s, then the read of the next
 * sublayer on the written state (kept in fp64, not rounded). */
int gro_write_then_read(int64_t n, int nb, int D, int r, double eps, const double *R,
                        const double *y, const double *s_prev, const double *gamma,
                        const double *Wd, const double *Wu, const double *Ww, double *R_out,
                        double *x, double *s_next)
{
    int st = gro_write(n, nb, D, R, y, s_prev, R_out);
    if (st)
        return st;
    return gro_read(n, nb, D, r, eps, R_out, gamma, Wd, Wu, Ww, x, s_next, NULL, NULL);
}

/* The combine of eq use_gate with the gates given instead of predicted:
 * x = (1/n_r) Σ_i G_i ⊙ RMSNorm(R_i; γ_i). G is [nb][D], the same for every token. */
int gro_read_fixed_gates(int64_t n, int nb, int D, double eps, const double *R,
                         const double *gamma, const double *G, double *x)
{
    if (n < 0 || nb < 1 || D < 1 || !R || !gamma || !G || !x)
        return -1;
    const size_t K = (size_t)nb * D;
    int failed = 0;
#pragma omp parallel
    {
        double *Rh = malloc(K * sizeof(double));
        double *inv = malloc((size_t)nb * sizeof(double));
        if (!Rh || !inv) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t) {
                group_rmsnorm(nb, D, eps, R + (size_t)t * K, gamma, Rh, inv);
                for (int c = 0; c < D; ++c) {
                    double acc = 0.0;
                    for (int i = 0; i < nb; ++i)
                        acc += G[(size_t)i * D + c] * Rh[(size_t)i * D + c];
                    x[(size_t)t * D + c] = acc / (double)nb;
                }
            }
        }
        free(Rh);
        free(inv);
    }
    return failed ? -2 : 0;
}

/* Round v to the nearest value with `bits` significant bits, ties to even (normal range).
 * bits = 8 is bfloat16 (7 stored fraction bits), bits = 24 is IEEE binary32. Used to model a
 * state stored in that format: the read after a write sees the stored value. */
static double round_significand(double v, int bits)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    int e;
    frexp(v, &e);                       /* v = m·2^e, 0.5 <= |m| < 1 */
    double scale = ldexp(1.0, bits - e); /* |v|·scale in [2^(bits-1), 2^bits) */
    return nearbyint(v * scale) / scale; /* default rounding mode: nearest, ties to even */
}

/* In place: v[e] = round_significand(v[e], bits) for e < n. */
int gro_round_significand(int64_t n, int bits, double *v)
{
    if (n < 0 || bits < 2 || bits > 52 || !v)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e)
        v[e] = round_significand(v[e], bits);
    return 0;
}

/* ---- FP8 state (OCP e4m3 "e4m3fn" codes, one power-of-two scale per 32-channel block) ----
 * The pages name FP8 storage of the widened state ("【论文解读】 Qwen3.8 Flash Next", §二.7)
 * without a format; this file fixes the one used here, as follows.
 * An e4m3 code is sign | 4 exponent bits (bias 7) | 3 fraction bits; exponent field 0 holds
 * the subnormals m/8 · 2^-6; 0x7F and 0xFF are NaN; there are no infinities. */

/* Value of one e4m3 code. */
static double fp8_decode(uint8_t code)
{
    const int sign = code >> 7, E = (code >> 3) & 15, m = code & 7;
    if (E == 15 && m == 7)
        return NAN;
    const double mag = E == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, E - 10);
    return sign ? -mag : mag;
}

/* Nearest e4m3 code to w (ties to even), for |w| <= 448 (larger magnitudes saturate to 448). */
static uint8_t fp8_encode(double w)
{
    if (isnan(w))
        return 0x7F;
    const uint8_t sign = signbit(w) ? 0x80 : 0;
    double a = fabs(w);
    if (a >= 448.0)
        return sign | 0x7E;               /* 448 = 2^8 · 1.75: exponent field 15, fraction 6 */
    if (a < ldexp(1.0, -6)) {             /* subnormal: a multiple of 2^-9 */
        const double m = nearbyint(ldexp(a, 9)); /* 0 .. 8; 8 is the smallest normal, 2^-6 */
        return sign | (uint8_t)m;
    }
    int E;
    frexp(a, &E);                         /* a = f·2^E, 0.5 <= f < 1: binary exponent E-1 */
    E -= 1;                               /* a in [2^E, 2^(E+1)) */
    double m = nearbyint(ldexp(a, 3 - E)); /* 8 .. 16 */
    if (m == 16.0) {
        m = 8.0;
        E += 1;
    }
    if (E + 7 > 15 || (E + 7 == 15 && m > 14.0))
        return sign | 0x7E;               /* rounding went past 448 */
    return sign | (uint8_t)(((E + 7) << 3) | ((int)m - 8));
}

/* Scale exponent of a block whose largest magnitude is a: the smallest e with a <= 448·2^e,
 * clamped to [-127, 127] (a = 0 gives -127). */
static int fp8_block_exponent(double a)
{
    if (!(a > 0.0))
        return -127;
    int E;
    const double f = frexp(a, &E);        /* a = f·2^E, f in [0.5, 1): significand 2f */
    int e = (E - 1) - 8;                  /* 448·2^e = 1.75·2^(e+8) */
    if (2.0 * f > 1.75)
        e += 1;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* Encode rows of D values (D a multiple of 32) into e4m3 codes [rows][D] and biased block
 * exponents [rows][D/32] (scale 2^(b-127)). The inputs are exact fp32 values (the stored
 * write result), so dividing by the power-of-two scale is exact. */
int gro_fp8_encode(int64_t rows, int D, const double *v, uint8_t *codes, uint8_t *scales)
{
    if (rows < 0 || D < 32 || D % 32 || !v || !codes || !scales)
        return -1;
    const int nblk = D / 32;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows; ++t) {
        for (int k = 0; k < nblk; ++k) {
            const double *vb = v + (size_t)t * D + (size_t)k * 32;
            double a = 0.0;
            for (int c = 0; c < 32; ++c)
                if (fabs(vb[c]) > a)
                    a = fabs(vb[c]);
            const int e = fp8_block_exponent(a);
            scales[(size_t)t * nblk + k] = (uint8_t)(e + 127);
            for (int c = 0; c < 32; ++c)
                codes[(size_t)t * D + (size_t)k * 32 + c] = fp8_encode(ldexp(vb[c], -e));
        }
    }
    return 0;
}

/* Decode codes [rows][D] with block exponents [rows][D/32] into values. */
int gro_fp8_decode(int64_t rows, int D, const uint8_t *codes, const uint8_t *scales, double *v)
{
    if (rows < 0 || D < 32 || D % 32 || !v || !codes || !scales)
        return -1;
    const int nblk = D / 32;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows; ++t)
        for (int c = 0; c < D; ++c)
            v[(size_t)t * D + c] = ldexp(fp8_decode(codes[(size_t)t * D + c]),
                                         (int)scales[(size_t)t * nblk + c / 32] - 127);
    return 0;
}

/* The value of each single code 0..255 (for checks against other e4m3 implementations). */
int gro_fp8_code_values(double *out)
{
    if (!out)
        return -1;
    for (int c = 0; c < 256; ++c)
        out[c] = fp8_decode((uint8_t)c);
    return 0;
}

/* Nearest e4m3 code of each value (|w| <= 448; ties to even), no block scale. */
int gro_fp8_round_codes(int64_t n, const double *w, uint8_t *codes)
{
    if (n < 0 || !w || !codes)
        return -1;
    for (int64_t e = 0; e < n; ++e)
        codes[e] = fp8_encode(w[e]);
    return 0;
}

/* Single-stream residual add x += y (the bandwidth reference path), n elements. */
int gro_residual_add(int64_t n, const double *y, double *x)
{
    if (n < 0 || !y || !x)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e)
        x[e] += y[e];
    return 0;
}

/* Number of threads the parallel loops above use (1 without OpenMP). */
int gro_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the thread count of the parallel loops (no-op without OpenMP). */
void gro_set_num_threads(int k)
{
#ifdef _OPENMP
    if (k > 0)
        omp_set_num_threads(k);
#else
    (void)k;
#endif
}
