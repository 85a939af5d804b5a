/*
 * ssim_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of the differentiable SSIM loss.
 * It exists to check the CUDA library against; it is never part of the product
 * path.  Only the tests, the package's smoke check and the benchmark's CPU
 * baseline may build, load or call it.  It shares no code, header, table or
 * constant with the CUDA sources, and the CUDA sources do not include it.
 *
 * What it follows:
 *   - fused-ssim README, introduction: an 11x11 Gaussian window with fixed
 *     weights "as per the original SSIM paper"; windows in 2D and 3D;
 *     any number of channels and batch items.
 *   - fused-ssim README, "Usage": padding "same" (output the size of the input)
 *     or "valid" (only windows that fit inside the image); the result is the
 *     mean of the SSIM map.
 *   - fused-ssim README, "Constraints": images lie in [0, 1], so the data range
 *     is 1 and the stabilising constants are C1 = (0.01*1)^2, C2 = (0.03*1)^2.
 *   - TriSSIM README, "How it works": the forward blurs five quantities
 *     (mu1, mu2, s11, s22, s12) -- read here as the raw moments E[x], E[y],
 *     E[x^2], E[y^2], E[xy] -- and the backward applies the blur's adjoint to
 *     the five upstream gradients, then the chain rule
 *         grad_img1 = B^T(g_mu1) + 2*img1*B^T(g_s11) + img2*B^T(g_s12)
 *         grad_img2 = B^T(g_mu2) + 2*img2*B^T(g_s22) + img1*B^T(g_s12).
 *   - fused-ssim README, "3D data": the same statistics with an 11x11x11 window.
 *
 * Every blur here is the DIRECT window sum (121 or 1331 terms per output);
 * there is no separable pass, no tiling and no reordering of any sum.  The
 * adjoint B^T is the transpose of B taken entry by entry.  Loops over
 * independent outputs may run on several threads (OpenMP); no sum is split.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   sigma = 1.5; weights normalised in double; "same" pads with zeros and does
 *   not renormalise border windows; no clamp on the variances; the mean of
 *   image n runs over its channels and output pixels; dL[n] is the upstream
 *   derivative of the loss with respect to mean[n].
 *
 * Layout: NCHW (2D) and NCDHW (3D), contiguous, row-major, double.
 * Padding code: 0 = valid, 1 = same (zero).
 * Every function returns 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TAPS 11
#define RADIUS 5

static const double SIGMA = 1.5;
static const double DATA_RANGE = 1.0;

static double c1_const(void) { return (0.01 * DATA_RANGE) * (0.01 * DATA_RANGE); }
static double c2_const(void) { return (0.03 * DATA_RANGE) * (0.03 * DATA_RANGE); }

/* ---------------------------------------------------------------- utilities */

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* The sampled 1D Gaussian, w_k proportional to exp(-(k-5)^2 / (2 sigma^2)),
 * k = 0..10, scaled so that the eleven weights sum to one. */
void oracle_gauss_window(double w[TAPS])
{
    double total = 0.0;
    for (int k = 0; k < TAPS; ++k) {
        double d = (double)(k - RADIUS);
        w[k] = exp(-(d * d) / (2.0 * SIGMA * SIGMA));
        total += w[k];
    }
    for (int k = 0; k < TAPS; ++k) w[k] /= total;
}

/* Extent of the output domain along one axis. */
int oracle_out_extent(int n, int padding)
{
    if (padding == 0) return n - (TAPS - 1);
    if (padding == 1) return n;
    return -1;
}

/* Offset between an output index and the first input its window touches:
 * window of output p covers inputs p - off .. p - off + 10. */
static int window_offset(int padding) { return padding == 0 ? 0 : RADIUS; }

static int check_extent(int n, int padding)
{
    if (padding != 0 && padding != 1) return -1;
    if (n < 1) return -1;
    if (padding == 0 && n < TAPS) return -1;
    return 0;
}

/* -------------------------------------------------------------- the 2D blur */

/* (B f)(i, j) = sum_{a,b} w_a w_b f(i + a - off, j + b - off), f = 0 outside
 * the H x W image.  out has the output extent Ho x Wo. */
int oracle_blur2d(const double *f, int H, int W, int padding, double *out)
{
    if (!f || !out || check_extent(H, padding) || check_extent(W, padding)) return -1;
    const int Ho = oracle_out_extent(H, padding), Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    double w[TAPS], win[TAPS][TAPS];
    oracle_gauss_window(w);
    for (int a = 0; a < TAPS; ++a)
        for (int b = 0; b < TAPS; ++b) win[a][b] = w[a] * w[b];

#pragma omp parallel for schedule(static)
    for (int i = 0; i < Ho; ++i) {
        for (int j = 0; j < Wo; ++j) {
            double acc = 0.0;
            for (int a = 0; a < TAPS; ++a) {
                const int r = i + a - off;
                if (r < 0 || r >= H) continue;
                for (int b = 0; b < TAPS; ++b) {
                    const int c = j + b - off;
                    if (c < 0 || c >= W) continue;
                    acc += win[a][b] * f[(size_t)r * W + c];
                }
            }
            out[(size_t)i * Wo + j] = acc;
        }
    }
    return 0;
}

/* The transpose of oracle_blur2d as a matrix: B has entry w_a w_b in row p,
 * column q = p + (a, b) - off, so
 *   (B^T g)(q) = sum_{a,b} w_a w_b g(q_i - a + off, q_j - b + off),
 * with g = 0 outside the Ho x Wo output domain.  out is H x W. */
int oracle_blur2d_adjoint(const double *g, int H, int W, int padding, double *out)
{
    if (!g || !out || check_extent(H, padding) || check_extent(W, padding)) return -1;
    const int Ho = oracle_out_extent(H, padding), Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    double w[TAPS], win[TAPS][TAPS];
    oracle_gauss_window(w);
    for (int a = 0; a < TAPS; ++a)
        for (int b = 0; b < TAPS; ++b) win[a][b] = w[a] * w[b];

#pragma omp parallel for schedule(static)
    for (int qi = 0; qi < H; ++qi) {
        for (int qj = 0; qj < W; ++qj) {
            double acc = 0.0;
            for (int a = 0; a < TAPS; ++a) {
                const int pi = qi - a + off;
                if (pi < 0 || pi >= Ho) continue;
                for (int b = 0; b < TAPS; ++b) {
                    const int pj = qj - b + off;
                    if (pj < 0 || pj >= Wo) continue;
                    acc += win[a][b] * g[(size_t)pi * Wo + pj];
                }
            }
            out[(size_t)qi * W + qj] = acc;
        }
    }
    return 0;
}

/* -------------------------------------------------------------- the 3D blur */

int oracle_blur3d(const double *f, int D, int H, int W, int padding, double *out)
{
    if (!f || !out || check_extent(D, padding) || check_extent(H, padding) ||
        check_extent(W, padding))
        return -1;
    const int Do = oracle_out_extent(D, padding), Ho = oracle_out_extent(H, padding),
              Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    double w[TAPS];
    oracle_gauss_window(w);

#pragma omp parallel for collapse(2) schedule(static)
    for (int k = 0; k < Do; ++k) {
        for (int i = 0; i < Ho; ++i) {
            for (int j = 0; j < Wo; ++j) {
                double acc = 0.0;
                for (int c = 0; c < TAPS; ++c) {
                    const int z = k + c - off;
                    if (z < 0 || z >= D) continue;
                    for (int a = 0; a < TAPS; ++a) {
                        const int r = i + a - off;
                        if (r < 0 || r >= H) continue;
                        for (int b = 0; b < TAPS; ++b) {
                            const int s = j + b - off;
                            if (s < 0 || s >= W) continue;
                            acc += w[c] * w[a] * w[b] * f[((size_t)z * H + r) * W + s];
                        }
                    }
                }
                out[((size_t)k * Ho + i) * Wo + j] = acc;
            }
        }
    }
    return 0;
}

int oracle_blur3d_adjoint(const double *g, int D, int H, int W, int padding, double *out)
{
    if (!g || !out || check_extent(D, padding) || check_extent(H, padding) ||
        check_extent(W, padding))
        return -1;
    const int Do = oracle_out_extent(D, padding), Ho = oracle_out_extent(H, padding),
              Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    double w[TAPS];
    oracle_gauss_window(w);

#pragma omp parallel for collapse(2) schedule(static)
    for (int qk = 0; qk < D; ++qk) {
        for (int qi = 0; qi < H; ++qi) {
            for (int qj = 0; qj < W; ++qj) {
                double acc = 0.0;
                for (int c = 0; c < TAPS; ++c) {
                    const int pk = qk - c + off;
                    if (pk < 0 || pk >= Do) continue;
                    for (int a = 0; a < TAPS; ++a) {
                        const int pi = qi - a + off;
                        if (pi < 0 || pi >= Ho) continue;
                        for (int b = 0; b < TAPS; ++b) {
                            const int pj = qj - b + off;
                            if (pj < 0 || pj >= Wo) continue;
                            acc += w[c] * w[a] * w[b] * g[((size_t)pk * Ho + pi) * Wo + pj];
                        }
                    }
                }
                out[((size_t)qk * H + qi) * W + qj] = acc;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------- SSIM at one output pixel */

/* SSIM from the five blurred raw moments, and its derivatives with respect to
 * each of them (the quotient rule applied to S = A1*A2 / (B1*B2)):
 *   sigma11 = e11 - mu1^2, sigma22 = e22 - mu2^2, sigma12 = e12 - mu1*mu2
 *   A1 = 2 mu1 mu2 + C1      A2 = 2 sigma12 + C2
 *   B1 = mu1^2 + mu2^2 + C1  B2 = sigma11 + sigma22 + C2
 * d[0..4] = dS/d(mu1, mu2, e11, e22, e12); d may be NULL. */
static double ssim_point(double mu1, double mu2, double e11, double e22, double e12,
                         double d[5])
{
    const double C1 = c1_const(), C2 = c2_const();
    const double s11 = e11 - mu1 * mu1;
    const double s22 = e22 - mu2 * mu2;
    const double s12 = e12 - mu1 * mu2;
    const double A1 = 2.0 * mu1 * mu2 + C1;
    const double A2 = 2.0 * s12 + C2;
    const double B1 = mu1 * mu1 + mu2 * mu2 + C1;
    const double B2 = s11 + s22 + C2;
    const double den = B1 * B2;
    const double S = (A1 * A2) / den;
    if (d) {
        /* derivatives of A1, A2, B1, B2 with respect to (mu1, mu2, e11, e22, e12) */
        const double dA1[5] = {2.0 * mu2, 2.0 * mu1, 0.0, 0.0, 0.0};
        const double dA2[5] = {-2.0 * mu2, -2.0 * mu1, 0.0, 0.0, 2.0};
        const double dB1[5] = {2.0 * mu1, 2.0 * mu2, 0.0, 0.0, 0.0};
        const double dB2[5] = {-2.0 * mu1, -2.0 * mu2, 1.0, 1.0, 0.0};
        for (int k = 0; k < 5; ++k) {
            const double dnum = dA1[k] * A2 + A1 * dA2[k];
            const double dden = dB1[k] * B2 + B1 * dB2[k];
            d[k] = dnum / den - S * dden / den;
        }
    }
    return S;
}

/* ------------------------------------------------------------- 2D SSIM loss */

/* Blur the five quantities x, y, x^2, y^2, x*y of one plane.
 * stats holds 5 maps of Ho*Wo each, in the order mu1, mu2, e11, e22, e12. */
static int plane_stats2d(const double *x, const double *y, int H, int W, int padding,
                         double *stats)
{
    const size_t n = (size_t)H * W;
    const size_t no = (size_t)oracle_out_extent(H, padding) * oracle_out_extent(W, padding);
    double *xx = malloc(n * sizeof(double)), *yy = malloc(n * sizeof(double)),
           *xy = malloc(n * sizeof(double));
    if (!xx || !yy || !xy) {
        free(xx); free(yy); free(xy);
        return -1;
    }
    for (size_t t = 0; t < n; ++t) {
        xx[t] = x[t] * x[t];
        yy[t] = y[t] * y[t];
        xy[t] = x[t] * y[t];
    }
    int rc = 0;
    rc |= oracle_blur2d(x, H, W, padding, stats + 0 * no);
    rc |= oracle_blur2d(y, H, W, padding, stats + 1 * no);
    rc |= oracle_blur2d(xx, H, W, padding, stats + 2 * no);
    rc |= oracle_blur2d(yy, H, W, padding, stats + 3 * no);
    rc |= oracle_blur2d(xy, H, W, padding, stats + 4 * no);
    free(xx); free(yy); free(xy);
    return rc;
}

/* The five blurred statistics of every plane: out is N*C*5*Ho*Wo, stat-major
 * inside each plane (mu1, mu2, e11, e22, e12). */
int oracle_ssim2d_stats(const double *x, const double *y, int N, int C, int H, int W,
                        int padding, double *out)
{
    if (!x || !y || !out || N < 1 || C < 1 || check_extent(H, padding) ||
        check_extent(W, padding))
        return -1;
    const size_t n = (size_t)H * W;
    const size_t no = (size_t)oracle_out_extent(H, padding) * oracle_out_extent(W, padding);
    for (size_t pl = 0; pl < (size_t)N * C; ++pl)
        if (plane_stats2d(x + pl * n, y + pl * n, H, W, padding, out + pl * 5 * no)) return -1;
    return 0;
}

/* Forward: mean[n] = (1 / (C*|Omega|)) * sum over channels and output pixels of
 * S; map (N*C*Ho*Wo) receives S when non-NULL. */
int oracle_ssim2d(const double *x, const double *y, int N, int C, int H, int W, int padding,
                  double *mean, double *map)
{
    if (!x || !y || !mean || N < 1 || C < 1 || check_extent(H, padding) ||
        check_extent(W, padding))
        return -1;
    const size_t n = (size_t)H * W;
    const size_t no = (size_t)oracle_out_extent(H, padding) * oracle_out_extent(W, padding);
    double *stats = malloc(5 * no * sizeof(double));
    if (!stats) return -1;
    for (int b = 0; b < N; ++b) {
        double total = 0.0;
        for (int c = 0; c < C; ++c) {
            const size_t pl = (size_t)b * C + c;
            if (plane_stats2d(x + pl * n, y + pl * n, H, W, padding, stats)) {
                free(stats);
                return -1;
            }
            for (size_t p = 0; p < no; ++p) {
                const double S = ssim_point(stats[p], stats[no + p], stats[2 * no + p],
                                            stats[3 * no + p], stats[4 * no + p], NULL);
                if (map) map[pl * no + p] = S;
                total += S;
            }
        }
        mean[b] = total / ((double)C * (double)no);
    }
    free(stats);
    return 0;
}

/* Backward: with dL[n] = dLoss/dmean[n], the upstream gradient of statistic k
 * at output pixel p is g_k(p) = dL[n] / (C*|Omega|) * dS/dk(p); then
 *   grad1 = B^T g_mu1 + 2 x B^T g_e11 + y B^T g_e12
 *   grad2 = B^T g_mu2 + 2 y B^T g_e22 + x B^T g_e12.
 * grad2 may be NULL. */
int oracle_ssim2d_grad(const double *x, const double *y, const double *dL, int N, int C,
                       int H, int W, int padding, double *grad1, double *grad2)
{
    if (!x || !y || !dL || !grad1 || N < 1 || C < 1 || check_extent(H, padding) ||
        check_extent(W, padding))
        return -1;
    const size_t n = (size_t)H * W;
    const size_t no = (size_t)oracle_out_extent(H, padding) * oracle_out_extent(W, padding);
    double *stats = malloc(5 * no * sizeof(double));
    double *g = malloc(5 * no * sizeof(double));   /* g_mu1, g_mu2, g_e11, g_e22, g_e12 */
    double *bt = malloc(5 * n * sizeof(double));   /* B^T of each */
    if (!stats || !g || !bt) {
        free(stats); free(g); free(bt);
        return -1;
    }
    int rc = 0;
    for (int b = 0; b < N && !rc; ++b) {
        const double scale = dL[b] / ((double)C * (double)no);
        for (int c = 0; c < C && !rc; ++c) {
            const size_t pl = (size_t)b * C + c;
            const double *xp = x + pl * n, *yp = y + pl * n;
            rc |= plane_stats2d(xp, yp, H, W, padding, stats);
            for (size_t p = 0; p < no; ++p) {
                double d[5];
                ssim_point(stats[p], stats[no + p], stats[2 * no + p], stats[3 * no + p],
                           stats[4 * no + p], d);
                for (int k = 0; k < 5; ++k) g[k * no + p] = scale * d[k];
            }
            for (int k = 0; k < 5; ++k)
                rc |= oracle_blur2d_adjoint(g + k * no, H, W, padding, bt + k * n);
            const double *bt_mu1 = bt, *bt_mu2 = bt + n, *bt_e11 = bt + 2 * n,
                         *bt_e22 = bt + 3 * n, *bt_e12 = bt + 4 * n;
            for (size_t q = 0; q < n; ++q) {
                grad1[pl * n + q] = bt_mu1[q] + 2.0 * xp[q] * bt_e11[q] + yp[q] * bt_e12[q];
                if (grad2)
                    grad2[pl * n + q] = bt_mu2[q] + 2.0 * yp[q] * bt_e22[q] + xp[q] * bt_e12[q];
            }
        }
    }
    free(stats); free(g); free(bt);
    return rc ? -1 : 0;
}

/* Window statistics of one 2D output pixel (i, j) of one plane, straight from
 * the definition of B.  s[0..4] = mu1, mu2, e11, e22, e12. */
static void pixel_stats2d(const double *x, const double *y, int H, int W, int off,
                          const double w[TAPS], int i, int j, double s[5])
{
    for (int k = 0; k < 5; ++k) s[k] = 0.0;
    for (int a = 0; a < TAPS; ++a) {
        const int r = i + a - off;
        if (r < 0 || r >= H) continue;
        for (int b = 0; b < TAPS; ++b) {
            const int c = j + b - off;
            if (c < 0 || c >= W) continue;
            const double wt = w[a] * w[b];
            const double xv = x[(size_t)r * W + c], yv = y[(size_t)r * W + c];
            s[0] += wt * xv;
            s[1] += wt * yv;
            s[2] += wt * (xv * xv);
            s[3] += wt * (yv * yv);
            s[4] += wt * (xv * yv);
        }
    }
}

/* The gradients at selected input elements only, for checks on images too
 * large for oracle_ssim2d_grad.  idx[t] is a flat NCHW index; g1[t] (and g2[t]
 * when non-NULL) receive the gradient there.  Same definitions as above,
 * evaluated one element at a time. */
int oracle_ssim2d_grad_at(const double *x, const double *y, const double *dL, int N, int C,
                          int H, int W, int padding, long long count, const long long *idx,
                          double *g1, double *g2)
{
    if (!x || !y || !dL || !idx || !g1 || N < 1 || C < 1 || count < 0 ||
        check_extent(H, padding) || check_extent(W, padding))
        return -1;
    const int Ho = oracle_out_extent(H, padding), Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    const size_t n = (size_t)H * W;
    double w[TAPS];
    oracle_gauss_window(w);
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (long long t = 0; t < count; ++t) {
        const long long f = idx[t];
        if (f < 0 || f >= (long long)N * C * (long long)n) {
            bad = 1;
            continue;
        }
        const size_t pl = (size_t)(f / (long long)n);
        const int qi = (int)((f % (long long)n) / W), qj = (int)(f % W);
        const int b = (int)(pl / (size_t)C);
        const double scale = dL[b] / ((double)C * (double)Ho * (double)Wo);
        const double *xp = x + pl * n, *yp = y + pl * n;
        double bt[5] = {0, 0, 0, 0, 0};
        for (int a = 0; a < TAPS; ++a) {
            const int pi = qi - a + off;
            if (pi < 0 || pi >= Ho) continue;
            for (int bb = 0; bb < TAPS; ++bb) {
                const int pj = qj - bb + off;
                if (pj < 0 || pj >= Wo) continue;
                double s[5], d[5];
                pixel_stats2d(xp, yp, H, W, off, w, pi, pj, s);
                ssim_point(s[0], s[1], s[2], s[3], s[4], d);
                for (int k = 0; k < 5; ++k) bt[k] += w[a] * w[bb] * (scale * d[k]);
            }
        }
        const double xv = xp[(size_t)qi * W + qj], yv = yp[(size_t)qi * W + qj];
        g1[t] = bt[0] + 2.0 * xv * bt[2] + yv * bt[4];
        if (g2) g2[t] = bt[1] + 2.0 * yv * bt[3] + xv * bt[4];
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------- 3D SSIM loss */

static int plane_stats3d(const double *x, const double *y, int D, int H, int W, int padding,
                         double *stats)
{
    const size_t n = (size_t)D * H * W;
    const size_t no = (size_t)oracle_out_extent(D, padding) * oracle_out_extent(H, padding) *
                      oracle_out_extent(W, padding);
    double *xx = malloc(n * sizeof(double)), *yy = malloc(n * sizeof(double)),
           *xy = malloc(n * sizeof(double));
    if (!xx || !yy || !xy) {
        free(xx); free(yy); free(xy);
        return -1;
    }
    for (size_t t = 0; t < n; ++t) {
        xx[t] = x[t] * x[t];
        yy[t] = y[t] * y[t];
        xy[t] = x[t] * y[t];
    }
    int rc = 0;
    rc |= oracle_blur3d(x, D, H, W, padding, stats + 0 * no);
    rc |= oracle_blur3d(y, D, H, W, padding, stats + 1 * no);
    rc |= oracle_blur3d(xx, D, H, W, padding, stats + 2 * no);
    rc |= oracle_blur3d(yy, D, H, W, padding, stats + 3 * no);
    rc |= oracle_blur3d(xy, D, H, W, padding, stats + 4 * no);
    free(xx); free(yy); free(xy);
    return rc;
}

static int check3d(int N, int C, int D, int H, int W, int padding)
{
    return (N < 1 || C < 1 || check_extent(D, padding) || check_extent(H, padding) ||
            check_extent(W, padding));
}

int oracle_ssim3d(const double *x, const double *y, int N, int C, int D, int H, int W,
                  int padding, double *mean, double *map)
{
    if (!x || !y || !mean || check3d(N, C, D, H, W, padding)) return -1;
    const size_t n = (size_t)D * H * W;
    const size_t no = (size_t)oracle_out_extent(D, padding) * oracle_out_extent(H, padding) *
                      oracle_out_extent(W, padding);
    double *stats = malloc(5 * no * sizeof(double));
    if (!stats) return -1;
    for (int b = 0; b < N; ++b) {
        double total = 0.0;
        for (int c = 0; c < C; ++c) {
            const size_t pl = (size_t)b * C + c;
            if (plane_stats3d(x + pl * n, y + pl * n, D, H, W, padding, stats)) {
                free(stats);
                return -1;
            }
            for (size_t p = 0; p < no; ++p) {
                const double S = ssim_point(stats[p], stats[no + p], stats[2 * no + p],
                                            stats[3 * no + p], stats[4 * no + p], NULL);
                if (map) map[pl * no + p] = S;
                total += S;
            }
        }
        mean[b] = total / ((double)C * (double)no);
    }
    free(stats);
    return 0;
}

int oracle_ssim3d_grad(const double *x, const double *y, const double *dL, int N, int C,
                       int D, int H, int W, int padding, double *grad1, double *grad2)
{
    if (!x || !y || !dL || !grad1 || check3d(N, C, D, H, W, padding)) return -1;
    const size_t n = (size_t)D * H * W;
    const size_t no = (size_t)oracle_out_extent(D, padding) * oracle_out_extent(H, padding) *
                      oracle_out_extent(W, padding);
    double *stats = malloc(5 * no * sizeof(double));
    double *g = malloc(5 * no * sizeof(double));
    double *bt = malloc(5 * n * sizeof(double));
    if (!stats || !g || !bt) {
        free(stats); free(g); free(bt);
        return -1;
    }
    int rc = 0;
    for (int b = 0; b < N && !rc; ++b) {
        const double scale = dL[b] / ((double)C * (double)no);
        for (int c = 0; c < C && !rc; ++c) {
            const size_t pl = (size_t)b * C + c;
            const double *xp = x + pl * n, *yp = y + pl * n;
            rc |= plane_stats3d(xp, yp, D, H, W, padding, stats);
            for (size_t p = 0; p < no; ++p) {
                double d[5];
                ssim_point(stats[p], stats[no + p], stats[2 * no + p], stats[3 * no + p],
                           stats[4 * no + p], d);
                for (int k = 0; k < 5; ++k) g[k * no + p] = scale * d[k];
            }
            for (int k = 0; k < 5; ++k)
                rc |= oracle_blur3d_adjoint(g + k * no, D, H, W, padding, bt + k * n);
            const double *bt_mu1 = bt, *bt_mu2 = bt + n, *bt_e11 = bt + 2 * n,
                         *bt_e22 = bt + 3 * n, *bt_e12 = bt + 4 * n;
            for (size_t q = 0; q < n; ++q) {
                grad1[pl * n + q] = bt_mu1[q] + 2.0 * xp[q] * bt_e11[q] + yp[q] * bt_e12[q];
                if (grad2)
                    grad2[pl * n + q] = bt_mu2[q] + 2.0 * yp[q] * bt_e22[q] + xp[q] * bt_e12[q];
            }
        }
    }
    free(stats); free(g); free(bt);
    return rc ? -1 : 0;
}

/* Window statistics of one 3D output voxel (k, i, j), from the definition. */
static void voxel_stats3d(const double *x, const double *y, int D, int H, int W, int off,
                          const double w[TAPS], int k, int i, int j, double s[5])
{
    for (int t = 0; t < 5; ++t) s[t] = 0.0;
    for (int c = 0; c < TAPS; ++c) {
        const int z = k + c - off;
        if (z < 0 || z >= D) continue;
        for (int a = 0; a < TAPS; ++a) {
            const int r = i + a - off;
            if (r < 0 || r >= H) continue;
            for (int b = 0; b < TAPS; ++b) {
                const int u = j + b - off;
                if (u < 0 || u >= W) continue;
                const double wt = w[c] * w[a] * w[b];
                const size_t at = ((size_t)z * H + r) * W + u;
                const double xv = x[at], yv = y[at];
                s[0] += wt * xv;
                s[1] += wt * yv;
                s[2] += wt * (xv * xv);
                s[3] += wt * (yv * yv);
                s[4] += wt * (xv * yv);
            }
        }
    }
}

/* S at the given output voxels only: idx[t] is a flat index into the NCDHW
 * output domain [N][C][Do][Ho][Wo]; out[t] = S there, the same direct
 * 11x11x11 window sums as oracle_ssim3d.  For volumes too large for the whole
 * map. */
int oracle_ssim3d_map_at(const double *x, const double *y, int N, int C, int D, int H, int W,
                         int padding, long long count, const long long *idx, double *out)
{
    if (!x || !y || !idx || !out || count < 0 || check3d(N, C, D, H, W, padding)) return -1;
    const int Do = oracle_out_extent(D, padding), Ho = oracle_out_extent(H, padding),
              Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    const size_t n = (size_t)D * H * W;
    const long long m = (long long)Do * Ho * Wo;
    double w[TAPS];
    oracle_gauss_window(w);
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (long long t = 0; t < count; ++t) {
        const long long f = idx[t];
        if (f < 0 || f >= (long long)N * C * m) {
            bad = 1;
            continue;
        }
        const size_t pl = (size_t)(f / m);
        const long long rem = f % m;
        const int pk = (int)(rem / ((long long)Ho * Wo));
        const int pi = (int)((rem / Wo) % Ho), pj = (int)(rem % Wo);
        double st[5];
        voxel_stats3d(x + pl * n, y + pl * n, D, H, W, off, w, pk, pi, pj, st);
        out[t] = ssim_point(st[0], st[1], st[2], st[3], st[4], NULL);
    }
    return bad ? -1 : 0;
}

/* 3D counterpart of oracle_ssim2d_grad_at; idx[t] is a flat NCDHW index. */
int oracle_ssim3d_grad_at(const double *x, const double *y, const double *dL, int N, int C,
                          int D, int H, int W, int padding, long long count,
                          const long long *idx, double *g1, double *g2)
{
    if (!x || !y || !dL || !idx || !g1 || count < 0 || check3d(N, C, D, H, W, padding))
        return -1;
    const int Do = oracle_out_extent(D, padding), Ho = oracle_out_extent(H, padding),
              Wo = oracle_out_extent(W, padding);
    const int off = window_offset(padding);
    const size_t n = (size_t)D * H * W;
    double w[TAPS];
    oracle_gauss_window(w);
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (long long t = 0; t < count; ++t) {
        const long long f = idx[t];
        if (f < 0 || f >= (long long)N * C * (long long)n) {
            bad = 1;
            continue;
        }
        const size_t pl = (size_t)(f / (long long)n);
        const long long rem = f % (long long)n;
        const int qk = (int)(rem / ((long long)H * W));
        const int qi = (int)((rem / W) % H), qj = (int)(rem % W);
        const int b = (int)(pl / (size_t)C);
        const double scale = dL[b] / ((double)C * (double)Do * (double)Ho * (double)Wo);
        const double *xp = x + pl * n, *yp = y + pl * n;
        double bt[5] = {0, 0, 0, 0, 0};
        for (int c = 0; c < TAPS; ++c) {
            const int pk = qk - c + off;
            if (pk < 0 || pk >= Do) continue;
            for (int a = 0; a < TAPS; ++a) {
                const int pi = qi - a + off;
                if (pi < 0 || pi >= Ho) continue;
                for (int bb = 0; bb < TAPS; ++bb) {
                    const int pj = qj - bb + off;
                    if (pj < 0 || pj >= Wo) continue;
                    double s[5], d[5];
                    voxel_stats3d(xp, yp, D, H, W, off, w, pk, pi, pj, s);
                    ssim_point(s[0], s[1], s[2], s[3], s[4], d);
                    for (int m = 0; m < 5; ++m) bt[m] += w[c] * w[a] * w[bb] * (scale * d[m]);
                }
            }
        }
        const size_t at = ((size_t)qk * H + qi) * W + qj;
        const double xv = xp[at], yv = yp[at];
        g1[t] = bt[0] + 2.0 * xv * bt[2] + yv * bt[4];
        if (g2) g2[t] = bt[1] + 2.0 * yv * bt[3] + xv * bt[4];
    }
    return bad ? -1 : 0;
}

/* SSIM and its five partial derivatives at given raw moments, exposed so the
 * tests can check the derivative formulas on their own. */
double oracle_ssim_point(double mu1, double mu2, double e11, double e22, double e12,
                         double *d5)
{
    return ssim_point(mu1, mu2, e11, e22, e12, d5);
}

/* ------------------------------------------- per-octave SSIM maps (pyramid) */

/* One octave down: out(i, j) is the mean of the pixels of the 2x2 block
 * (2i .. 2i+1, 2j .. 2j+1) that lie inside the H x W plane, so out is
 * ceil(H/2) x ceil(W/2) and a ragged last row or column averages the one or two
 * pixels it has.  (The ssimulacra2 hand-off page names a 2x downscale between
 * octaves without a formula; this is the plain box mean.) */
int oracle_downscale2x(const double *f, int H, int W, double *out)
{
    if (!f || !out || H < 1 || W < 1) return -1;
    const int Hd = (H + 1) / 2, Wd = (W + 1) / 2;
    for (int i = 0; i < Hd; ++i) {
        for (int j = 0; j < Wd; ++j) {
            double acc = 0.0;
            int cnt = 0;
            for (int a = 0; a < 2; ++a) {
                const int r = 2 * i + a;
                if (r >= H) continue;
                for (int b = 0; b < 2; ++b) {
                    const int c = 2 * j + b;
                    if (c >= W) continue;
                    acc += f[(size_t)r * W + c];
                    ++cnt;
                }
            }
            out[(size_t)i * Wd + j] = acc / (double)cnt;
        }
    }
    return 0;
}

/* The SSIM map split into its two factors, S = l * cs with
 *   l  = (2 mu1 mu2 + C1) / (mu1^2 + mu2^2 + C1)        (luminance)
 *   cs = (2 sigma12 + C2) / (sigma11 + sigma22 + C2)    (contrast-structure),
 * from the same five blurred moments as oracle_ssim2d.  Maps (each N*C*Ho*Wo,
 * any may be NULL) receive l, cs and S; means (3*N, or NULL) receives the
 * per-image means of l, cs and S over channels and output pixels, in that
 * order (means[0..N) for l, [N..2N) for cs, [2N..3N) for S). */
int oracle_ssim2d_components(const double *x, const double *y, int N, int C, int H, int W,
                             int padding, double *l_map, double *cs_map, double *s_map,
                             double *means)
{
    if (!x || !y || N < 1 || C < 1 || check_extent(H, padding) || check_extent(W, padding))
        return -1;
    const double C1 = c1_const(), C2 = c2_const();
    const size_t n = (size_t)H * W;
    const size_t no = (size_t)oracle_out_extent(H, padding) * oracle_out_extent(W, padding);
    double *stats = malloc(5 * no * sizeof(double));
    if (!stats) return -1;
    for (int b = 0; b < N; ++b) {
        double tl = 0.0, tcs = 0.0, ts = 0.0;
        for (int c = 0; c < C; ++c) {
            const size_t pl = (size_t)b * C + c;
            if (plane_stats2d(x + pl * n, y + pl * n, H, W, padding, stats)) {
                free(stats);
                return -1;
            }
            for (size_t p = 0; p < no; ++p) {
                const double mu1 = stats[p], mu2 = stats[no + p];
                const double s11 = stats[2 * no + p] - mu1 * mu1;
                const double s22 = stats[3 * no + p] - mu2 * mu2;
                const double s12 = stats[4 * no + p] - mu1 * mu2;
                const double l = (2.0 * mu1 * mu2 + C1) / (mu1 * mu1 + mu2 * mu2 + C1);
                const double cs = (2.0 * s12 + C2) / (s11 + s22 + C2);
                const double S = l * cs;
                if (l_map) l_map[pl * no + p] = l;
                if (cs_map) cs_map[pl * no + p] = cs;
                if (s_map) s_map[pl * no + p] = S;
                tl += l;
                tcs += cs;
                ts += S;
            }
        }
        if (means) {
            const double cnt = (double)C * (double)no;
            means[b] = tl / cnt;
            means[N + b] = tcs / cnt;
            means[2 * N + b] = ts / cnt;
        }
    }
    free(stats);
    return 0;
}
