/*
 * kfac_oracle.c -- plain, slow, double-precision CPU oracle for the K-FAC
 * curvature step.  TEST INFRASTRUCTURE ONLY: the product path (the CUDA
 * library under second_order_optimisation_gb300/) never calls, links or
 * loads this file, and this file shares no code, header or constant with it.
 *
 * Source: Osawa, Tsuji, Ueno, Naruse, Yokota, Matsuoka, "Large-Scale
 * Distributed Second-Order Optimization Using Kronecker-Factored Approximate
 * Curvature for Deep Convolutional Neural Networks" (cited below as
 * "Osawa et al.").  Section/equation numbers are the paper's.
 *
 * What the paper fixes and what is a reading of it:
 *   - E[.] is the mean over the samples of the mini-batch (section 3.1, Eq. 1).
 *   - The curvature is block diagonal over layers (section 3.2, Eq. 4) and
 *     each block is the Kronecker product G (x) A, A built from the layer's
 *     input activations, G from the gradients of the layer's output
 *     (section 3.2, Eq. 5).
 *   - The inverse of the Kronecker product is the Kronecker product of the
 *     inverses (section 3.2, Eq. 6), so the preconditioned gradient of a
 *     weight matrix grad[dG x dA] is G^-1 grad A^-1 (section 3.2, Eq. 7).
 *   - The BatchNorm Fisher is taken as diagonal (section 1, contributions).
 *   Readings (the paper is silent; see the repository's design notes):
 *   - convolution rows: every output position of every sample is one row of
 *     the patch matrix P (im2col), zero padding outside the image, column
 *     index (r*kw + s)*C_in + c; an FC bias is a trailing column of ones;
 *   - the factor statistic is the mean over the M rows: Fhat = P^T P / M;
 *   - running average F <- xi*F + (1-xi)*Fhat, starting from F = I;
 *   - damping split by pi = sqrt((tr A/dA)/(tr G/dG)):
 *     dA_damp = pi*sqrt(gamma), dG_damp = sqrt(gamma)/pi;
 *   - inverse via Cholesky F = U^T U, then U^-1, then U^-1 U^-T;
 *   - BN: F_c = mean_i x_ic^2, g_c = mean_i x_ic, out_c = g_c/(F_c + gamma).
 *
 * All arrays are row-major doubles.  Functions return 0 on success.
 * Parity status of every function is stated in its comment; all are pinned
 * by the CPU tests (closed forms, brute force, library special cases).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- threads */

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ----------------------------------------------------------------- im2col */

/* Output spatial extent of a convolution along one axis. */
static long out_extent(long in, long k, long stride, long pad)
{
    return (in + 2 * pad - k) / stride + 1;
}

/*
 * Patch matrix of a convolution layer (the layer input whose outer product
 * gives A in Osawa et al. section 3.2, Eq. 5; reading: im2col rows).
 *   x  : NHWC input [n][h][w][c]
 *   P  : [M][d], M = n*Ho*Wo, d = kh*kw*c (+1 when append_one)
 *   row m = (img*Ho + ho)*Wo + wo,
 *   P[m][(r*kw + s)*c + ch] = x[img][ho*sh - ph + r][wo*sw - pw + s][ch],
 *   zero outside the image; P[m][d-1] = 1 when append_one (bias column).
 * A fully connected layer is the case h = w = kh = kw = 1.
 * Pinned: conv output P*W^T equals a library direct convolution (tests).
 */
int orc_im2col(const double *x, long n, long h, long w, long c,
               long kh, long kw, long sh, long sw, long ph, long pw,
               int append_one, double *P)
{
    long Ho = out_extent(h, kh, sh, ph), Wo = out_extent(w, kw, sw, pw);
    if (Ho <= 0 || Wo <= 0) return 1;
    long d = kh * kw * c + (append_one ? 1 : 0);
    for (long img = 0; img < n; ++img)
        for (long ho = 0; ho < Ho; ++ho)
            for (long wo = 0; wo < Wo; ++wo) {
                long m = (img * Ho + ho) * Wo + wo;
                double *row = P + m * d;
                for (long r = 0; r < kh; ++r)
                    for (long s = 0; s < kw; ++s) {
                        long hi = ho * sh - ph + r, wi = wo * sw - pw + s;
                        int inside = hi >= 0 && hi < h && wi >= 0 && wi < w;
                        for (long ch = 0; ch < c; ++ch)
                            row[(r * kw + s) * c + ch] =
                                inside ? x[((img * h + hi) * w + wi) * c + ch] : 0.0;
                    }
                if (append_one) row[d - 1] = 1.0;
            }
    return 0;
}

/* ------------------------------------------------------ factor statistics */

/*
 * S = P^T P (full symmetric d x d), the un-normalised Kronecker-factor
 * statistic (Osawa et al. section 3.2, Eq. 5).  Each entry is accumulated
 * over m = 0..M-1 in order; the lower triangle is copied from the upper so
 * that S is exactly symmetric.
 * Pinned: brute force over tiny convolutions; rank one at batch size one.
 */
int orc_gram(const double *P, long M, long d, double *S)
{
    double *Pt = (double *)malloc(sizeof(double) * (size_t)(M * d));
    if (!Pt) return 2;
    for (long m = 0; m < M; ++m)
        for (long i = 0; i < d; ++i) Pt[i * M + m] = P[m * d + i];
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < d; ++i) {
        const double *pi = Pt + i * M;
        for (long j = i; j < d; ++j) {
            const double *pj = Pt + j * M;
            double acc = 0.0;
            for (long m = 0; m < M; ++m) acc += pi[m] * pj[m];
            S[i * d + j] = acc;
        }
    }
    for (long i = 0; i < d; ++i)
        for (long j = 0; j < i; ++j) S[i * d + j] = S[j * d + i];
    free(Pt);
    return 0;
}

/*
 * One running-average update of a Kronecker factor with the mean statistic
 * of M rows: F <- xi*F + (1 - xi) * (P^T P)/M  (reading: the paper is silent
 * on the running average; xi = 0 gives the plain statistic of Eq. 5).
 * F is a full symmetric d x d matrix, updated in place.
 * Pinned: closed form xi^k F0 + (1 - xi^k) Fhat after k equal updates.
 */
int orc_factor_ema(double *F, const double *P, long M, long d, double xi)
{
    double *S = (double *)malloc(sizeof(double) * (size_t)(d * d));
    if (!S) return 2;
    int rc = orc_gram(P, M, d, S);
    if (rc) { free(S); return rc; }
    for (long k = 0; k < d * d; ++k) F[k] = xi * F[k] + (1.0 - xi) * S[k] / (double)M;
    free(S);
    return 0;
}

/*
 * Selected entries of the un-normalised statistic of a convolution layer,
 * computed straight from the layer input without forming P:
 *   out[t] = sum_m P[m][ii[t]] * P[m][jj[t]]  (m in order),
 * with P defined as in orc_im2col.  Used for sampled checks at sizes where
 * the full statistic is too slow on the CPU.
 * Pinned: equals the corresponding entries of orc_gram(orc_im2col(x)).
 */
int orc_gram_entries(const double *x, long n, long h, long w, long c,
                     long kh, long kw, long sh, long sw, long ph, long pw,
                     int append_one, const long *ii, const long *jj, long T,
                     double *out)
{
    long Ho = out_extent(h, kh, sh, ph), Wo = out_extent(w, kw, sw, pw);
    if (Ho <= 0 || Wo <= 0) return 1;
    long dcore = kh * kw * c;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < T; ++t) {
        long col[2] = {ii[t], jj[t]};
        long r[2], s[2], ch[2];
        int one[2];
        for (int q = 0; q < 2; ++q) {
            one[q] = append_one && col[q] == dcore;
            long rs = one[q] ? 0 : col[q] / c;
            ch[q] = one[q] ? 0 : col[q] % c;
            r[q] = rs / kw;
            s[q] = rs % kw;
        }
        double acc = 0.0;
        for (long img = 0; img < n; ++img)
            for (long ho = 0; ho < Ho; ++ho)
                for (long wo = 0; wo < Wo; ++wo) {
                    double v[2];
                    for (int q = 0; q < 2; ++q) {
                        if (one[q]) { v[q] = 1.0; continue; }
                        long hi = ho * sh - ph + r[q], wi = wo * sw - pw + s[q];
                        v[q] = (hi >= 0 && hi < h && wi >= 0 && wi < w)
                                   ? x[((img * h + hi) * w + wi) * c + ch[q]] : 0.0;
                    }
                    acc += v[0] * v[1];
                }
        out[t] = acc;
    }
    return 0;
}

/*
 * Weight gradient of a layer from its patch matrix and output gradients:
 *   grad[dG][dA] = Gam^T P / nsamples,
 * Gam = output gradients [M][dG] with the same row order as P.  (Reading: the
 * loss is a mean over samples, Osawa et al. Eq. 1, and the gradients are
 * taken as given per row, so the sum over positions is divided by the sample
 * count only.)
 * Pinned: equals the autograd weight gradient of a library convolution.
 */
int orc_weight_grad(const double *P, const double *Gam, long M, long dA, long dG,
                    long nsamples, double *grad)
{
#pragma omp parallel for schedule(static)
    for (long o = 0; o < dG; ++o)
        for (long i = 0; i < dA; ++i) {
            double acc = 0.0;
            for (long m = 0; m < M; ++m) acc += Gam[m * dG + o] * P[m * dA + i];
            grad[o * dA + i] = acc / (double)nsamples;
        }
    return 0;
}

/* --------------------------------------------------------------- damping */

/*
 * Damping split by pi (reading; the paper states no damping scheme):
 *   pi = sqrt((tr A / dA) / (tr G / dG)),
 *   damp_A = pi * sqrt(gamma), damp_G = sqrt(gamma) / pi,
 * so that damp_A * damp_G = gamma.  With pi_split = 0 both are sqrt(gamma).
 * Pinned: the explicit expansion (A+dA I)(x)(G+dG I) and invariance of the
 * damped Kronecker product under A -> cA, G -> G/c.
 */
int orc_pi_damping(const double *A, long dA, const double *G, long dG,
                   double gamma, int pi_split, double *damp_A, double *damp_G)
{
    double sg = sqrt(gamma);
    if (!pi_split) { *damp_A = sg; *damp_G = sg; return 0; }
    double trA = 0.0, trG = 0.0;
    for (long i = 0; i < dA; ++i) trA += A[i * dA + i];
    for (long i = 0; i < dG; ++i) trG += G[i * dG + i];
    double pi = sqrt((trA / (double)dA) / (trG / (double)dG));
    *damp_A = pi * sg;
    *damp_G = sg / pi;
    return 0;
}

/* ------------------------------------------------------------- inversion */

/*
 * Cholesky factor of an SPD matrix, upper form A = U^T U, right-looking,
 * in place on the upper triangle (the lower triangle is set to zero).
 * Returns 0, or k+1 when the k-th pivot is not positive (A not PD).
 * Pinned: matches a library Cholesky (transposed lower factor).
 */
int orc_cholesky_upper(double *A, long n)
{
    for (long k = 0; k < n; ++k) {
        double p = A[k * n + k];
        if (!(p > 0.0)) return (int)(k + 1);
        p = sqrt(p);
        A[k * n + k] = p;
        for (long j = k + 1; j < n; ++j) A[k * n + j] /= p;
#pragma omp parallel for schedule(static) if (n - k > 256)
        for (long i = k + 1; i < n; ++i) {
            double uki = A[k * n + i];
            for (long j = i; j < n; ++j) A[i * n + j] -= uki * A[k * n + j];
        }
    }
    for (long i = 0; i < n; ++i)
        for (long j = 0; j < i; ++j) A[i * n + j] = 0.0;
    return 0;
}

/*
 * Inverse of an upper-triangular matrix, in place (column-by-column back
 * substitution of U X = I).  Pinned: U * U^-1 = I.
 */
int orc_trtri_upper(double *U, long n)
{
    double *X = (double *)calloc((size_t)(n * n), sizeof(double));
    if (!X) return 2;
#pragma omp parallel for schedule(dynamic, 4) if (n > 256)
    for (long j = 0; j < n; ++j) {
        X[j * n + j] = 1.0 / U[j * n + j];
        for (long i = j - 1; i >= 0; --i) {
            double acc = 0.0;
            for (long k = i + 1; k <= j; ++k) acc += U[i * n + k] * X[k * n + j];
            X[i * n + j] = -acc / U[i * n + i];
        }
    }
    memcpy(U, X, sizeof(double) * (size_t)(n * n));
    free(X);
    return 0;
}

/*
 * Product V V^T of an upper-triangular V (here V = U^-1), written as a full
 * symmetric matrix: (U^T U)^-1 = U^-1 U^-T.  Pinned: inverse check.
 */
int orc_lauum_upper(const double *V, long n, double *out)
{
#pragma omp parallel for schedule(dynamic, 4) if (n > 256)
    for (long i = 0; i < n; ++i)
        for (long j = i; j < n; ++j) {
            double acc = 0.0;
            for (long k = j; k < n; ++k) acc += V[i * n + k] * V[j * n + k];
            out[i * n + j] = acc;
            out[j * n + i] = acc;
        }
    return 0;
}

/*
 * Damped inverse (F + damp I)^-1 of a symmetric factor (Osawa et al.
 * section 3.2, Eq. 6, with the damping reading above), by Cholesky,
 * triangular inverse and the U^-1 U^-T product.  F is full symmetric.
 * Returns 0 or the 1-based index of the first non-positive pivot.
 */
int orc_damped_inverse(const double *F, long n, double damp, double *Finv)
{
    double *U = (double *)malloc(sizeof(double) * (size_t)(n * n));
    if (!U) return -2;
    memcpy(U, F, sizeof(double) * (size_t)(n * n));
    for (long i = 0; i < n; ++i) U[i * n + i] += damp;
    int info = orc_cholesky_upper(U, n);
    if (info) { free(U); return info; }
    orc_trtri_upper(U, n);
    orc_lauum_upper(U, n, Finv);
    free(U);
    return 0;
}

/* -------------------------------------------------------- preconditioning */

/*
 * Preconditioned gradient of one layer (Osawa et al. section 3.2, Eq. 6-7):
 *   out[dG][dA] = Ginv * grad * Ainv,
 * the row-major form of (G (x) A)^-1 vec(grad) for symmetric A and G.
 * Evaluated as Ginv * (grad * Ainv), plain triple loops.
 * Pinned: explicit Kronecker solve on tiny factors.
 */
int orc_precondition(const double *Ginv, long dG, const double *grad, long dA,
                     const double *Ainv, double *out)
{
    double *T = (double *)malloc(sizeof(double) * (size_t)(dG * dA));
    if (!T) return 2;
#pragma omp parallel for schedule(static)
    for (long o = 0; o < dG; ++o)
        for (long j = 0; j < dA; ++j) {
            double acc = 0.0;
            for (long k = 0; k < dA; ++k) acc += grad[o * dA + k] * Ainv[k * dA + j];
            T[o * dA + j] = acc;
        }
#pragma omp parallel for schedule(static)
    for (long o = 0; o < dG; ++o)
        for (long j = 0; j < dA; ++j) {
            double acc = 0.0;
            for (long k = 0; k < dG; ++k) acc += Ginv[o * dG + k] * T[k * dA + j];
            out[o * dA + j] = acc;
        }
    free(T);
    return 0;
}

/*
 * Selected rows of the preconditioned gradient (Eq. 7 as above), for checks
 * at sizes where the full product is too slow on the CPU:
 *   out[t][j] = sum_o Ginv[rows[t]][o] * sum_k grad[o][k] * Ainv[k][j],
 * evaluated as (Ginv[rows[t]] * grad) * Ainv, plain loops.
 * Pinned: equals the corresponding rows of orc_precondition.
 */
int orc_precondition_rows(const double *Ginv, long dG, const double *grad, long dA,
                          const double *Ainv, const long *rows, long nrows, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nrows; ++t) {
        double *u = (double *)malloc(sizeof(double) * (size_t)dA);
        const double *g = Ginv + rows[t] * dG;
        for (long k = 0; k < dA; ++k) u[k] = 0.0;
        for (long o = 0; o < dG; ++o) {
            const double go = g[o];
            for (long k = 0; k < dA; ++k) u[k] += go * grad[o * dA + k];
        }
        for (long j = 0; j < dA; ++j) out[t * dA + j] = 0.0;
        for (long k = 0; k < dA; ++k) {
            const double uk = u[k];
            for (long j = 0; j < dA; ++j) out[t * dA + j] += uk * Ainv[k * dA + j];
        }
        free(u);
    }
    return 0;
}

/*
 * Weight update with the preconditioned gradient (Osawa et al. section 3.2,
 * Eq. 8: w <- w - eta * G, G the natural gradient of Eq. 7):
 *   w[o][j] <- w[o][j] - eta * P[o][j].
 * Pinned: eta = 0 leaves w unchanged; w = 0, eta = 1 gives -P; linearity in eta.
 */
int orc_weight_update(double *w, const double *P, long dG, long dA, double eta)
{
    for (long o = 0; o < dG; ++o)
        for (long j = 0; j < dA; ++j) w[o * dA + j] -= eta * P[o * dA + j];
    return 0;
}

/*
 * Packed storage of a symmetric factor (section 1, contributions: the
 * symmetry of the Kronecker factors is exploited to reduce overhead).
 * Reading: the upper triangle is kept row after row, row i holding the
 * entries j = i .. d-1, so that entry (i, j), i <= j, sits at position
 * i*d - i*(i+1)/2 + j of the d(d+1)/2 stored values.  pack reads the upper
 * triangle of F [d][d]; unpack writes both triangles.
 */
int orc_pack_upper(const double *F, long d, double *out)
{
    long t = 0;
    for (long i = 0; i < d; ++i)
        for (long j = i; j < d; ++j) out[t++] = F[i * d + j];
    return 0;
}

int orc_unpack_upper(const double *Fp, long d, double *F)
{
    long t = 0;
    for (long i = 0; i < d; ++i)
        for (long j = i; j < d; ++j) {
            F[i * d + j] = Fp[t];
            F[j * d + i] = Fp[t];
            ++t;
        }
    return 0;
}

/*
 * Steps of the stale-factor schedule (Osawa et al. section 1: after a few
 * hundred iterations the Fisher matrix need not be refreshed every step):
 * step t (0-based) refreshes the factors and their inverses when
 * t < warmup, or when (t - warmup) is a multiple of every; other steps
 * precondition with the inverses of the last refresh.
 * Pinned: every = 1 refreshes every step; warmup >= steps refreshes every
 * step; the count of refreshes over T steps has a closed form.
 */
int orc_is_refresh_step(long t, long warmup, long every)
{
    if (every < 1) return 1;
    if (t < warmup) return 1;
    return (t - warmup) % every == 0;
}

/* -------------------------------------------------------------- BatchNorm */

/*
 * Diagonal Fisher of a BatchNorm parameter vector (Osawa et al. section 1:
 * the BN Fisher is approximated as diagonal) from per-sample gradients
 * x[ns][C]:
 *   F_c    = xi*F_c + (1 - xi) * mean_i x_ic^2   (xi = 0: plain mean),
 *   gmean_c = mean_i x_ic                        (the mini-batch gradient),
 *   out_c   = gmean_c / (F_c + gamma)            (damped diagonal solve).
 * Pinned: diagonal of the explicit per-sample outer-product Fisher; constant
 * input closed form.
 */
int orc_bn_diag_fisher(const double *x, long ns, long C, double gamma, double xi,
                       double *F, double *gmean, double *out)
{
    for (long c = 0; c < C; ++c) {
        double s = 0.0, s2 = 0.0;
        for (long i = 0; i < ns; ++i) {
            double v = x[i * C + c];
            s += v;
            s2 += v * v;
        }
        double f = s2 / (double)ns;
        F[c] = xi * F[c] + (1.0 - xi) * f;
        gmean[c] = s / (double)ns;
        out[c] = gmean[c] / (F[c] + gamma);
    }
    return 0;
}
