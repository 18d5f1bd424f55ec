/*
 * oracle.c -- plain, slow, fp64 CPU reference for RMSNorm and LayerNorm,
 * forward and backward, over the contiguous last dimension of a row-major
 * [M, N] tensor.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes follows the page "PyTorch atinge desempenho SOTA em
 * normalizacao com torch.compile" (matsubara.tec.br):
 *   - its paragraph on LayerNorm (2016) and RMSNorm (2019): LayerNorm
 *     normalises with the mean and the variance along one dimension and then
 *     applies the trainable gamma (weight) and beta (bias); RMSNorm replaces
 *     the mean/variance by the root mean square and has no beta;
 *   - its paragraph on the forward pass: a reduction along a contiguous
 *     dimension followed by pointwise operations;
 *   - its paragraph on the backward pass: the gradients dX (input), dW
 *     (gamma) and, for LayerNorm, dB (beta).
 * The page prints no formula.  The plainest textbook reading is used and is
 * written out once here (all arithmetic in double):
 *
 *   LayerNorm   mu = (1/N) sum_j x_j
 *               v  = (1/N) sum_j (x_j - mu)^2          (population variance)
 *               r  = 1 / sqrt(v + eps)                  (eps inside the root)
 *               xhat_j = (x_j - mu) * r
 *               y_j = xhat_j * gamma_j + beta_j
 *   RMSNorm     ms = (1/N) sum_j x_j^2
 *               r  = 1 / sqrt(ms + eps)
 *               xhat_j = x_j * r
 *               y_j = xhat_j * gamma_j
 *   Backward    g_j = dy_j * gamma_j
 *               c = (1/N) sum_j g_j * xhat_j
 *               a = (1/N) sum_j g_j                     (LayerNorm only)
 *               LayerNorm dx_j = r * (g_j - a - xhat_j * c)
 *               RMSNorm   dx_j = r * (g_j - xhat_j * c)
 *               dgamma_j = sum over rows of dy_ij * xhat_ij
 *               dbeta_j  = sum over rows of dy_ij        (LayerNorm only)
 *
 * The backward formulas are the derivative of y with respect to x, gamma and
 * beta under the forward definition above (chain rule through mu and r);
 * the tests pin them to central finite differences of the forward.
 *
 * Every statistic is recomputed here in double from the inputs; nothing
 * saved by another implementation is reused.  bf16 inputs are widened
 * exactly (bf16 is the top half of an IEEE binary32).
 *
 * Fused residual add + norm (the "fusion with surrounding operations" that
 * the same page and the kernel-fusion paragraph of "Otimizacao de
 * Performance de GPU" credit): the residual stream is updated and
 * normalised in one pass,
 *   h = bf16(x + r)        (the sum is formed in binary32, then rounded to
 *                           nearest-even bf16: h is a stored tensor, and the
 *                           oracle takes that rounding decision exactly as
 *                           the kernels do)
 *   y = norm(h)            (the definitions above, on the bf16 values of h)
 * and its backward adds the gradient dh that reaches h through the residual
 * path:  dx = dr = (norm backward of dy at h) + dh.
 *
 * FP8 output (the page "Otimizacao de Performance de GPU", introl.com, in
 * its December 2025 update, reports FP8 training as production ready on
 * Blackwell; it gives no format or scaling, so the plainest readings are
 * used).  y is quantised to E4M3 (the OCP 8-bit floating point format
 * "E4M3FN": 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite 448, subnormals m/8 * 2^-6)
 * with round to nearest, ties to even, and saturation to +-448.  Two
 * scalings:
 *   per row     s_i = amax_i / 448, q_ij = E4M3(y_ij / s_i), computed as
 *               (y_ij / amax_i) * 448 so that the row maximum maps to 448
 *               exactly; a row of zeros has s_i = 1.
 *   MX blocks   blocks of 32 consecutive columns share a power-of-two
 *               scale X = 2^e, e = floor(log2(amax_block)) - 8 (8 being the
 *               largest E4M3 exponent), clamped below at -127, stored as an
 *               E8M0 byte e + 127; q = E4M3(y / X).  This is the conversion
 *               rule of the OCP Microscaling Formats (MX) v1.0
 *               specification, section 6.3; the scaled block maximum lies
 *               in [256, 512), and values from 448 up saturate.
 * The value rounded to E4M3 is formed in fp64: exactly for MX (division by
 * a power of two), within 2^-52 relative for per-row scaling.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_RMS 0
#define ORACLE_LAYER 1

/* bf16 bit pattern -> exact double value. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void widen_row(const uint16_t *src, int64_t n, double *dst)
{
    for (int64_t j = 0; j < n; ++j)
        dst[j] = bf16_bits_to_double(src[j]);
}

/* Row statistics: *mu receives the mean (0 for RMSNorm), *r the reciprocal
 * of sqrt(variance-or-mean-square + eps). */
static void row_stats(const double *x, int64_t n, double eps, int mode,
                      double *mu, double *r)
{
    if (mode == ORACLE_LAYER) {
        double s = 0.0;
        for (int64_t j = 0; j < n; ++j)
            s += x[j];
        double m = s / (double)n;
        double q = 0.0;
        for (int64_t j = 0; j < n; ++j)
            q += (x[j] - m) * (x[j] - m);
        double v = q / (double)n;
        *mu = m;
        *r = 1.0 / sqrt(v + eps);
    } else {
        double q = 0.0;
        for (int64_t j = 0; j < n; ++j)
            q += x[j] * x[j];
        double ms = q / (double)n;
        *mu = 0.0;
        *r = 1.0 / sqrt(ms + eps);
    }
}

/* Forward of one row.  beta may be NULL (treated as zero). */
static void fwd_row(const double *x, const double *gamma, const double *beta,
                    int64_t n, double eps, int mode,
                    double *y, double *mu_out, double *r_out)
{
    double mu, r;
    row_stats(x, n, eps, mode, &mu, &r);
    for (int64_t j = 0; j < n; ++j) {
        double xhat = (x[j] - mu) * r;
        double b = (mode == ORACLE_LAYER && beta) ? beta[j] : 0.0;
        y[j] = xhat * gamma[j] + b;
    }
    if (mu_out)
        *mu_out = mu;
    if (r_out)
        *r_out = r;
}

/* Backward of one row: writes dx (if non-NULL) and adds this row's
 * contribution to dgamma / dbeta (if non-NULL). The *_abs arrays, if given,
 * accumulate the sums of absolute summands (used as tolerance scales). */
static void bwd_row(const double *dy, const double *x, const double *gamma,
                    int64_t n, double eps, int mode, double *dx,
                    double *dgamma, double *dbeta,
                    double *dgamma_abs, double *dbeta_abs)
{
    double mu, r;
    row_stats(x, n, eps, mode, &mu, &r);
    double sum_g = 0.0, sum_gxhat = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double xhat = (x[j] - mu) * r;
        double g = dy[j] * gamma[j];
        sum_g += g;
        sum_gxhat += g * xhat;
    }
    double a = (mode == ORACLE_LAYER) ? sum_g / (double)n : 0.0;
    double c = sum_gxhat / (double)n;
    for (int64_t j = 0; j < n; ++j) {
        double xhat = (x[j] - mu) * r;
        double g = dy[j] * gamma[j];
        if (dx)
            dx[j] = r * (g - a - xhat * c);
        if (dgamma)
            dgamma[j] += dy[j] * xhat;
        if (dgamma_abs)
            dgamma_abs[j] += fabs(dy[j] * xhat);
        if (mode == ORACLE_LAYER) {
            if (dbeta)
                dbeta[j] += dy[j];
            if (dbeta_abs)
                dbeta_abs[j] += fabs(dy[j]);
        }
    }
}

/* binary32 -> bf16 bit pattern, round to nearest, ties to even (NaN kept
 * quiet).  Written from the definition: add half an ulp of bf16 (0x7FFF)
 * plus the parity of the kept low bit, then truncate. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* h = bf16(x + r) over n elements, the sum formed in binary32. */
static void residual_add_row(const uint16_t *x, const uint16_t *r, int64_t n,
                             uint16_t *h)
{
    for (int64_t j = 0; j < n; ++j) {
        float a = (float)bf16_bits_to_double(x[j]);
        float b = (float)bf16_bits_to_double(r[j]);
        float s = a + b;
        h[j] = float_to_bf16_rne(s);
    }
}

/* ---------------------------------------------------------------- f64 API */

/* Forward over all M rows of double inputs.  y: [M, N]; rstd, mean: [M]
 * (mean may be NULL).  Returns 0, or -1 on bad arguments. */
int oracle_fwd_f64(const double *x, const double *gamma, const double *beta,
                   int64_t M, int64_t N, double eps, int mode,
                   double *y, double *rstd, double *mean)
{
    if (!x || !gamma || !y || M < 0 || N < 1)
        return -1;
    for (int64_t i = 0; i < M; ++i) {
        double mu, r;
        fwd_row(x + i * N, gamma, beta, N, eps, mode, y + i * N, &mu, &r);
        if (rstd)
            rstd[i] = r;
        if (mean)
            mean[i] = mu;
    }
    return 0;
}

/* Backward over all M rows of double inputs.  dx: [M, N]; dgamma, dbeta:
 * [N], overwritten (dbeta may be NULL).  Returns 0, or -1. */
int oracle_bwd_f64(const double *dy, const double *x, const double *gamma,
                   int64_t M, int64_t N, double eps, int mode,
                   double *dx, double *dgamma, double *dbeta)
{
    if (!dy || !x || !gamma || M < 0 || N < 1)
        return -1;
    if (dgamma)
        memset(dgamma, 0, sizeof(double) * (size_t)N);
    if (dbeta)
        memset(dbeta, 0, sizeof(double) * (size_t)N);
    for (int64_t i = 0; i < M; ++i)
        bwd_row(dy + i * N, x + i * N, gamma, N, eps, mode,
                dx ? dx + i * N : NULL, dgamma, dbeta, NULL, NULL);
    return 0;
}

/* --------------------------------------------------------------- bf16 API */

/* Forward on bf16 inputs (bit patterns), for the rows listed in `rows`
 * (all rows 0..M-1 in order when rows == NULL, nrows == M).  Output row k
 * of y / rstd / mean belongs to input row rows[k].  Streams one row at a
 * time, so [M, N] double tensors are never formed. */
int oracle_fwd_bf16(const uint16_t *x, const uint16_t *gamma,
                    const uint16_t *beta, int64_t M, int64_t N, double eps,
                    int mode, const int64_t *rows, int64_t nrows,
                    double *y, double *rstd, double *mean)
{
    if (!x || !gamma || M < 0 || N < 1 || nrows < 0)
        return -1;
    if (!rows && nrows != M)
        return -1;
    double *xr = malloc(sizeof(double) * (size_t)N);
    double *g = malloc(sizeof(double) * (size_t)N);
    double *b = beta ? malloc(sizeof(double) * (size_t)N) : NULL;
    double *yr = y ? NULL : malloc(sizeof(double) * (size_t)N);
    if (!xr || !g || (beta && !b) || (!y && !yr)) {
        free(xr); free(g); free(b); free(yr);
        return -2;
    }
    widen_row(gamma, N, g);
    if (beta)
        widen_row(beta, N, b);
    int rc = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= M) {
            rc = -1;
            break;
        }
        widen_row(x + i * N, N, xr);
        double mu, r;
        fwd_row(xr, g, b, N, eps, mode, y ? y + k * N : yr, &mu, &r);
        if (rstd)
            rstd[k] = r;
        if (mean)
            mean[k] = mu;
    }
    free(xr); free(g); free(b); free(yr);
    return rc;
}

/* dx on bf16 inputs for the listed rows (same row convention as above). */
int oracle_bwd_dx_bf16(const uint16_t *dy, const uint16_t *x,
                       const uint16_t *gamma, int64_t M, int64_t N,
                       double eps, int mode, const int64_t *rows,
                       int64_t nrows, double *dx)
{
    if (!dy || !x || !gamma || !dx || M < 0 || N < 1 || nrows < 0)
        return -1;
    if (!rows && nrows != M)
        return -1;
    double *xr = malloc(sizeof(double) * (size_t)N);
    double *dyr = malloc(sizeof(double) * (size_t)N);
    double *g = malloc(sizeof(double) * (size_t)N);
    if (!xr || !dyr || !g) {
        free(xr); free(dyr); free(g);
        return -2;
    }
    widen_row(gamma, N, g);
    int rc = 0;
    for (int64_t k = 0; k < nrows; ++k) {
        int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= M) {
            rc = -1;
            break;
        }
        widen_row(x + i * N, N, xr);
        widen_row(dy + i * N, N, dyr);
        bwd_row(dyr, xr, g, N, eps, mode, dx + k * N, NULL, NULL, NULL, NULL);
    }
    free(xr); free(dyr); free(g);
    return rc;
}

/* Column reductions over ALL rows (in increasing row order) on bf16 inputs:
 * dgamma_j = sum_i dy_ij * xhat_ij, dbeta_j = sum_i dy_ij (LayerNorm), plus
 * the matching sums of absolute summands.  Any output pointer may be NULL.
 * gamma is needed because the per-row statistics do not depend on it but
 * the shared row routine takes it; it does not enter dgamma or dbeta. */
int oracle_param_grads_bf16(const uint16_t *dy, const uint16_t *x,
                            const uint16_t *gamma, int64_t M, int64_t N,
                            double eps, int mode, double *dgamma,
                            double *dbeta, double *dgamma_abs,
                            double *dbeta_abs)
{
    if (!dy || !x || !gamma || M < 0 || N < 1)
        return -1;
    double *xr = malloc(sizeof(double) * (size_t)N);
    double *dyr = malloc(sizeof(double) * (size_t)N);
    double *g = malloc(sizeof(double) * (size_t)N);
    if (!xr || !dyr || !g) {
        free(xr); free(dyr); free(g);
        return -2;
    }
    widen_row(gamma, N, g);
    if (dgamma) memset(dgamma, 0, sizeof(double) * (size_t)N);
    if (dbeta) memset(dbeta, 0, sizeof(double) * (size_t)N);
    if (dgamma_abs) memset(dgamma_abs, 0, sizeof(double) * (size_t)N);
    if (dbeta_abs) memset(dbeta_abs, 0, sizeof(double) * (size_t)N);
    for (int64_t i = 0; i < M; ++i) {
        widen_row(x + i * N, N, xr);
        widen_row(dy + i * N, N, dyr);
        bwd_row(dyr, xr, g, N, eps, mode, NULL, dgamma, dbeta, dgamma_abs,
                dbeta_abs);
    }
    free(xr); free(dyr); free(g);
    return 0;
}

/* ------------------------------------------------- fused residual add API */

/* h = bf16(x + r) for all M rows (bit patterns). */
int oracle_residual_add_bf16(const uint16_t *x, const uint16_t *r, int64_t M,
                             int64_t N, uint16_t *h)
{
    if (!x || !r || !h || M < 0 || N < 1)
        return -1;
    for (int64_t i = 0; i < M; ++i)
        residual_add_row(x + i * N, r + i * N, N, h + i * N);
    return 0;
}

/* dx = (norm backward of dy at h) + dh for the listed rows (row convention
 * of oracle_bwd_dx_bf16); h, dy, dh are bf16 bit patterns. */
int oracle_add_bwd_dx_bf16(const uint16_t *dy, const uint16_t *h,
                           const uint16_t *dh, const uint16_t *gamma,
                           int64_t M, int64_t N, double eps, int mode,
                           const int64_t *rows, int64_t nrows, double *dx)
{
    if (!dh)
        return -1;
    int rc = oracle_bwd_dx_bf16(dy, h, gamma, M, N, eps, mode, rows, nrows, dx);
    if (rc != 0)
        return rc;
    for (int64_t k = 0; k < nrows; ++k) {
        int64_t i = rows ? rows[k] : k;
        for (int64_t j = 0; j < N; ++j)
            dx[k * N + j] += bf16_bits_to_double(dh[i * N + j]);
    }
    return 0;
}

/* ----------------------------------------------------------- FP8 (E4M3) */

#define ORACLE_FP8_ROW 0
#define ORACLE_FP8_MX 1
#define E4M3_MAX 448.0
#define MX_BLOCK 32

/* Exact value of an E4M3 code (NaN for S.1111.111). */
static double e4m3_value(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 code to the real value v, ties to the even mantissa,
 * magnitudes from 448 up saturate to 448; NaN gives 0x7F.  The scaled
 * quantities below are exact (multiplication by powers of two), and
 * nearbyint in the default rounding mode rounds half to even. */
static uint8_t e4m3_code(double v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= E4M3_MAX)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal binade: spacing 2^-9; m == 8 is the smallest normal,
         * whose code is also 8 */
        double m = nearbyint(ldexp(a, 9));
        return sign | (uint8_t)m;
    }
    int e2;
    frexp(a, &e2);               /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;              /* floor(log2 a), in [-6, 8] */
    double m = nearbyint(ldexp(a, 3 - e));   /* in [8, 16] */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

int oracle_e4m3_encode(const double *v, int64_t n, uint8_t *out)
{
    if ((!v || !out) && n > 0)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_code(v[i]);
    return 0;
}

int oracle_e4m3_decode(const uint8_t *c, int64_t n, double *out)
{
    if ((!c || !out) && n > 0)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_value(c[i]);
    return 0;
}

/* Forward with E4M3 output for the listed rows (row convention of
 * oracle_fwd_bf16).  With r non-NULL the row is first h = bf16(x + r).
 * Outputs per listed row k:
 *   y[k*N + j]   the exact fp64 forward output;
 *   q[k*N + j]   its E4M3 code under the scaling;
 *   per row:     amax[k], scale[k] = amax/448 (1 for a zero row);
 *   MX:          amax[k*nb + b], scale[k*nb + b] = 2^e, ebyte[k*nb + b] =
 *                e + 127, with nb = N / 32 (N must be a multiple of 32).
 * ebyte may be NULL; it is ignored for per-row scaling. */
int oracle_fwd_fp8_bf16(const uint16_t *x, const uint16_t *r,
                        const uint16_t *gamma, const uint16_t *beta,
                        int64_t M, int64_t N, double eps, int mode,
                        int scaling, const int64_t *rows, int64_t nrows,
                        double *y, uint8_t *q, double *amax, double *scale,
                        uint8_t *ebyte)
{
    if (!x || !gamma || !y || !q || !amax || !scale || M < 0 || N < 1 ||
        nrows < 0 || (!rows && nrows != M))
        return -1;
    if (scaling != ORACLE_FP8_ROW && scaling != ORACLE_FP8_MX)
        return -1;
    if (scaling == ORACLE_FP8_MX && N % MX_BLOCK != 0)
        return -1;
    int64_t nb = N / MX_BLOCK;
    uint16_t *hrow = r ? malloc(sizeof(uint16_t) * (size_t)N) : NULL;
    if (r && !hrow)
        return -2;
    int rc = 0;
    for (int64_t k = 0; k < nrows && rc == 0; ++k) {
        int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= M) {
            rc = -1;
            break;
        }
        const uint16_t *src = x + i * N;
        if (r) {
            residual_add_row(x + i * N, r + i * N, N, hrow);
            src = hrow;
        }
        double *yk = y + k * N;
        rc = oracle_fwd_bf16(src, gamma, beta, 1, N, eps, mode, NULL, 1, yk,
                             NULL, NULL);
        if (rc != 0)
            break;
        if (scaling == ORACLE_FP8_ROW) {
            double am = 0.0;
            for (int64_t j = 0; j < N; ++j)
                if (fabs(yk[j]) > am)
                    am = fabs(yk[j]);
            amax[k] = am;
            scale[k] = am > 0.0 ? am / E4M3_MAX : 1.0;
            for (int64_t j = 0; j < N; ++j)
                q[k * N + j] = e4m3_code(am > 0.0 ? (yk[j] / am) * E4M3_MAX : yk[j]);
        } else {
            for (int64_t b = 0; b < nb; ++b) {
                const double *yb = yk + b * MX_BLOCK;
                double am = 0.0;
                for (int j = 0; j < MX_BLOCK; ++j)
                    if (fabs(yb[j]) > am)
                        am = fabs(yb[j]);
                int e = -127;
                if (am > 0.0) {
                    int e2;
                    frexp(am, &e2);
                    e = (e2 - 1) - 8;
                    if (e < -127)
                        e = -127;
                }
                amax[k * nb + b] = am;
                scale[k * nb + b] = ldexp(1.0, e);
                if (ebyte)
                    ebyte[k * nb + b] = (uint8_t)(e + 127);
                for (int j = 0; j < MX_BLOCK; ++j)
                    q[k * N + b * MX_BLOCK + j] = e4m3_code(ldexp(yb[j], -e));
            }
        }
    }
    free(hrow);
    return rc;
}

/*
 * Normalisation feeding a GEMM (the "Lazy Pre-Norm" fusion named in item 4,
 * "Lazy Pre-Norm and Multi-CTA Norm Fusion", of the page "Towards Free
 * Normalization: Fusing Normalization into GEMM and Attention Kernels"; its
 * items 9 and 10 describe the GEMM that consumes the normalised rows).  The
 * page gives no formula; the plainest reading is a pre-norm linear layer:
 *
 *   y   = norm(x)                (the forward definition above, in double,
 *                                 with gamma and beta; y is NOT rounded)
 *   out_ik = sum_j y_ij * W_kj   (W is [Nout, K] row-major: one row per
 *                                 output feature, K = the normalised width)
 *
 * Written as the definition: the normalised row in double, then one dot
 * product per output feature in increasing j.  How a fused kernel
 * rearranges the arithmetic (folding gamma into W, applying rstd and the
 * mean after the contraction) is its own business; the result here is the
 * composition itself.  `rows` selects output rows as in oracle_fwd_bf16.
 */
int oracle_norm_gemm_bf16(const uint16_t *x, const uint16_t *gamma,
                          const uint16_t *beta, const uint16_t *w, int64_t M,
                          int64_t K, int64_t Nout, double eps, int mode,
                          const int64_t *rows, int64_t nrows, double *out,
                          double *rstd, double *mean)
{
    if (!x || !gamma || !w || !out || M < 0 || K < 1 || Nout < 1 || nrows < 0)
        return -1;
    if (!rows && nrows != M)
        return -1;
    double *xr = malloc(sizeof(double) * (size_t)K);
    double *g = malloc(sizeof(double) * (size_t)K);
    double *b = beta ? malloc(sizeof(double) * (size_t)K) : NULL;
    double *yr = malloc(sizeof(double) * (size_t)K);
    double *wr = malloc(sizeof(double) * (size_t)K);
    if (!xr || !g || (beta && !b) || !yr || !wr) {
        free(xr); free(g); free(b); free(yr); free(wr);
        return -2;
    }
    widen_row(gamma, K, g);
    if (beta)
        widen_row(beta, K, b);
    int rc = 0;
    for (int64_t k = 0; k < nrows && rc == 0; ++k) {
        int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= M) {
            rc = -1;
            break;
        }
        widen_row(x + i * K, K, xr);
        double mu, r;
        fwd_row(xr, g, b, K, eps, mode, yr, &mu, &r);
        if (rstd)
            rstd[k] = r;
        if (mean)
            mean[k] = mu;
        for (int64_t o = 0; o < Nout; ++o) {
            widen_row(w + o * K, K, wr);
            double s = 0.0;
            for (int64_t j = 0; j < K; ++j)
                s += yr[j] * wr[j];
            out[k * Nout + o] = s;
        }
    }
    free(xr); free(g); free(b); free(yr); free(wr);
    return rc;
}
