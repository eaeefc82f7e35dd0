/*
 * Plain fp64 CPU oracle for the fused residual-Add + LayerNorm row operation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or constant with the
 * CUDA library: it decodes and rounds the 16-bit formats itself, from their
 * IEEE definitions, and computes every row with the slow two-pass formula.
 *
 * What it computes, for each row i of X and R ([rows, H], row-major):
 *   A_ij   = x_ij + r_ij                         ("算子融合的收益量化" section 1:
 *                                                 the residual add whose sum A
 *                                                 the fused kernel keeps on chip)
 *   mean_i = (1/H) * sum_j A_ij                  ("算子融合与Kernel合并" 4.2,
 *   var_i  = (1/H) * sum_j (A_ij - mean_i)^2      fused_layernorm: two passes,
 *   std_i  = sqrt(var_i + eps)                     biased variance, eps inside
 *   Y_ij   = gamma_j * (A_ij - mean_i) / std_i     the square root, per-element
 *            + beta_j                              gamma and beta)
 *   rstd_i = 1 / std_i
 * The page's one-pass sum / sum-of-squares shortcut (same page, 4.3) is not
 * used: it loses the variance when mean >> std.
 *
 * Readings where the pages are silent:
 *   - statistics use the unrounded sum A (fp64); with round_A != 0 the sum is
 *     first rounded to the I/O dtype, which is what a two-kernel chain that
 *     stores A in that dtype computes;
 *   - the A output is A rounded to the I/O dtype (round to nearest, ties to
 *     even), returned as a double;
 *   - Y, mean and rstd are returned unrounded in fp64.
 *
 * Row softmax ("算子融合与Kernel合并" 4.3, fused_softmax), per row i of X:
 *   max_i  = max_j x_ij
 *   sum_i  = sum_j exp(x_ij - max_i)
 *   Y_ij   = exp(x_ij - max_i) / sum_i
 * in the page's order: a max pass, an exp-sum pass, a divide pass; fp64
 * throughout, libm exp.
 *
 * Bias + GELU + residual ("算子融合的收益量化", the three-kernel chain of the
 * diagram before section 1: BiasAdd, GELU, Residual), per element:
 *   v_ij = x_ij + bias_j
 *   Y_ij = GELU(v_ij) + r_ij,   GELU(v) = v * Phi(v) = v/2 * (1 + erf(v / sqrt 2))
 * (the exact, erf form; the page names no variant), fp64 with libm erf.
 *
 * Backward of the fused operation (the pages give no backward: this is the
 * textbook derivative of the definition above).  Inputs: dY, the stored sum A,
 * the per-row mean and rstd as saved, gamma, and optionally dA_in, a gradient
 * reaching A from elsewhere (A is also the residual stream).  Per row:
 *   xhat_j = (A_j - mean) * rstd,   g_j = dY_j * gamma_j
 *   dA_j   = rstd * (g_j - (1/H) sum_k g_k - xhat_j (1/H) sum_k g_k xhat_k) + dA_in_j
 *   dX = dR = dA
 * and over rows:  dgamma_j = sum_i dY_ij xhat_ij,  dbeta_j = sum_i dY_ij.
 *
 * dtype codes: 0 = IEEE binary32, 1 = IEEE binary16, 2 = bfloat16.
 * Return value: 0 on success, -1 on a bad argument.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math), so
 * that x86-64 and aarch64 give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* IEEE 754 binary16: sign, 5-bit exponent with bias 15, 10-bit fraction.
 * Normal: (1 + f/2^10) * 2^(e-15) = (2^10 + f) * 2^(e-25).
 * Subnormal (e = 0): f * 2^-24. */
static double decode_binary16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: sign, 8-bit exponent with bias 127, 7-bit fraction.
 * Normal: (2^7 + f) * 2^(e-134).  Subnormal (e = 0): f * 2^-133. */
static double decode_bfloat16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

static double decode_at(const void *src, int dtype, int64_t k)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)src)[k];
    uint16_t bits = ((const uint16_t *)src)[k];
    return dtype == ORACLE_F16 ? decode_binary16(bits) : decode_bfloat16(bits);
}

/* Round v to a binary format with p significand bits (hidden bit included),
 * smallest normal exponent emin and largest exponent emax, to nearest with
 * ties to even.  Below 2^emin the spacing stays 2^(emin-p+1) (subnormals).
 * A result beyond the largest finite value becomes an infinity. */
static double round_binary(double v, int p, int emin, int emax)
{
    if (!isfinite(v) || v == 0.0)
        return v;
    int e2;
    frexp(fabs(v), &e2);          /* |v| in [2^(e2-1), 2^e2) */
    int ex = e2 - 1;
    if (ex < emin)
        ex = emin;
    double q = ldexp(v, p - 1 - ex);          /* v / ulp(v) */
    double n = nearbyint(q);                  /* default mode: nearest, ties even */
    double res = ldexp(n, ex - p + 1);
    double maxfinite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(res) > maxfinite)
        return copysign(INFINITY, v);
    return res;
}

static double round_to_dtype(double v, int dtype)
{
    switch (dtype) {
    case ORACLE_F32:  return round_binary(v, 24, -126, 127);
    case ORACLE_F16:  return round_binary(v, 11, -14, 15);
    default:          return round_binary(v, 8, -126, 127);
    }
}

static int bad_dtype(int dtype)
{
    return dtype != ORACLE_F32 && dtype != ORACLE_F16 && dtype != ORACLE_BF16;
}

int oracle_decode(const void *src, int dtype, int64_t n, double *out)
{
    if (bad_dtype(dtype) || n < 0 || (n > 0 && (!src || !out)))
        return -1;
    for (int64_t k = 0; k < n; ++k)
        out[k] = decode_at(src, dtype, k);
    return 0;
}

int oracle_round(const double *src, int dtype, int64_t n, double *out)
{
    if (bad_dtype(dtype) || n < 0 || (n > 0 && (!src || !out)))
        return -1;
    for (int64_t k = 0; k < n; ++k)
        out[k] = round_to_dtype(src[k], dtype);
    return 0;
}

/* A = X + R elementwise (exact in fp64 for 16-bit inputs); round_A != 0
 * rounds each sum to the I/O dtype. */
int oracle_add(const void *x, const void *r, int dtype, int64_t n, int round_A, double *a)
{
    if (bad_dtype(dtype) || n < 0 || (n > 0 && (!x || !r || !a)))
        return -1;
    for (int64_t k = 0; k < n; ++k) {
        double s = decode_at(x, dtype, k) + decode_at(r, dtype, k);
        a[k] = round_A ? round_to_dtype(s, dtype) : s;
    }
    return 0;
}

/* LayerNorm of one row of H doubles, in the page's order: mean, then the
 * biased variance around it, then std = sqrt(var + eps) and the affine map. */
static void layernorm_row(const double *a, const float *gamma, const float *beta, int64_t H,
                          double eps, double *y, double *mean_out, double *rstd_out)
{
    double sum = 0.0;
    for (int64_t j = 0; j < H; ++j)
        sum += a[j];
    double mean = sum / (double)H;

    double var = 0.0;
    for (int64_t j = 0; j < H; ++j)
        var += (a[j] - mean) * (a[j] - mean);
    double std = sqrt(var / (double)H + eps);

    if (y)
        for (int64_t j = 0; j < H; ++j)
            y[j] = (double)gamma[j] * (a[j] - mean) / std + (double)beta[j];
    if (mean_out)
        *mean_out = mean;
    if (rstd_out)
        *rstd_out = 1.0 / std;
}

int oracle_layernorm(const double *a, const float *gamma, const float *beta, int64_t rows,
                     int64_t H, double eps, double *y, double *mean, double *rstd)
{
    if (rows < 0 || H <= 0 || !(eps >= 0.0) || (rows > 0 && (!a || !gamma || !beta)))
        return -1;
    for (int64_t i = 0; i < rows; ++i)
        layernorm_row(a + i * H, gamma, beta, H, eps, y ? y + i * H : NULL,
                      mean ? mean + i : NULL, rstd ? rstd + i : NULL);
    return 0;
}

/* The fused operation: per row, A = X + R (kept in fp64, or rounded to the
 * dtype when round_A != 0), then LayerNorm of that row.  Every output is
 * optional; a_out receives A rounded to the I/O dtype. */
int oracle_add_layernorm(const void *x, const void *r, int dtype, const float *gamma,
                         const float *beta, int64_t rows, int64_t H, double eps, int round_A,
                         double *y, double *a_out, double *mean, double *rstd)
{
    if (bad_dtype(dtype) || rows < 0 || H <= 0 || !(eps >= 0.0))
        return -1;
    if (rows > 0 && (!x || !r || !gamma || !beta))
        return -1;
    double *row = (double *)malloc((size_t)H * sizeof(double));
    if (!row)
        return -1;
    const size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    for (int64_t i = 0; i < rows; ++i) {
        const char *xi = (const char *)x + (size_t)(i * H) * esz;
        const char *ri = (const char *)r + (size_t)(i * H) * esz;
        oracle_add(xi, ri, dtype, H, round_A, row);
        layernorm_row(row, gamma, beta, H, eps, y ? y + i * H : NULL,
                      mean ? mean + i : NULL, rstd ? rstd + i : NULL);
        if (a_out)
            for (int64_t j = 0; j < H; ++j)
                a_out[i * H + j] = round_to_dtype(row[j], dtype);
    }
    free(row);
    return 0;
}

/* Softmax of one row of H decoded values, in the page's three passes. */
static void softmax_row(const double *x, int64_t H, double *y, double *max_out, double *sum_out)
{
    double mx = -INFINITY;
    for (int64_t j = 0; j < H; ++j)
        if (x[j] > mx)
            mx = x[j];
    double sum = 0.0;
    for (int64_t j = 0; j < H; ++j)
        sum += exp(x[j] - mx);
    for (int64_t j = 0; j < H; ++j)
        y[j] = exp(x[j] - mx) / sum;
    if (max_out)
        *max_out = mx;
    if (sum_out)
        *sum_out = sum;
}

/* Row softmax of X ([rows, H] in dtype); y receives fp64 [rows, H];
 * row_max / row_sum (optional) receive max_i and sum_i. */
int oracle_softmax(const void *x, int dtype, int64_t rows, int64_t H, double *y,
                   double *row_max, double *row_sum)
{
    if (bad_dtype(dtype) || rows < 0 || H <= 0 || (rows > 0 && (!x || !y)))
        return -1;
    double *row = (double *)malloc((size_t)H * sizeof(double));
    if (!row)
        return -1;
    const size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    for (int64_t i = 0; i < rows; ++i) {
        const char *xi = (const char *)x + (size_t)(i * H) * esz;
        for (int64_t j = 0; j < H; ++j)
            row[j] = decode_at(xi, dtype, j);
        softmax_row(row, H, y + i * H, row_max ? row_max + i : NULL, row_sum ? row_sum + i : NULL);
    }
    free(row);
    return 0;
}

static double gelu_exact(double v)
{
    return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
}

/* Y = GELU(X + bias) + R over [rows, H]; bias fp32 [H]; y fp64 [rows, H].
 * round_intermediates != 0: the three-kernel chain, which stores X + bias and
 * GELU of it in the I/O dtype (each rounded to nearest even) before the next
 * step reads them. */
int oracle_bias_gelu_residual(const void *x, const void *r, int dtype, const float *bias,
                              int64_t rows, int64_t H, int round_intermediates, double *y)
{
    if (bad_dtype(dtype) || rows < 0 || H <= 0 || (rows > 0 && (!x || !r || !bias || !y)))
        return -1;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < H; ++j) {
            const int64_t k = i * H + j;
            double v = decode_at(x, dtype, k) + (double)bias[j];
            if (round_intermediates)
                v = round_to_dtype(v, dtype);
            double g = gelu_exact(v);
            if (round_intermediates)
                g = round_to_dtype(g, dtype);
            y[k] = g + decode_at(r, dtype, k);
        }
    return 0;
}

/* Backward; dy, a, dres in dtype ([rows, H]); mean, rstd fp32 [rows]; gamma
 * fp32 [H]; dres may be NULL.  Outputs fp64: dx [rows, H], dgamma, dbeta [H]
 * (each output may be NULL). */
int oracle_add_layernorm_bwd(const void *dy, const void *a, const float *mean, const float *rstd,
                             const float *gamma, const void *dres, int dtype, int64_t rows,
                             int64_t H, double *dx, double *dgamma, double *dbeta)
{
    if (bad_dtype(dtype) || rows < 0 || H <= 0)
        return -1;
    if (rows > 0 && (!dy || !a || !mean || !rstd || !gamma))
        return -1;
    double *xhat = (double *)malloc((size_t)H * sizeof(double));
    double *g = (double *)malloc((size_t)H * sizeof(double));
    if (!xhat || !g) {
        free(xhat);
        free(g);
        return -1;
    }
    if (dgamma)
        for (int64_t j = 0; j < H; ++j)
            dgamma[j] = 0.0;
    if (dbeta)
        for (int64_t j = 0; j < H; ++j)
            dbeta[j] = 0.0;
    for (int64_t i = 0; i < rows; ++i) {
        const double mu = (double)mean[i], rs = (double)rstd[i];
        double sg = 0.0, sgx = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            const int64_t k = i * H + j;
            const double dyk = decode_at(dy, dtype, k);
            xhat[j] = (decode_at(a, dtype, k) - mu) * rs;
            g[j] = dyk * (double)gamma[j];
            sg += g[j];
            sgx += g[j] * xhat[j];
            if (dgamma)
                dgamma[j] += dyk * xhat[j];
            if (dbeta)
                dbeta[j] += dyk;
        }
        const double mg = sg / (double)H, mgx = sgx / (double)H;
        if (dx)
            for (int64_t j = 0; j < H; ++j) {
                double d = rs * (g[j] - mg - xhat[j] * mgx);
                if (dres)
                    d += decode_at(dres, dtype, i * H + j);
                dx[i * H + j] = d;
            }
    }
    free(xhat);
    free(g);
    return 0;
}
