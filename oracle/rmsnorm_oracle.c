/*
 * Plain fp64 CPU oracle for RMSNorm forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library. The CUDA library
 * never links, includes or calls it, and it shares no code with the CUDA
 * library: this file decodes its own inputs and does its own arithmetic.
 *
 * What it computes (one row i of an M x N row-major matrix, columns j):
 *
 *   forward   r_i    = 1 / sqrt( (1/N) * sum_j x_ij^2 + eps )
 *             y_ij   = x_ij * r_i * w_j
 *       "Chapter 13: Fused RMSNorm" (hello-gpu), section 13.1, the defining
 *       equation; eps sits inside the square root and the mean divides by
 *       the true column count N (same page, section 13.1 figure walk-through
 *       and the note under "why the mask cannot change the denominator").
 *       The same definition is written as rms(x) = sqrt(mean(x^2) + eps),
 *       y = x / rms * w in "Profiling, GPU utilisation and writing a fused
 *       kernel", Problem 15.
 *
 *   backward  xhat_ij = x_ij * r_i
 *             g_ij    = dy_ij * w_j
 *             c_i     = (1/N) * sum_j g_ij * xhat_ij
 *             dx_ij   = r_i * (g_ij - xhat_ij * c_i)
 *             dw_j    = sum_i dy_ij * xhat_ij
 *       "RMSNorm backward (almost) without the column reduction", sections
 *       "The backward pass" and "The naive kernel" (the page's equations
 *       were lost in extraction; its kernels compute the input gradient as
 *       r*w*g - x*mean(w*g*x)*r^3 and the weight contribution g*x*r with g
 *       the incoming gradient, which is the expression above expanded).
 *
 *   residual add (fused before the norm)
 *             h_ij   = x_ij + res_ij, stored in the activation type
 *             y, r   = the forward above applied to the stored h
 *             backward: the norm's input gradient at h plus dres (the
 *             gradient reaching h from its other uses); it is the gradient
 *             of both x and res, since h = x + res. dw is the weight
 *             gradient above with h in place of x.
 *       "Profiling, GPU utilisation and writing a fused kernel", Problem 15:
 *       the practice step that extends the kernel with a residual tensor,
 *       writes x + residual back and normalises that sum (the text under the
 *       listing calls this fusion the bigger win in a real model). The sum
 *       is rounded once into the stored type, so the fused op equals adding
 *       in that type and then normalising.
 *
 * Every sum runs in ascending index order in double precision. The CPU
 * reference of the hello-gpu chapter (section 13.4) accumulates the sum of
 * squares in double as well. r_i is always recomputed from x here; the
 * backward never reads an rstd produced elsewhere.
 *
 * Inputs are read in their stored type (fp64, fp32, bf16 or fp16; the weight
 * may have its own type, e.g. an fp32 master weight with bf16 activations --
 * "What a tuned RMSNorm kernel actually costs on Hopper", section 07) and
 * converted to double exactly; outputs are double. Where the caller passes a
 * list of row indices, only those rows of y, r and dx are produced (so huge
 * matrices can be checked on a sample); dw always covers every row.
 *
 * Parity status: every function here is pinned by the tests under tests/
 * (printed worked examples, closed forms, finite differences and an
 * independent library autograd cross-check).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F64 0
#define ORACLE_F32 1
#define ORACLE_BF16 2
#define ORACLE_F16 3

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* IEEE 754 binary16: sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * exponent 0 encodes subnormals (fraction * 2^-24), exponent 31 inf/NaN. */
static double half_bits_to_double(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

/*
 * Round v to the nearest number of a binary floating-point format with p
 * significant bits, smallest normal exponent emin and largest exponent emax:
 * IEEE 754 round to nearest, ties to the even significand; below 2^emin the
 * spacing stays 2^(emin-p+1) (subnormals); a result beyond the largest finite
 * value becomes an infinity of v's sign. nearbyint rounds in the current
 * mode, which is to nearest even unless a caller changed it.
 */
static double round_to_format(double v, int p, int emin, int emax)
{
    double q, r, maxf;
    int e;
    if (v != v || v == 0.0 || isinf(v))
        return v;
    frexp(v, &e); /* |v| = f * 2^e with 1/2 <= f < 1 */
    e -= 1;       /* 2^e <= |v| < 2^(e+1) */
    if (e < emin)
        e = emin;
    q = ldexp(1.0, e - (p - 1));
    r = nearbyint(v / q) * q;
    maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > maxf)
        return copysign(INFINITY, v);
    return r;
}

/* The value that storing v in dtype keeps: fp32 (24 bits, exponents
 * -126..127), bf16 (8 bits, same exponent range), fp16 (11 bits, -14..15). */
static double round_to_dtype(double v, int dtype)
{
    if (dtype == ORACLE_F32)
        return round_to_format(v, 24, -126, 127);
    if (dtype == ORACLE_BF16)
        return round_to_format(v, 8, -126, 127);
    if (dtype == ORACLE_F16)
        return round_to_format(v, 11, -14, 15);
    return v;
}

/* Element k of an array stored as dtype, as an exact double. */
static double load_as_double(const void *base, int dtype, int64_t k)
{
    if (dtype == ORACLE_F64)
        return ((const double *)base)[k];
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[k];
    if (dtype == ORACLE_F16)
        return half_bits_to_double(((const uint16_t *)base)[k]);
    /* bf16: the 16 stored bits are the high half of an IEEE binary32. */
    {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[k]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
}

static int dtype_ok(int dtype)
{
    return dtype == ORACLE_F64 || dtype == ORACLE_F32 || dtype == ORACLE_BF16 ||
           dtype == ORACLE_F16;
}

static int check_args(const void *x, int64_t M, int64_t N, int dtype)
{
    if (M < 0 || N <= 0)
        return ORACLE_BAD_ARG;
    if (!dtype_ok(dtype))
        return ORACLE_BAD_ARG;
    if (M > 0 && x == NULL)
        return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* r_i = 1 / sqrt(mean_j x_ij^2 + eps) for one row. */
static double row_rstd(const void *x, int dtype, int64_t i, int64_t N, double eps)
{
    double sum_sq = 0.0;
    int64_t j;
    for (j = 0; j < N; ++j) {
        double v = load_as_double(x, dtype, i * N + j);
        sum_sq += v * v;
    }
    return 1.0 / sqrt(sum_sq / (double)N + eps);
}

/* Row index number k of the requested set: rows[k], or k when rows is NULL. */
static int64_t pick_row(const int64_t *rows, int64_t k)
{
    return rows ? rows[k] : k;
}

static int check_rows(const int64_t *rows, int64_t nrows, int64_t M)
{
    int64_t k;
    if (rows == NULL)
        return nrows == M ? ORACLE_OK : ORACLE_BAD_ARG;
    for (k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= M)
            return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/*
 * Forward. x is stored as dtype, w as w_dtype. y_out is nrows x N (row k of
 * y_out is row pick_row(k) of the matrix), r_out has nrows entries. Either
 * output may be NULL.
 */
int oracle_rmsnorm_fwd(const void *x, const void *w, int64_t M, int64_t N,
                       double eps, int dtype, int w_dtype, const int64_t *rows,
                       int64_t nrows, double *y_out, double *r_out)
{
    int64_t k, j;
    if (check_args(x, M, N, dtype) || check_rows(rows, nrows, M) || !dtype_ok(w_dtype))
        return ORACLE_BAD_ARG;
    if (nrows > 0 && y_out && w == NULL)
        return ORACLE_BAD_ARG;
    for (k = 0; k < nrows; ++k) {
        int64_t i = pick_row(rows, k);
        double r = row_rstd(x, dtype, i, N, eps);
        if (r_out)
            r_out[k] = r;
        if (y_out)
            for (j = 0; j < N; ++j)
                y_out[k * N + j] = load_as_double(x, dtype, i * N + j) * r *
                                   load_as_double(w, w_dtype, j);
    }
    return ORACLE_OK;
}

/* Backward input gradient for the requested rows; dx_out is nrows x N. x
 * and dy are stored as dtype, w as w_dtype. */
int oracle_rmsnorm_bwd_dx(const void *x, const void *w, const void *dy,
                          int64_t M, int64_t N, double eps, int dtype, int w_dtype,
                          const int64_t *rows, int64_t nrows, double *dx_out)
{
    int64_t k, j;
    if (check_args(x, M, N, dtype) || check_rows(rows, nrows, M) || !dtype_ok(w_dtype))
        return ORACLE_BAD_ARG;
    if (nrows > 0 && (w == NULL || dy == NULL || dx_out == NULL))
        return ORACLE_BAD_ARG;
    for (k = 0; k < nrows; ++k) {
        int64_t i = pick_row(rows, k);
        double r = row_rstd(x, dtype, i, N, eps);
        double c = 0.0;
        for (j = 0; j < N; ++j) {
            double xhat = load_as_double(x, dtype, i * N + j) * r;
            double g = load_as_double(dy, dtype, i * N + j) *
                       load_as_double(w, w_dtype, j);
            c += g * xhat;
        }
        c /= (double)N;
        for (j = 0; j < N; ++j) {
            double xhat = load_as_double(x, dtype, i * N + j) * r;
            double g = load_as_double(dy, dtype, i * N + j) *
                       load_as_double(w, w_dtype, j);
            dx_out[k * N + j] = r * (g - xhat * c);
        }
    }
    return ORACLE_OK;
}

/* Backward weight gradient over all M rows, rows summed in ascending order. */
int oracle_rmsnorm_bwd_dw(const void *x, const void *dy, int64_t M, int64_t N,
                          double eps, int dtype, double *dw_out)
{
    int64_t i, j;
    if (check_args(x, M, N, dtype) || dw_out == NULL)
        return ORACLE_BAD_ARG;
    if (M > 0 && dy == NULL)
        return ORACLE_BAD_ARG;
    for (j = 0; j < N; ++j)
        dw_out[j] = 0.0;
    for (i = 0; i < M; ++i) {
        double r = row_rstd(x, dtype, i, N, eps);
        for (j = 0; j < N; ++j) {
            double xhat = load_as_double(x, dtype, i * N + j) * r;
            dw_out[j] += load_as_double(dy, dtype, i * N + j) * xhat;
        }
    }
    return ORACLE_OK;
}

/* Rounds n doubles into dtype's values (exposed so that the rounding can be
 * checked on its own). */
int oracle_round_to_dtype(const double *v, int64_t n, int dtype, double *out)
{
    int64_t k;
    if (n < 0 || !dtype_ok(dtype) || (n > 0 && (v == NULL || out == NULL)))
        return ORACLE_BAD_ARG;
    for (k = 0; k < n; ++k)
        out[k] = round_to_dtype(v[k], dtype);
    return ORACLE_OK;
}

/* h_ij = x_ij + res_ij as stored in dtype. */
static double stored_sum(const void *x, const void *res, int dtype, int64_t k)
{
    return round_to_dtype(load_as_double(x, dtype, k) + load_as_double(res, dtype, k), dtype);
}

/*
 * Residual add, then the forward. x and res are stored as dtype, w as
 * w_dtype. For each requested row: h_out (the stored sum, nrows x N), y_out
 * (nrows x N) and r_out (nrows). Any output may be NULL.
 */
int oracle_rmsnorm_add_fwd(const void *x, const void *res, const void *w, int64_t M,
                           int64_t N, double eps, int dtype, int w_dtype,
                           const int64_t *rows, int64_t nrows, double *h_out,
                           double *y_out, double *r_out)
{
    int64_t k, j;
    if (check_args(x, M, N, dtype) || check_rows(rows, nrows, M) || !dtype_ok(w_dtype))
        return ORACLE_BAD_ARG;
    if (nrows > 0 && (res == NULL || (y_out && w == NULL)))
        return ORACLE_BAD_ARG;
    for (k = 0; k < nrows; ++k) {
        int64_t i = pick_row(rows, k);
        double sum_sq = 0.0, r;
        for (j = 0; j < N; ++j) {
            double h = stored_sum(x, res, dtype, i * N + j);
            sum_sq += h * h;
        }
        r = 1.0 / sqrt(sum_sq / (double)N + eps);
        if (r_out)
            r_out[k] = r;
        for (j = 0; j < N; ++j) {
            double h = stored_sum(x, res, dtype, i * N + j);
            if (h_out)
                h_out[k * N + j] = h;
            if (y_out)
                y_out[k * N + j] = h * r * load_as_double(w, w_dtype, j);
        }
    }
    return ORACLE_OK;
}

/*
 * Backward of the residual add plus norm. h is the stored sum the forward
 * wrote (as dtype), dres the gradient that reaches h from its other uses (as
 * dtype, or NULL for none). dx_out (nrows x N) is the norm's input gradient at
 * h plus dres: the gradient of x and of res alike.
 */
int oracle_rmsnorm_add_bwd_dx(const void *h, const void *w, const void *dy, const void *dres,
                              int64_t M, int64_t N, double eps, int dtype, int w_dtype,
                              const int64_t *rows, int64_t nrows, double *dx_out)
{
    int64_t k, j;
    int rc = oracle_rmsnorm_bwd_dx(h, w, dy, M, N, eps, dtype, w_dtype, rows, nrows, dx_out);
    if (rc != ORACLE_OK || dres == NULL)
        return rc;
    for (k = 0; k < nrows; ++k) {
        int64_t i = pick_row(rows, k);
        for (j = 0; j < N; ++j)
            dx_out[k * N + j] += load_as_double(dres, dtype, i * N + j);
    }
    return ORACLE_OK;
}
