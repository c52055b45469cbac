/*
 * Plain CPU oracle for the output-stationary tiled matrix multiply C = A @ B.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the GPU
 * library: only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes, and where each piece comes from:
 *
 *  - orc_gemm / orc_gemm_entries: the plain definition of the product,
 *    C[i,j] = sum_k A[i,k] * B[k,j] with A of shape M x K and B of shape K x N,
 *    both row-major ("Reading a matrix multiply through its tiles", intro;
 *    "Tiled Matrix Multiplication", the "Actual Computation Pattern" note of
 *    the idiomatic kernel).  Tiling only reorders this sum, so the oracle is
 *    the definition itself: a naive i-k-j loop with an FP64 accumulator over
 *    the inputs exactly as the GPU sees them (already rounded to their
 *    storage type, then widened exactly).  It also accumulates
 *    sum_k |A[i,k] * B[k,j]|, the scale of the element-wise error bound.
 *
 *  - orc_round: conversion of an FP64 value to the output storage type with
 *    IEEE round-to-nearest-even (the pages leave the rounding open; nearest-
 *    even is the IEEE default and the reading taken here).  The helion kernel
 *    of "Writing a matmul GPU kernel" accumulates in FP32 and stores into a
 *    tensor of the input dtype, which is where this conversion happens.
 *
 *  - orc_traffic: the tile-level traffic and working-set model of "Reading a
 *    matrix multiply through its tiles", sections "What fits in local
 *    storage?", "Count the repeated reads" and "Edge tiles still matter".  It
 *    walks the output-stationary loop nest of "Keep one output tile resident"
 *    tile by tile and counts the actual row, column and reduction extents of
 *    every tile, so partial edge tiles are counted exactly.
 *
 *  - orc_tile_ranges: the slicing of one dimension into consecutive tiles,
 *    the last one partial (helion's hl.tile in "Writing a matmul GPU kernel":
 *    size 10 with tile 4 gives 0:4, 4:8, 8:10).
 *
 * Every function returns 0 on success and a negative value on bad arguments.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Storage types understood by the oracle (its own numbering). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---------------------------------------------------------------- widening */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)               /* zero or subnormal: frac * 2^-24 */
        v = ldexp((double)frac, -24);
    else if (expo == 31)         /* inf or nan */
        v = frac ? NAN : INFINITY;
    else                         /* normal: (1024 + frac) * 2^(expo-25) */
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[idx];
    if (dtype == ORC_F16)
        return half_bits_to_double(((const uint16_t *)base)[idx]);
    return bf16_bits_to_double(((const uint16_t *)base)[idx]);
}

static int dtype_ok(int dtype)
{
    return dtype == ORC_F32 || dtype == ORC_F16 || dtype == ORC_BF16;
}

int orc_widen(const void *src, int dtype, int64_t n, double *dst)
{
    if (!dtype_ok(dtype) || n < 0 || (n > 0 && (!src || !dst)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = load_elem(src, dtype, i);
    return 0;
}

/* ---------------------------------------------------------------- rounding */

/* Round x to the nearest value with `p` significand bits, smallest normal
 * exponent `emin` and largest finite value `maxf`, ties to even; values that
 * round beyond maxf become infinities.  Every step is an exact scaling by a
 * power of two or an exact integer rounding, so the result is correctly
 * rounded directly from the FP64 input (no double rounding). */
static double round_to_format(double x, int p, int emin, double maxf)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    int e;
    frexp(x, &e);            /* |x| = m * 2^e with m in [0.5, 1) */
    e -= 1;                  /* now |x| in [2^e, 2^(e+1)) */
    if (e < emin)
        e = emin;            /* subnormal range: fixed quantum */
    double q = ldexp(1.0, e - (p - 1));
    double r = x / q;        /* exact */
    double fl = floor(r);
    double diff = r - fl;    /* exact, in [0, 1) */
    double n;
    if (diff > 0.5)
        n = fl + 1.0;
    else if (diff < 0.5)
        n = fl;
    else                     /* tie: pick the even neighbour */
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double y = n * q;        /* exact */
    if (fabs(y) > maxf)
        return x > 0 ? INFINITY : -INFINITY;
    return y;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* Encode a value that is already exactly representable in binary16. */
static uint16_t double_to_half_bits_exact(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (isinf(v))
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    e -= 1;                                   /* a in [2^e, 2^(e+1)) */
    if (e < -14)                              /* subnormal */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    uint16_t frac = (uint16_t)(a / ldexp(1.0, e - 10) - 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | frac;
}

int orc_round(const double *src, int64_t n, int dtype, void *dst)
{
    if (!dtype_ok(dtype) || n < 0 || (n > 0 && (!src || !dst)))
        return -1;
    for (int64_t i = 0; i < n; ++i) {
        double x = src[i];
        if (dtype == ORC_F32) {
            /* binary32: 24 significand bits, emin -126 */
            double y = round_to_format(x, 24, -126, 3.4028234663852886e38);
            ((float *)dst)[i] = isnan(y) ? NAN : (float)y;   /* exact */
        } else if (dtype == ORC_F16) {
            /* binary16: 11 significand bits, emin -14, max 65504 */
            double y = round_to_format(x, 11, -14, 65504.0);
            ((uint16_t *)dst)[i] = double_to_half_bits_exact(y);
        } else {
            /* bfloat16: 8 significand bits, binary32's exponent range */
            double y = round_to_format(x, 8, -126, 3.3895313892515355e38);
            uint32_t u = isnan(y) ? 0x7fc00000u : float_bits((float)y);
            ((uint16_t *)dst)[i] = (uint16_t)(u >> 16);      /* exact */
        }
    }
    return 0;
}

/* ------------------------------------------------------------ the product */

struct gemm_job {
    const void *A, *B;
    int dtype;
    int64_t M, N, K;
    double *C, *Cabs;
    int64_t row_begin, row_end;
};

/* One output row at a time: acc[j] += A[i,k] * B[k,j] for k ascending. */
static void *gemm_rows(void *arg)
{
    struct gemm_job *job = (struct gemm_job *)arg;
    int64_t N = job->N, K = job->K;
    double *brow = (double *)malloc(sizeof(double) * (size_t)(N ? N : 1));
    if (!brow)
        return (void *)1;
    for (int64_t i = job->row_begin; i < job->row_end; ++i) {
        double *c = job->C + i * N;
        double *cabs = job->Cabs ? job->Cabs + i * N : NULL;
        for (int64_t j = 0; j < N; ++j) {
            c[j] = 0.0;
            if (cabs)
                cabs[j] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            double a = load_elem(job->A, job->dtype, i * K + k);
            for (int64_t j = 0; j < N; ++j)
                brow[j] = load_elem(job->B, job->dtype, k * N + j);
            for (int64_t j = 0; j < N; ++j) {
                double prod = a * brow[j];
                c[j] += prod;
                if (cabs)
                    cabs[j] += fabs(prod);
            }
        }
    }
    free(brow);
    return NULL;
}

/* C (M x N, FP64) = A (M x K) @ B (K x N), both in storage type `dtype`.
 * Cabs (may be NULL) receives sum_k |A[i,k] * B[k,j]|.  Rows are split over
 * `nthreads` host threads (<= 0 means one). */
int orc_gemm(const void *A, const void *B, int dtype, int64_t M, int64_t N,
             int64_t K, double *C, double *Cabs, int nthreads)
{
    if (!dtype_ok(dtype) || M < 0 || N < 0 || K < 0)
        return -1;
    if (M * N > 0 && !C)
        return -1;
    if (M * N > 0 && K > 0 && (!A || !B))
        return -1;
    if (M == 0 || N == 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > M)
        nthreads = (int)M;
    struct gemm_job *jobs = (struct gemm_job *)calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof *tids);
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        struct gemm_job j = {A, B, dtype, M, N, K, C, Cabs,
                             M * t / nthreads, M * (t + 1) / nthreads};
        jobs[t] = j;
        if (pthread_create(&tids[t], NULL, gemm_rows, &jobs[t]) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret)
            rc = -2;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* The general form: C = alpha * op(A) @ op(B) + beta * C_in, where op(A) is
 * M x K and op(B) is K x N.  op = 0 takes the matrix as stored (A row-major
 * M x K, B row-major K x N); op = 1 takes its transpose (A stored row-major
 * K x M, B stored row-major N x K), the transposed loadings the puzzle page
 * lists for pre-transposed inputs ("Tiled Matrix Multiplication",
 * "Educational: When would transposed loading be useful?").  C_in (storage
 * type c_dtype, row-major M x N) is read only when beta != 0, the
 * accumulate-into-the-output form of torch.addmm that the helion kernel
 * builds its tiles with ("Writing a matmul GPU kernel").  Cabs receives
 * |alpha| * sum_k |op(A)[i,k] op(B)[k,j]|.  Single-threaded, row by row. */
int orc_gemm_general(const void *A, const void *B, int dtype, int64_t M, int64_t N, int64_t K,
                     int op_a, int op_b, double alpha, double beta, const void *C_in,
                     int c_dtype, double *C, double *Cabs)
{
    if (!dtype_ok(dtype) || !dtype_ok(c_dtype) || M < 0 || N < 0 || K < 0)
        return -1;
    if ((op_a != 0 && op_a != 1) || (op_b != 0 && op_b != 1))
        return -1;
    if (M * N > 0 && !C)
        return -1;
    if (M * N > 0 && K > 0 && (!A || !B))
        return -1;
    if (M * N > 0 && beta != 0.0 && !C_in)
        return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t ia = op_a ? k * M + i : i * K + k;
                int64_t ib = op_b ? j * K + k : k * N + j;
                double prod = load_elem(A, dtype, ia) * load_elem(B, dtype, ib);
                acc += prod;
                acc_abs += fabs(prod);
            }
            double c = alpha * acc;
            if (beta != 0.0)
                c += beta * load_elem(C_in, c_dtype, i * N + j);
            C[i * N + j] = c;
            if (Cabs)
                Cabs[i * N + j] = fabs(alpha) * acc_abs;
        }
    }
    return 0;
}

/* Selected entries C[rows[s], cols[s]], each a single k-ascending dot
 * product; used where the full product is too large to form on the host. */
int orc_gemm_entries(const void *A, const void *B, int dtype, int64_t M,
                     int64_t N, int64_t K, const int64_t *rows,
                     const int64_t *cols, int64_t count, double *out,
                     double *out_abs)
{
    if (!dtype_ok(dtype) || M < 0 || N < 0 || K < 0 || count < 0)
        return -1;
    if (count > 0 && (!rows || !cols || !out))
        return -1;
    if (K > 0 && count > 0 && (!A || !B))
        return -1;
    for (int64_t s = 0; s < count; ++s) {
        int64_t i = rows[s], j = cols[s];
        if (i < 0 || i >= M || j < 0 || j >= N)
            return -1;
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = load_elem(A, dtype, i * K + k) * load_elem(B, dtype, k * N + j);
            acc += prod;
            acc_abs += fabs(prod);
        }
        out[s] = acc;
        if (out_abs)
            out_abs[s] = acc_abs;
    }
    return 0;
}

/* ------------------------------------------------------ traffic and tiles */

/* Slice [0, n) into consecutive tiles of size t, the last one partial.
 * Writes up to `cap` (start, length) pairs and returns the tile count. */
int64_t orc_tile_ranges(int64_t n, int64_t t, int64_t *starts, int64_t *lens,
                        int64_t cap)
{
    if (n < 0 || t <= 0)
        return -1;
    int64_t count = 0;
    for (int64_t s = 0; s < n; s += t) {
        if (count < cap) {
            starts[count] = s;
            lens[count] = (n - s < t) ? n - s : t;
        }
        ++count;
    }
    return count;
}

/* Result slots written by orc_traffic (all int64). */
enum {
    TR_A_ELEMS = 0,     /* A elements read, summed over every tile step   */
    TR_B_ELEMS,         /* B elements read                                */
    TR_C_ELEMS,         /* C elements written (once per output tile)      */
    TR_BYTES,           /* A, B bytes at in_bytes plus C bytes at c_bytes */
    TR_FLOPS,           /* multiply + add counted as two operations       */
    TR_TILES,           /* output tiles                                   */
    TR_STEPS,           /* tile steps along K, summed over output tiles   */
    TR_WS_MAX,          /* largest per-step working set in bytes          */
    TR_WS_FULL,         /* working set of one full tm x tn x tk step      */
    TR_COUNT
};

/* Walk the output-stationary loop nest (for each output tile: for each K
 * tile: read an A tile and a B tile; then write the C tile once) and count
 * the actual extents of every tile.  The per-step working set is the
 * resident A tile, B tile (input bytes) and C accumulator (acc_bytes); double
 * buffering and padding are excluded, as in the pages' model. */
int orc_traffic(int64_t M, int64_t N, int64_t K, int64_t tm, int64_t tn,
                int64_t tk, int64_t in_bytes, int64_t acc_bytes,
                int64_t c_bytes, int64_t *res)
{
    if (M < 0 || N < 0 || K < 0 || tm <= 0 || tn <= 0 || tk <= 0 || !res)
        return -1;
    for (int s = 0; s < TR_COUNT; ++s)
        res[s] = 0;
    res[TR_WS_FULL] = tm * tk * in_bytes + tk * tn * in_bytes + tm * tn * acc_bytes;
    for (int64_t mo = 0; mo < M; mo += tm) {
        int64_t rm = (M - mo < tm) ? M - mo : tm;
        for (int64_t no = 0; no < N; no += tn) {
            int64_t rn = (N - no < tn) ? N - no : tn;
            res[TR_TILES] += 1;
            for (int64_t ko = 0; ko < K; ko += tk) {
                int64_t rk = (K - ko < tk) ? K - ko : tk;
                res[TR_A_ELEMS] += rm * rk;
                res[TR_B_ELEMS] += rk * rn;
                res[TR_FLOPS] += 2 * rm * rn * rk;
                res[TR_STEPS] += 1;
                int64_t ws = rm * rk * in_bytes + rk * rn * in_bytes + rm * rn * acc_bytes;
                if (ws > res[TR_WS_MAX])
                    res[TR_WS_MAX] = ws;
            }
            res[TR_C_ELEMS] += rm * rn;
        }
    }
    res[TR_BYTES] = (res[TR_A_ELEMS] + res[TR_B_ELEMS]) * in_bytes + res[TR_C_ELEMS] * c_bytes;
    return 0;
}
