/*
 * oracle.c -- the CPU reference for the pipelined tiled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes, and where that is stated:
 *
 *  - The GEMM of the tiled kernel, C[M,N] = A[M,K] . B[N,K]^T, with B stored
 *    [N,K] and contracted over its second index ("transpose_B=True"):
 *    tutorial chapter 11 "Pipeline and autotuning", section 1.1 (the tiled
 *    GEMM body) and section 3.5 (the kernel signature with A:(M,K), B:(N,K),
 *    and the check function (a.float() @ b.float().T)).  Software pipelining
 *    changes only throughput, never the value (same chapter, section 2.4), so
 *    the oracle is the plain definition:
 *        R[i][j] = sum_{k<K} A[i][k] * B[j][k]
 *    summed in order k = 0..K-1 in IEEE binary64, together with the error
 *    scale S[i][j] = sum_k |A[i][k] * B[j][k]|.
 *  - Exact decoding of binary16 and bfloat16 bit patterns (subnormals, signed
 *    zeros, infinities and NaN included), from the IEEE 754-2008 binary16
 *    format and the bfloat16 format (the top half of binary32).
 *  - Round-to-nearest-even from binary64 to binary16 / bfloat16, written from
 *    the IEEE 754 definition of that rounding: the value is scaled by its
 *    ulp, rounded to an integer with ties to even, and scaled back;
 *    magnitudes that round past the largest finite value become infinity.
 *  - The shared-memory bound of a pipelined tile: num_stages copies of one A
 *    tile (block_M x block_K) and one B tile (block_K x block_N), times the
 *    element size -- chapter 11, section 4.5 ("multi-buffering and the
 *    on-chip capacity limit"), and section 3.7 for the config-space prune.
 *  - The FLOP count 2*M*N*K of one GEMM: "Stage 04 - GEMM main line" notes,
 *    exercise 3 (TFLOPS = 2*M*N*K / latency).
 *
 * Every function is pinned by tests that do not reuse this code: hand-worked
 * cases, exact integer arithmetic, identity and zero matrices, numpy's and
 * torch's own conversions, and the numbers the pages print for the budget.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---- decoding (IEEE 754 binary16; bfloat16 = upper 16 bits of binary32) -- */

double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

double oracle_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);              /* subnormal: m * 2^-133 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);   /* (1.m) * 2^(e-127) */
    return sign ? -v : v;
}

static double decode(uint16_t x, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(x) : oracle_f16_to_f64(x);
}

void oracle_decode(const uint16_t *in, double *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode(in[i], dtype);
}

/* ---- rounding binary64 -> 16-bit formats, nearest-even ------------------ */

/* Round x to the format with p significant bits, minimum normal exponent
 * emin (value 2^emin) and largest finite value maxf; return the rounded value
 * as a double (exact), +-inf on overflow. */
static double round_to_format(double x, int p, int emin, double maxf)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    int E;
    frexp(x, &E);                 /* |x| in [2^(E-1), 2^E) */
    int eunit = E - p;            /* ulp exponent for a normal number */
    if (E - 1 < emin)
        eunit = emin - (p - 1);   /* subnormal range: fixed ulp */
    double q = ldexp(x, -eunit);  /* exact: scaling by a power of two */
    double r = nearbyint(q);      /* default rounding mode: ties to even */
    double v = ldexp(r, eunit);
    if (fabs(v) > maxf)
        return x > 0 ? INFINITY : -INFINITY;
    return v;
}

static uint16_t encode_exact(double v, int mant_bits, int bias, int exp_max_field)
{
    /* v is an exact value of the format (or +-inf); NaN is handled by the
     * callers before rounding. */
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | (uint16_t)(exp_max_field << mant_bits);
    if (a == 0.0)
        return sign;
    int E;
    double f = frexp(a, &E);      /* a = f * 2^E, f in [0.5, 1) */
    int biased = E - 1 + bias;
    if (biased >= 1) {
        uint32_t m = (uint32_t)ldexp(f * 2.0 - 1.0, mant_bits);
        return sign | (uint16_t)((biased << mant_bits) | m);
    }
    /* subnormal: a = m * 2^(1 - bias - mant_bits) */
    uint32_t m = (uint32_t)ldexp(a, bias - 1 + mant_bits);
    return sign | (uint16_t)m;
}

uint16_t oracle_f64_to_f16(double x)
{
    if (isnan(x))
        return 0x7E00;
    double v = round_to_format(x, 11, -14, 65504.0);
    return encode_exact(v, 10, 15, 31);
}

uint16_t oracle_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double maxf = ldexp(255.0, 120);  /* (2 - 2^-7) * 2^127 */
    double v = round_to_format(x, 8, -126, maxf);
    return encode_exact(v, 7, 127, 255);
}

void oracle_round(const double *in, uint16_t *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == ORACLE_BF16 ? oracle_f64_to_bf16(in[i]) : oracle_f64_to_f16(in[i]);
}

/* ---- the GEMM ----------------------------------------------------------- */

/* One entry: R = sum_k a[k] * b[k] in order, S = sum_k |a[k] * b[k]|. */
static void dot(const double *a, const double *b, int64_t K, double *r, double *s)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = a[k] * b[k];
        acc += p;
        mag += fabs(p);
    }
    *r = acc;
    *s = mag;
}

/* Full product.  A: M x K and B: N x K row-major 16-bit patterns of `dtype`.
 * R and S: M x N row-major (S may be NULL).  Returns 0, or -1 on a bad
 * argument or when working memory cannot be had. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                int dtype, double *R, double *S)
{
    if (M < 0 || N < 0 || K < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return -1;
    if (M == 0 || N == 0)
        return 0;
    double *Ad = malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *Bd = malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -1;
    }
    oracle_decode(A, Ad, M * K, dtype);
    oracle_decode(B, Bd, N * K, dtype);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double r, s;
            dot(Ad + i * K, Bd + j * K, K, &r, &s);
            R[i * N + j] = r;
            if (S)
                S[i * N + j] = s;
        }
    }
    free(Ad);
    free(Bd);
    return 0;
}

/* Selected entries (rows[t], cols[t]) for t < n, of the same product; for
 * sizes whose full product is too slow on the host.  R[t], S[t] receive the
 * results (S may be NULL). */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                        int dtype, const int64_t *rows, const int64_t *cols, int64_t n,
                        double *R, double *S)
{
    if (M < 0 || N < 0 || K < 0 || n < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N)
            return -1;
    int fail = 0;
#pragma omp parallel
    {
        double *a = malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double *b = malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!a || !b) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t t = 0; t < n; ++t) {
                oracle_decode(A + rows[t] * K, a, K, dtype);
                oracle_decode(B + cols[t] * K, b, K, dtype);
                double r, s;
                dot(a, b, K, &r, &s);
                R[t] = r;
                if (S)
                    S[t] = s;
            }
        }
        free(a);
        free(b);
    }
    return fail ? -1 : 0;
}

/* The product of operands already decoded to binary64 (A: M x K, B: N x K
 * row-major), rows [row0, row0 + nrows) only; R: nrows x N.  Same entries,
 * same summation order as oracle_gemm.  Lets a timed sample of a large
 * workload measure the sums with the operands resident, decoded once. */
int oracle_gemm_decoded_rows(int64_t M, int64_t N, int64_t K, const double *Ad, const double *Bd,
                             int64_t row0, int64_t nrows, double *R)
{
    if (M < 0 || N < 0 || K < 0 || row0 < 0 || nrows < 0 || row0 + nrows > M)
        return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = row0; i < row0 + nrows; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double r, s;
            dot(Ad + i * K, Bd + j * K, K, &r, &s);
            R[(i - row0) * N + j] = r;
        }
    }
    return 0;
}

/* Rows [row0, row0 + nrows) of the product, all N columns; used to time a
 * bounded sample of a large workload.  R: nrows x N. */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                     int dtype, int64_t row0, int64_t nrows, double *R)
{
    if (row0 < 0 || nrows < 0 || row0 + nrows > M)
        return -1;
    return oracle_gemm(nrows, N, K, A + row0 * K, B, dtype, R, NULL);
}

/* ---- the pages' shared-memory bound and FLOP count ---------------------- */

/* num_stages * (A tile + B tile) bytes: the upper bound of the pipeline's
 * shared footprint before any reuse of storage. */
int64_t oracle_smem_bound(int64_t block_M, int64_t block_N, int64_t block_K, int64_t num_stages,
                          int64_t elem_bytes)
{
    int64_t a_tile = block_M * block_K * elem_bytes;
    int64_t b_tile = block_K * block_N * elem_bytes;
    return num_stages * (a_tile + b_tile);
}

/* Largest num_stages whose bound fits in `budget` bytes (0 if none). */
int64_t oracle_max_stages(int64_t block_M, int64_t block_N, int64_t block_K, int64_t elem_bytes,
                          int64_t budget)
{
    int64_t per = oracle_smem_bound(block_M, block_N, block_K, 1, elem_bytes);
    return per > 0 ? budget / per : 0;
}

double oracle_flops(int64_t M, int64_t N, int64_t K)
{
    return 2.0 * (double)M * (double)N * (double)K;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
