/*
 * tcg_oracle.c -- CPU oracle for the mixed-precision tensor-core GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only tests/, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   D = alpha * op(A) * op(B) + beta * C            (column-major, BLAS style)
 *
 *  - "Programming Tensor Cores in CUDA 9", section "CUDA 9.0 中张量核的编程访问"
 *    (the wmma_example kernel): alpha/beta epilogue applied elementwise to the
 *    accumulated product, column-major storage with leading dimensions.
 *  - same page, section "什么是张量核?" and Figure 2: FP16 inputs, full-precision
 *    (exact) products, accumulation in FP32.  The oracle accumulates the exact
 *    products in FP64, i.e. it computes the exact sum up to FP64 rounding (each
 *    product of two <=11-bit significands is exact in FP64).
 *  - same page, section "如何在 cuBLAS 中使用张量核" (the cublasGemmEx call):
 *    the argument list m, n, k, alpha, A/lda, B/ldb, beta, C/ldc with transa and
 *    transb; C is overwritten by D.
 *  - "CUDA Handbook, 17.5 Tensor Cores": in TF32 mode an FP32 input is rounded
 *    to TF32 (8-bit exponent, 10-bit mantissa) before it enters the product.
 *    The rounding is taken as round-to-nearest-even; Inf and NaN pass through.
 *  - "NVIDIA Tensor Core混合精度计算原理与应用解析", section 2.3: round-to-
 *    nearest-even at the final output.  The oracle rounds once, from FP64, to
 *    the output type (FP32, FP16 or BF16).
 *  - BLAS convention for the degenerate cases: k == 0 or alpha == 0 gives
 *    D = beta * C and A, B are not read; beta == 0 means C is not read.
 *
 * Formats (decoded here with this file's own bit arithmetic):
 *  - FP16: 1 sign, 5 exponent, 10 mantissa bits, bias 15, subnormals
 *    ("Mixed-Precision Programming with CUDA 8", Figure 1).
 *  - BF16: 1 sign, 8 exponent, 7 mantissa bits, bias 127 (the upper half of an
 *    IEEE binary32; the pages name the type without defining it).
 *  - FP32: IEEE binary32.
 *  - FP8 E4M3: 1 sign, 4 exponent, 3 mantissa bits, bias 7, subnormals, no
 *    infinities, S.1111.111 is NaN (largest finite 448); FP8 E5M2: 1 sign, 5
 *    exponent, 2 mantissa bits, bias 15, subnormals, IEEE-style Inf/NaN ("NVIDIA
 *    Tensor Core混合精度计算原理与应用解析", section 4.3.1: the two FP8 formats, E4M3
 *    with the smaller range and higher precision, E5M2 the other way round; the
 *    pages give no bit layouts, these are the standard ones).
 */
#include <math.h>
#include <fenv.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_F8E4M3 = 3, ORC_F8E5M2 = 4 };
enum { ORC_OP_N = 0, ORC_OP_T = 1 };

/* ------------------------------------------------------------------------ */
/* Decoding                                                                 */
/* ------------------------------------------------------------------------ */

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-14 * 2^-10 */
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

double orc_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0xFF)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -133);             /* f * 2^-126 * 2^-7 */
    else
        v = ldexp((double)(128 + f), e - 134);  /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

double orc_f8e4m3_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int f = b & 0x7;
    double v;
    if (e == 0xF && f == 0x7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);               /* f * 2^-6 * 2^-3 */
    else
        v = ldexp((double)(8 + f), e - 10);     /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

double orc_f8e5m2_to_f64(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1F;
    int f = b & 0x3;
    double v;
    if (e == 0x1F)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -16);              /* f * 2^-14 * 2^-2 */
    else
        v = ldexp((double)(4 + f), e - 17);     /* (1 + f/4) * 2^(e-15) */
    return sign ? -v : v;
}

double orc_f32_to_f64(uint32_t u)
{
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* ------------------------------------------------------------------------ */
/* Rounding (round to nearest, ties to even)                                */
/* ------------------------------------------------------------------------ */

/* Round a finite, non-negative x to the nearest multiple of 2^(E - mbits),
 * E = max(floor(log2 x), emin), ties to even.  x / q is exact (q is a power of
 * two) and nearbyint rounds ties to even under the default rounding mode. */
static double round_to_quantum(double x, int mbits, int emin)
{
    if (x == 0.0)
        return 0.0;
    int e2;
    frexp(x, &e2);          /* x = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;         /* floor(log2 x) */
    if (E < emin)
        E = emin;
    double q = ldexp(1.0, E - mbits);
    return nearbyint(x / q) * q;
}

/* FP32 bits -> TF32 value kept in FP32 bits (low 13 mantissa bits zero). */
uint32_t orc_tf32_round_bits(uint32_t u)
{
    float x;
    memcpy(&x, &u, sizeof x);
    if (isnan(x))
        return (u & 0x80000000u) | 0x7FC00000u;          /* quiet NaN */
    if (isinf(x))
        return u;
    double a = fabs((double)x);
    double r = round_to_quantum(a, 10, -126);             /* 10 mantissa bits */
    if (r >= ldexp(1.0, 128))
        r = INFINITY;                                     /* past the TF32 max */
    float y = (float)r;                                   /* exact */
    uint32_t v;
    memcpy(&v, &y, sizeof v);
    return v | (u & 0x80000000u);
}

uint16_t orc_f64_to_f16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return sign | 0x7E00;
    double a = fabs(x);
    double r = round_to_quantum(a, 10, -14);
    if (r >= 65536.0)                                     /* 2^16: past 65504 */
        return sign | 0x7C00;
    if (r < ldexp(1.0, -14))                              /* subnormal or zero */
        return sign | (uint16_t)(r * ldexp(1.0, 24));
    int e2;
    double f = frexp(r, &e2);                             /* r = f * 2^e2 */
    int E = e2 - 1;
    uint16_t mant = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | mant;
}

uint16_t orc_f64_to_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return sign | 0x7FC0;
    double a = fabs(x);
    double r = round_to_quantum(a, 7, -126);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float y = (float)r;                                   /* exact */
    uint32_t v;
    memcpy(&v, &y, sizeof v);
    return sign | (uint16_t)(v >> 16);
}

float orc_f64_to_f32_rne(double x)
{
    return (float)x;     /* C conversion under the default (nearest-even) mode */
}

/* Element loads in the three storage types. */
static double load_elem(const void *base, int type, int64_t idx, int tf32)
{
    switch (type) {
    case ORC_F16:
        return orc_f16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_BF16:
        return orc_bf16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_F8E4M3:
        return orc_f8e4m3_to_f64(((const uint8_t *)base)[idx]);
    case ORC_F8E5M2:
        return orc_f8e5m2_to_f64(((const uint8_t *)base)[idx]);
    default: {
        uint32_t u = ((const uint32_t *)base)[idx];
        return orc_f32_to_f64(tf32 ? orc_tf32_round_bits(u) : u);
    }
    }
}

static void store_elem(void *base, int type, int64_t idx, double r)
{
    switch (type) {
    case ORC_F16:
        ((uint16_t *)base)[idx] = orc_f64_to_f16_rne(r);
        break;
    case ORC_BF16:
        ((uint16_t *)base)[idx] = orc_f64_to_bf16_rne(r);
        break;
    default:
        ((float *)base)[idx] = orc_f64_to_f32_rne(r);
        break;
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    int transa, transb;
    int64_t m, n, k;
    double alpha, beta;
    const void *A; int atype; int64_t lda;
    const void *B; int btype; int64_t ldb;
    const void *C; int ctype; int64_t ldc;
    int tf32;
    int64_t i0, i1, j0, j1;   /* block of D to compute: rows [i0,i1), cols [j0,j1) */
    void *D; int64_t ldd;      /* output block, column-major, in ctype */
    double *R;                 /* optional: alpha*S + beta*C in FP64 */
    double *absAB;             /* optional: sum_p |a_ip| |b_pj| */
    double *opA;               /* decoded op(A) rows i0..i1, row-major, k per row */
    double *opB;               /* decoded op(B) cols j0..j1, column-major, k per col */
    int64_t jstart, jstop;     /* this worker's columns (relative) */
} gemm_job;

static void *gemm_worker(void *arg)
{
    gemm_job *g = (gemm_job *)arg;
    int64_t rows = g->i1 - g->i0;
    int no_product = (g->k == 0 || g->alpha == 0.0);
    for (int64_t jj = g->jstart; jj < g->jstop; ++jj) {
        const double *bcol = g->opB + jj * g->k;
        int64_t j = g->j0 + jj;
        for (int64_t ii = 0; ii < rows; ++ii) {
            int64_t i = g->i0 + ii;
            double s = 0.0, sabs = 0.0;
            if (!no_product) {
                const double *arow = g->opA + ii * g->k;
                for (int64_t p = 0; p < g->k; ++p) {     /* S_ij = sum_p a_ip b_pj */
                    s += arow[p] * bcol[p];
                    sabs += fabs(arow[p]) * fabs(bcol[p]);
                }
            }
            double r;
            if (g->beta == 0.0) {                         /* C is not read */
                r = no_product ? 0.0 : g->alpha * s;
            } else {
                double c = load_elem(g->C, g->ctype, i + j * g->ldc, 0);
                r = no_product ? g->beta * c : g->alpha * s + g->beta * c;
            }
            int64_t o = ii + jj * g->ldd;
            store_elem(g->D, g->ctype, o, r);             /* one RNE to the output type */
            if (g->R)
                g->R[o] = r;
            if (g->absAB)
                g->absAB[o] = sabs;
        }
    }
    return NULL;
}

/*
 * orc_gemm: block [i0,i1) x [j0,j1) of D = alpha*op(A)*op(B) + beta*C.
 * A, B, C are the caller's full column-major arrays; D (and R, absAB if not
 * NULL) receive the block, column-major with leading dimension ldd.
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int orc_gemm(int transa, int transb, int64_t m, int64_t n, int64_t k,
             double alpha, const void *A, int atype, int64_t lda,
             const void *B, int btype, int64_t ldb,
             double beta, const void *C, int ctype, int64_t ldc,
             int tf32, int64_t i0, int64_t i1, int64_t j0, int64_t j1,
             void *D, int64_t ldd, double *R, double *absAB, int nthreads)
{
    if (m < 0 || n < 0 || k < 0 || i0 < 0 || i1 > m || i0 > i1 || j0 < 0 || j1 > n ||
        j0 > j1 || ldd < i1 - i0)
        return -1;
    int64_t rows = i1 - i0, cols = j1 - j0;
    if (rows == 0 || cols == 0)
        return 0;
    int no_product = (k == 0 || alpha == 0.0);
    double *opA = NULL, *opB = NULL;
    if (!no_product) {
        opA = (double *)malloc(sizeof(double) * (size_t)(rows * k));
        opB = (double *)malloc(sizeof(double) * (size_t)(cols * k));
        if (!opA || !opB) {
            free(opA);
            free(opB);
            return -2;
        }
        /* op(A)[i][p] = A[i + p*lda] (N) or A[p + i*lda] (T) */
        for (int64_t ii = 0; ii < rows; ++ii)
            for (int64_t p = 0; p < k; ++p) {
                int64_t i = i0 + ii;
                int64_t idx = transa == ORC_OP_N ? i + p * lda : p + i * lda;
                opA[ii * k + p] = load_elem(A, atype, idx, tf32);
            }
        /* op(B)[p][j] = B[p + j*ldb] (N) or B[j + p*ldb] (T) */
        for (int64_t jj = 0; jj < cols; ++jj)
            for (int64_t p = 0; p < k; ++p) {
                int64_t j = j0 + jj;
                int64_t idx = transb == ORC_OP_N ? p + j * ldb : j + p * ldb;
                opB[jj * k + p] = load_elem(B, btype, idx, tf32);
            }
    }
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > cols)
        nthreads = (int)cols;
    gemm_job *jobs = (gemm_job *)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th); free(opA); free(opB);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        gemm_job *g = &jobs[t];
        g->transa = transa; g->transb = transb;
        g->m = m; g->n = n; g->k = k; g->alpha = alpha; g->beta = beta;
        g->A = A; g->atype = atype; g->lda = lda;
        g->B = B; g->btype = btype; g->ldb = ldb;
        g->C = C; g->ctype = ctype; g->ldc = ldc;
        g->tf32 = tf32;
        g->i0 = i0; g->i1 = i1; g->j0 = j0; g->j1 = j1;
        g->D = D; g->ldd = ldd; g->R = R; g->absAB = absAB;
        g->opA = opA; g->opB = opB;
        g->jstart = cols * t / nthreads;
        g->jstop = cols * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
    gemm_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(jobs); free(th); free(opA); free(opB);
    return 0;
}

/* Array forms of the scalar routines, for the Python wrapper and its pins. */
void orc_f16_to_f64_array(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(in[i]);
}
void orc_bf16_to_f64_array(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}
void orc_f8e4m3_to_f64_array(const uint8_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f8e4m3_to_f64(in[i]);
}
void orc_f8e5m2_to_f64_array(const uint8_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f8e5m2_to_f64(in[i]);
}
void orc_tf32_round_bits_array(const uint32_t *in, uint32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_tf32_round_bits(in[i]);
}
void orc_f64_to_f16_array(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f16_rne(in[i]);
}
void orc_f64_to_bf16_array(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16_rne(in[i]);
}
void orc_f64_to_f32_array(const double *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f32_rne(in[i]);
}
