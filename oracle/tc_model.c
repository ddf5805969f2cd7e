/*
 * tc_model.c -- block-FMA model of a tensor-core dot product, for the oracle.
 *
 * TEST INFRASTRUCTURE ONLY, like tcg_oracle.c (whose decoders it uses): nothing on the
 * product path links, loads or calls it.
 *
 * What it computes ("NVIDIA Tensor Core混合精度计算原理与应用解析", section 2.2 and the
 * per-generation descriptions of section 4):
 *
 *  - The k products of a dot product are taken in k order in blocks of `block`
 *    consecutive products (the block FMA size N_FMA, section 2.2.2).  Each product of
 *    two inputs is exact.
 *  - One block and the running accumulator c are added as follows (section 2.2.1, the
 *    accumulator width and its alignment, and section 4.1, products kept unnormalised):
 *      * every nonzero term gets an alignment exponent: a product a*b gets ea + eb, the
 *        sum of its inputs' exponents (exp_sum = 1; a subnormal input counts with its
 *        format's smallest normal exponent), or the exponent of the product itself
 *        (exp_sum = 0); the accumulator gets its own exponent (the smallest FP32 normal
 *        exponent when it is subnormal);
 *      * e_max is the largest alignment exponent of the block's nonzero terms;
 *      * every term is cut toward zero to a multiple of 2^(e_max - frac) (section 2.3:
 *        intermediate results are truncated) -- frac = the accumulator's fraction bits
 *        plus its extra alignment bits, e.g. 22 for the 2+22-bit accumulator of
 *        section 4.1, 24 for the 2+23+1-bit one of section 4.2.1;
 *      * the cut terms are added exactly and the sum becomes the new FP32 accumulator,
 *        rounded toward zero (norm_rne = 0) or to nearest even (norm_rne = 1), FP32
 *        subnormals kept.
 *  - With K split into ranges (the library's split-K scheduling, not a step of the pages)
 *    every range of k_per_split products is accumulated on its own, from zero and with
 *    blocks counted from the range's start, and the range results are added in range
 *    order in FP32 (nearest even); that sum is the accumulator below.
 *  - The accumulator after the last block enters the GEMM's epilogue in FP32, as the
 *    library computes it: r = alpha * acc, then r = fma(beta, c, r) when beta != 0 (each
 *    rounded to nearest even in FP32; the order of these two roundings is the library's
 *    choice, the pages' wmma example writes alpha * acc + beta * c), then one
 *    round-to-nearest-even to the output type.  k == 0 or alpha == 0 give beta * c in
 *    FP32 (zero when beta == 0) without reading A or B.
 *  - Inf/NaN products make the block's result the IEEE sum of its non-finite terms
 *    (NaN for 0 * Inf or for Inf - Inf), which then stays in the accumulator.
 *
 * With block = k, a large frac and norm_rne = 1 nothing is cut and the accumulator is the
 * exact sum rounded once to nearest even; with alpha = 1, beta = 0 and an FP32 output
 * that is what orc_gemm computes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

enum { MD_F16 = 0, MD_BF16 = 1, MD_F32 = 2, MD_F8E4M3 = 3, MD_F8E5M2 = 4 };

double orc_f16_to_f64(uint16_t h);
double orc_bf16_to_f64(uint16_t b);
double orc_f8e4m3_to_f64(uint8_t b);
double orc_f8e5m2_to_f64(uint8_t b);
double orc_f32_to_f64(uint32_t u);
uint32_t orc_tf32_round_bits(uint32_t u);
uint16_t orc_f64_to_f16_rne(double x);
uint16_t orc_f64_to_bf16_rne(double x);

/* Smallest normal exponent of each input format. */
static int min_normal_exp(int type)
{
    switch (type) {
    case MD_F16: return -14;
    case MD_F8E4M3: return -6;
    case MD_F8E5M2: return -14;
    default: return -126;          /* BF16, FP32/TF32 */
    }
}

static double load(const void *base, int type, int64_t idx, int tf32)
{
    switch (type) {
    case MD_F16: return orc_f16_to_f64(((const uint16_t *)base)[idx]);
    case MD_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[idx]);
    case MD_F8E4M3: return orc_f8e4m3_to_f64(((const uint8_t *)base)[idx]);
    case MD_F8E5M2: return orc_f8e5m2_to_f64(((const uint8_t *)base)[idx]);
    default: {
        uint32_t u = ((const uint32_t *)base)[idx];
        return orc_f32_to_f64(tf32 ? orc_tf32_round_bits(u) : u);
    }
    }
}

/* floor(log2|x|) of a finite nonzero double (exact, through frexp). */
static int exponent_of(double x)
{
    int e;
    frexp(x, &e);
    return e - 1;
}

/* Alignment exponent of a nonzero finite input x of format `type`. */
static int input_exp(double x, int type)
{
    int emin = min_normal_exp(type);
    if (fabs(x) < ldexp(1.0, emin))
        return emin;                              /* subnormal: 0.m x 2^emin */
    return exponent_of(x);
}

typedef __int128 i128;
typedef unsigned __int128 u128;

static int bitlen(u128 u)
{
    int n = 0;
    while (u) {
        u >>= 1;
        ++n;
    }
    return n;
}

/* s * 2^q as an FP32 value: round toward zero or to nearest even, subnormals kept. */
static float to_fp32(i128 s, int q, int rne)
{
    if (s == 0)
        return 0.0f;
    int neg = s < 0;
    u128 u = neg ? (u128)(-s) : (u128)s;
    int e = bitlen(u) - 1 + q;                    /* exponent of the leading bit */
    int qe = e >= -126 ? e - 23 : -149;           /* FP32 quantum at that exponent */
    double v;
    if (qe > q) {
        int shift = qe - q;
        u128 keep = u >> shift;
        u128 rem = u - (keep << shift);
        if (rne) {
            u128 half = (u128)1 << (shift - 1);
            if (rem > half || (rem == half && (keep & 1)))
                keep += 1;
        }
        v = ldexp((double)keep, qe);              /* keep < 2^25: exact */
    } else {
        v = ldexp((double)u, q);                  /* u has <= 24 significant bits */
    }
    if (v >= 0x1p128)
        v = rne ? INFINITY : (double)3.4028234663852886e38;   /* overflow: Inf or FLT_MAX */
    return (float)(neg ? -v : v);
}

/* One accumulator: the block-FMA sum of a[0..k) * b[0..k) (ea, eb: alignment exponents
 * of the inputs).  Returns the FP32 accumulator. */
static float model_dot(const double *a, const int *ea, const double *b, const int *eb,
                       int64_t k, int block, int frac, int norm_rne, int exp_sum)
{
    float c = 0.0f;                                   /* the FP32 accumulator */
    for (int64_t k0 = 0; k0 < k; k0 += block) {
        int64_t k1 = k0 + block < k ? k0 + block : k;
        double t[1024];
        int et[1024];
        int nt = 0, nonfinite = 0;
        double special = 0.0;                         /* IEEE sum of the non-finite terms */
        if (isfinite(c) == 0) {
            nonfinite = 1;
            special = c;
        }
        for (int64_t p = k0; p < k1; ++p) {
            double prod = a[p] * b[p];                /* exact: <= 11-bit significands */
            if (!isfinite(a[p]) || !isfinite(b[p]) || !isfinite(prod)) {
                special = nonfinite ? special + prod : prod;
                nonfinite = 1;
                continue;
            }
            if (prod == 0.0)
                continue;                             /* a zero product has no exponent */
            t[nt] = prod;
            et[nt] = exp_sum ? ea[p] + eb[p] : exponent_of(prod);
            ++nt;
        }
        if (nonfinite) {
            c = (float)special;
            continue;
        }
        if (c != 0.0f) {
            t[nt] = c;
            et[nt] = fabs(c) < 0x1p-126 ? -126 : exponent_of(c);
            ++nt;
        }
        if (nt == 0)
            continue;                                 /* nothing to add: c stays */
        int emax = et[0];
        for (int r = 1; r < nt; ++r)
            if (et[r] > emax)
                emax = et[r];
        int q = emax - frac;                          /* the cut: multiples of 2^q */
        i128 s = 0;
        for (int r = 0; r < nt; ++r)
            s += (i128)trunc(ldexp(t[r], -q));        /* toward zero, exact below 2^63 */
        c = to_fp32(s, q, norm_rne);
    }
    return c;
}

typedef struct {
    int64_t k;
    float alpha, beta;
    const void *C; int ctype; int64_t ldc;
    int64_t i0, i1, j0;
    void *D; int64_t ldd;
    const double *opA, *opB;                          /* decoded rows of op(A), columns of op(B) */
    const int *expA, *expB;
    int block, frac, norm_rne, exp_sum, splits;
    int64_t k_per_split;
    int64_t jstart, jstop;                            /* this worker's columns (relative) */
} model_job;

static float load_c32(const void *C, int ctype, int64_t idx)
{
    switch (ctype) {
    case MD_F16: return (float)orc_f16_to_f64(((const uint16_t *)C)[idx]);
    case MD_BF16: return (float)orc_bf16_to_f64(((const uint16_t *)C)[idx]);
    default: return ((const float *)C)[idx];
    }
}

static void store_out(void *D, int ctype, int64_t idx, float r)
{
    switch (ctype) {
    case MD_F16: ((uint16_t *)D)[idx] = orc_f64_to_f16_rne((double)r); break;
    case MD_BF16: ((uint16_t *)D)[idx] = orc_f64_to_bf16_rne((double)r); break;
    default: ((float *)D)[idx] = r; break;
    }
}

static void *model_worker(void *arg)
{
    model_job *g = (model_job *)arg;
    int64_t rows = g->i1 - g->i0;
    int no_product = (g->k == 0 || g->alpha == 0.0f);
    for (int64_t jj = g->jstart; jj < g->jstop; ++jj) {
        int64_t j = g->j0 + jj;
        for (int64_t ii = 0; ii < rows; ++ii) {
            int64_t i = g->i0 + ii;
            float r;
            if (no_product) {
                r = g->beta == 0.0f ? 0.0f : g->beta * load_c32(g->C, g->ctype, i + j * g->ldc);
            } else {
                float acc = 0.0f;
                for (int s = 0; s < g->splits; ++s) {
                    int64_t p0 = s * g->k_per_split;
                    int64_t p1 = p0 + g->k_per_split < g->k ? p0 + g->k_per_split : g->k;
                    float part = model_dot(g->opA + ii * g->k + p0, g->expA + ii * g->k + p0,
                                           g->opB + jj * g->k + p0, g->expB + jj * g->k + p0,
                                           p1 - p0, g->block, g->frac, g->norm_rne,
                                           g->exp_sum);
                    acc = s == 0 ? part : acc + part;        /* FP32, nearest even */
                }
                r = g->alpha * acc;                                   /* FP32, nearest even */
                if (g->beta != 0.0f)
                    r = fmaf(g->beta, load_c32(g->C, g->ctype, i + j * g->ldc), r);
            }
            store_out(g->D, g->ctype, ii + jj * g->ldd, r);
        }
    }
    return NULL;
}

/*
 * orc_gemm_model: block [i0,i1) x [j0,j1) of D = alpha*op(A)*op(B) + beta*C with the
 * accumulator of the block-FMA model and the epilogue described at the top; arguments as
 * orc_gemm (column-major, BLAS style), plus the model's parameters and the K split
 * (splits = 1: none; else ranges of k_per_split, the last one non-empty).  frac must be at most 60 and block at most 1023
 * (the cut terms of a block are summed as 128-bit integers).  Returns 0, -1 on bad
 * arguments, -2 on allocation failure.
 */
int orc_gemm_model(int transa, int transb, int64_t m, int64_t n, int64_t k, double alpha,
                   const void *A, int atype, int64_t lda, const void *B, int btype, int64_t ldb,
                   double beta, const void *C, int ctype, int64_t ldc, int tf32, int64_t i0,
                   int64_t i1, int64_t j0, int64_t j1, void *D, int64_t ldd, int block, int frac,
                   int norm_rne, int exp_sum, int splits, int64_t k_per_split, int nthreads)
{
    if (m < 0 || n < 0 || k < 0 || i0 < 0 || i1 > m || i0 > i1 || j0 < 0 || j1 > n ||
        j0 > j1 || ldd < i1 - i0 || block < 1 || block > 1023 || frac < 0 || frac > 60 ||
        splits < 1 || (splits > 1 && (k_per_split < 1 || (splits - 1) * k_per_split >= k)))
        return -1;
    if (splits == 1)
        k_per_split = k;
    int64_t rows = i1 - i0, cols = j1 - j0;
    if (rows == 0 || cols == 0)
        return 0;
    float alphaf = (float)alpha, betaf = (float)beta;      /* the library takes FP32 scalars */
    int no_product = (k == 0 || alphaf == 0.0f);
    double *opA = NULL, *opB = NULL;
    int *expA = NULL, *expB = NULL;
    if (!no_product) {
        opA = (double *)malloc(sizeof(double) * (size_t)(rows * k));
        opB = (double *)malloc(sizeof(double) * (size_t)(cols * k));
        expA = (int *)malloc(sizeof(int) * (size_t)(rows * k));
        expB = (int *)malloc(sizeof(int) * (size_t)(cols * k));
        if (!opA || !opB || !expA || !expB) {
            free(opA); free(opB); free(expA); free(expB);
            return -2;
        }
        for (int64_t ii = 0; ii < rows; ++ii)
            for (int64_t p = 0; p < k; ++p) {
                int64_t i = i0 + ii;
                double v = load(A, atype, transa == 0 ? i + p * lda : p + i * lda, tf32);
                opA[ii * k + p] = v;
                expA[ii * k + p] = (v != 0.0 && isfinite(v)) ? input_exp(v, atype) : 0;
            }
        for (int64_t jj = 0; jj < cols; ++jj)
            for (int64_t p = 0; p < k; ++p) {
                int64_t j = j0 + jj;
                double v = load(B, btype, transb == 0 ? p + j * ldb : j + p * ldb, tf32);
                opB[jj * k + p] = v;
                expB[jj * k + p] = (v != 0.0 && isfinite(v)) ? input_exp(v, btype) : 0;
            }
    }
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > cols)
        nthreads = (int)cols;
    model_job *jobs = (model_job *)calloc((size_t)nthreads, sizeof(model_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th); free(opA); free(opB); free(expA); free(expB);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        model_job *g = &jobs[t];
        g->k = k; g->alpha = alphaf; g->beta = betaf;
        g->C = C; g->ctype = ctype; g->ldc = ldc;
        g->i0 = i0; g->i1 = i1; g->j0 = j0;
        g->D = D; g->ldd = ldd;
        g->opA = opA; g->opB = opB; g->expA = expA; g->expB = expB;
        g->block = block; g->frac = frac; g->norm_rne = norm_rne; g->exp_sum = exp_sum;
        g->splits = splits; g->k_per_split = k_per_split;
        g->jstart = cols * t / nthreads;
        g->jstop = cols * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, model_worker, &jobs[t]);
    model_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(jobs); free(th); free(opA); free(opB); free(expA); free(expB);
    return 0;
}
