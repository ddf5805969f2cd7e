/*
 * Exhaustive check of a TF32 rounding routine over all 2^32 FP32 bit patterns
 * against a second, independent formulation written here with integer bit
 * arithmetic only:
 *
 *   finite x:  add 0x0FFF plus bit 13 of the pattern, then clear the low 13
 *              bits (round to nearest on the 13 dropped bits, ties to even; a
 *              carry into the exponent field is the correct next binade, and
 *              the largest finite values carry into the Inf pattern);
 *   Inf:       unchanged;
 *   NaN:       any NaN is accepted (compared by class).
 *
 * The routine under test (the oracle's) uses FP64 quantum arithmetic instead.
 * Test code only.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef uint32_t (*round_fn)(uint32_t);

static uint32_t tf32_by_bits(uint32_t u)
{
    return (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
}

static int is_nan_bits(uint32_t u)
{
    return (u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0;
}

typedef struct {
    round_fn fn;
    uint64_t lo, hi;
    uint64_t mismatches;
    uint32_t first_bad;
} job_t;

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    for (uint64_t x = j->lo; x < j->hi; ++x) {
        uint32_t u = (uint32_t)x;
        uint32_t got = j->fn(u);
        int ok;
        if (is_nan_bits(u))
            ok = is_nan_bits(got) && is_nan_bits(got & 0xFFFFE000u);  /* NaN survives truncation */
        else
            ok = got == tf32_by_bits(u);
        if (!ok) {
            if (j->mismatches == 0)
                j->first_bad = u;
            ++j->mismatches;
        }
    }
    return NULL;
}

/* Returns the number of mismatching patterns; *first_bad gets the first one. */
uint64_t tf32_exhaustive_mismatches(round_fn fn, int nthreads, uint32_t *first_bad)
{
    if (nthreads < 1)
        nthreads = 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    const uint64_t total = 1ull << 32;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].lo = total * (uint64_t)t / (uint64_t)nthreads;
        jobs[t].hi = total * (uint64_t)(t + 1) / (uint64_t)nthreads;
        pthread_create(&th[t], NULL, worker, &jobs[t]);
    }
    uint64_t bad = 0;
    *first_bad = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].mismatches && bad == 0)
            *first_bad = jobs[t].first_bad;
        bad += jobs[t].mismatches;
    }
    free(jobs);
    free(th);
    return bad;
}
