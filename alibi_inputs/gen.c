/*
 * Seeded synthetic input generator (shared by the oracle tests, the GPU tests
 * and the benchmark). It holds no attention arithmetic: random numbers and
 * storage-format rounding only.
 *
 * Stream (seed, sid), element n:
 *   key   = mix64((mix64(seed + G) ^ sid) + G)
 *   u64_n = mix64(key + (n + 1) G)            G = 0x9E3779B97F4A7C15
 *   u01_n = (u64_n >> 11) * 2^-53              uniform in [0, 1)
 * mix64 is the SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014).
 * Normal element n: Box-Muller, cosine branch, on u01_{2n} and u01_{2n+1}:
 *   sqrt(-2 log1p(-u01_{2n})) * cos(2 pi u01_{2n+1})   (fp64, then rounded to fp32)
 * Uniform element n on [lo, hi): lo + (hi - lo) u01_n.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t gen_stream_key(uint64_t seed, uint64_t sid)
{
    return mix64((mix64(seed + GOLDEN) ^ sid) + GOLDEN);
}

static inline double u01(uint64_t key, uint64_t n)
{
    return (double)(mix64(key + (n + 1) * GOLDEN) >> 11) * 0x1.0p-53;
}

typedef struct {
    uint64_t key, start, count;
    int kind; /* 0 normal, 1 uniform */
    double lo, hi, scale;
    float *out;
} job_t;

static void *run(void *arg)
{
    const job_t *j = (const job_t *)arg;
    const double two_pi = 6.283185307179586476925286766559;
    for (uint64_t e = 0; e < j->count; ++e) {
        const uint64_t n = j->start + e;
        double x;
        if (j->kind == 0) {
            const double a = u01(j->key, 2 * n), b = u01(j->key, 2 * n + 1);
            x = sqrt(-2.0 * log1p(-a)) * cos(two_pi * b) * j->scale;
        } else {
            x = j->lo + (j->hi - j->lo) * u01(j->key, n);
        }
        j->out[e] = (float)x;
    }
    return NULL;
}

static void dispatch(uint64_t key, uint64_t start, uint64_t count, int kind, double lo, double hi, double scale,
                     float *out, int nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if ((uint64_t)nthreads > count / 65536 + 1) nthreads = (int)(count / 65536 + 1);
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    uint64_t per = (count + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t s = (uint64_t)t * per;
        uint64_t c = s >= count ? 0 : (count - s < per ? count - s : per);
        jobs[t] = (job_t){key, start + s, c, kind, lo, hi, scale, out + s};
        if (nthreads == 1 || pthread_create(&th[t], NULL, run, &jobs[t]) != 0) {
            run(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
}

void gen_normal_f32(uint64_t seed, uint64_t sid, uint64_t start, uint64_t count, double scale, float *out,
                    int nthreads)
{
    dispatch(gen_stream_key(seed, sid), start, count, 0, 0.0, 0.0, scale, out, nthreads);
}

void gen_uniform_f32(uint64_t seed, uint64_t sid, uint64_t start, uint64_t count, double lo, double hi, float *out,
                     int nthreads)
{
    dispatch(gen_stream_key(seed, sid), start, count, 1, lo, hi, 1.0, out, nthreads);
}
