/*
 * synth.c -- seeded, counter-based synthetic inputs.
 *
 * Shared by the tests, the benchmark and the CPU oracle's callers.  It holds
 * none of the quantisation or GEMM arithmetic: only random numbers, their
 * rounding to BF16 input tensors, and the expert-routing scores that decide
 * how MoE rows are grouped.
 *
 * Generator: element i of stream `key` is mix64(key + (i + 1) * 0x9E3779B97F4A7C15),
 * where mix64 is the SplitMix64 output function (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).  A uniform
 * in (0, 1) takes the top 53 bits plus one half.  Normals use the
 * Box-Muller transform on consecutive pairs (even index: cos, odd: sin).
 * Student-t(df) is Z / sqrt(chi2_df / df) with chi2_df a sum of df squared
 * normals from a second stream.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t syn_mix64(uint64_t z) { return mix64(z); }

uint64_t syn_u64(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

double syn_uniform(uint64_t key, uint64_t i)
{
    return ((double)(syn_u64(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

double syn_normal(uint64_t key, uint64_t i)
{
    uint64_t p = i >> 1;
    double u1 = syn_uniform(key, 2 * p), u2 = syn_uniform(key, 2 * p + 1);
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

static inline uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lower = u & 0xFFFFu, upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1;
    return (uint16_t)upper;
}

/* kind 0: sigma * Z
 * kind 1: sigma * Z, times `factor` where uniform(key2, i) < p (outliers)
 * kind 2: sigma * Student-t(df = (int)p) with the chi-square from key2 */
typedef struct {
    int kind;
    uint64_t key, key2;
    uint64_t start;
    int64_t n;
    double sigma, p, factor;
    uint16_t *out_bf16;
    float *out_f32;
    int t, nt;
} gen_job;

static double gen_value(const gen_job *j, uint64_t i)
{
    double z = syn_normal(j->key, i);
    if (j->kind == 1) {
        if (syn_uniform(j->key2, i) < j->p)
            z *= j->factor;
    } else if (j->kind == 2) {
        int df = (int)j->p;
        double chi = 0.0;
        for (int d = 0; d < df; ++d) {
            double w = syn_normal(j->key2, i * (uint64_t)df + (uint64_t)d);
            chi += w * w;
        }
        z = z / sqrt(chi / (double)df);
    }
    return j->sigma * z;
}

static void *gen_main(void *p)
{
    gen_job *j = (gen_job *)p;
    int64_t per = (j->n + j->nt - 1) / j->nt;
    int64_t a = (int64_t)j->t * per, b = a + per < j->n ? a + per : j->n;
    for (int64_t k = a; k < b; ++k) {
        float f = (float)gen_value(j, j->start + (uint64_t)k);
        if (j->out_bf16)
            j->out_bf16[k] = f32_to_bf16_rne(f);
        if (j->out_f32)
            j->out_f32[k] = f;
    }
    return NULL;
}

static void run_gen(gen_job proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    gen_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].t = t;
        jobs[t].nt = nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, gen_main, &jobs[t]);
    gen_main(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
}

/* Fill out[k] (BF16 bits) and/or outf[k] (FP32) for k in [0, n), element
 * index start + k of the chosen distribution. */
void syn_fill(int kind, uint64_t key, uint64_t key2, uint64_t start, int64_t n,
              double sigma, double p, double factor, uint16_t *out_bf16, float *out_f32,
              int nthreads)
{
    gen_job j;
    memset(&j, 0, sizeof j);
    j.kind = kind;
    j.key = key;
    j.key2 = key2;
    j.start = start;
    j.n = n;
    j.sigma = sigma;
    j.p = p;
    j.factor = factor;
    j.out_bf16 = out_bf16;
    j.out_f32 = out_f32;
    run_gen(j, nthreads);
}

/* Routing scores for synthetic MoE grouping: logits[t][e] = sum_d x[t][d] * c[e][d]
 * in double, x given as BF16 bits [T][D], c as FP32 [E][D].  Plain loops in a
 * fixed order so that every machine forms the same groups. */
typedef struct {
    const uint16_t *x;
    const float *c;
    int64_t T, D, E;
    double *logits;
    int t, nt;
} lg_job;

static void *lg_main(void *p)
{
    lg_job *j = (lg_job *)p;
    for (int64_t t = j->t; t < j->T; t += j->nt) {
        for (int64_t e = 0; e < j->E; ++e) {
            double acc = 0.0;
            for (int64_t d = 0; d < j->D; ++d) {
                uint32_t u = (uint32_t)j->x[t * j->D + d] << 16;
                float xf;
                memcpy(&xf, &u, 4);
                acc += (double)xf * (double)j->c[e * j->D + d];
            }
            j->logits[t * j->E + e] = acc;
        }
    }
    return NULL;
}

void syn_route_logits(const uint16_t *x, const float *c, int64_t T, int64_t D, int64_t E,
                      double *logits, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    lg_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        lg_job j = {x, c, T, D, E, logits, t, nthreads};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, lg_main, &jobs[t]);
    lg_main(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
}
