/*
 * sampler_norm_oracle.c -- the float64 CPU oracle for the kernels that sit
 * beside the MoE layer in a denoising step: RMSNorm, the Categorical entropy
 * of the vocabulary logits, and the Gumbel-max sampler with its argmax.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load this library.  It shares no
 * code, header, table or constant with the CUDA library, and neither side
 * includes or links the other.
 *
 * Sources (page title -- section):
 *   [NORM] "dg-w4-kernels" -- RMSNorm: y = x / sqrt(mean(x^2) + eps) * weight
 *          in one kernel; "Inference: Making every denoising pass fast" --
 *          RMSNorm: each activation rescaled by its root-mean-square
 *          magnitude, checked with a relative-error tolerance.
 *   [ENT]  "dg-w4-kernels" -- Sampler: fused_entropy returns the entropy in
 *          nats of Categorical(logits) over the last axis, [256, 262144] fp32,
 *          in one streaming pass.
 *   [GUM]  same section: gumbel_argmax_sample(logits, seed) returns a sample
 *          of Categorical(logits) by the Gumbel-max trick and the plain argmax
 *          from the same pass; the noise is Philox generated inline.
 *   [PHX]  Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw,
 *          "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011): four
 *          32-bit counter words, two key words, ten rounds of two 32x32->64
 *          multiplications with the round constants below, the key bumped by
 *          the two Weyl constants between rounds.
 *
 * Readings where the pages are silent (each is repeated at its function):
 *   S1 entropy of a row is -sum_i p_i ln p_i with p = softmax(row); terms with
 *      p_i = 0 (a logit of -inf) contribute 0.  A row needs one finite logit.
 *   S2 noise for row t, column i under (seed, offset): Philox4x32-10 with key
 *      (seed low word, seed high word) and counter (i / 4, t, offset low word,
 *      offset high word); column i takes output word i % 4.
 *   S3 a 32-bit word r becomes v = (r + 1/2) / 2^32 in (0, 1), the
 *      exponential variate E = -ln(1 - v) and the Gumbel variate g = -ln(E).
 *   S4 sample = argmax_i (logit_i + g_i), argmax = argmax_i logit_i, ties to
 *      the lower index in both.
 *   S5 RMSNorm: x and weight are bf16, the result is rounded to bf16 once;
 *      the oracle returns it unrounded (float64).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bfloat16: the high half of a binary32 pattern. */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* [NORM] y = x / sqrt(mean(x^2) + eps) * weight, per row, in float64 (S5).  */
/* ------------------------------------------------------------------------ */
void oracle_rmsnorm(const uint16_t *x, const uint16_t *weight, int M, int d, double eps,
                    double *y)
{
    for (int t = 0; t < M; t++) {
        const uint16_t *row = x + (int64_t)t * d;
        double ss = 0.0;
        for (int c = 0; c < d; c++) {
            const double v = bf16_value(row[c]);
            ss += v * v;
        }
        const double inv = 1.0 / sqrt(ss / d + eps);
        for (int c = 0; c < d; c++)
            y[(int64_t)t * d + c] = bf16_value(row[c]) * inv * bf16_value(weight[c]);
    }
}

/* ------------------------------------------------------------------------ */
/* [PHX] Philox4x32-10.                                                      */
/* ------------------------------------------------------------------------ */
#define PHX_MUL_A 0xD2511F53u   /* multiplies counter word 0 */
#define PHX_MUL_B 0xCD9E8D57u   /* multiplies counter word 2 */
#define PHX_WEYL_A 0x9E3779B9u  /* added to key word 0 after each round */
#define PHX_WEYL_B 0xBB67AE85u  /* added to key word 1 after each round */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        const uint64_t pa = (uint64_t)PHX_MUL_A * c[0];
        const uint64_t pb = (uint64_t)PHX_MUL_B * c[2];
        const uint32_t a_hi = (uint32_t)(pa >> 32), a_lo = (uint32_t)pa;
        const uint32_t b_hi = (uint32_t)(pb >> 32), b_lo = (uint32_t)pb;
        const uint32_t n0 = b_hi ^ c[1] ^ k0;
        const uint32_t n1 = b_lo;
        const uint32_t n2 = a_hi ^ c[3] ^ k1;
        const uint32_t n3 = a_lo;
        c[0] = n0;
        c[1] = n1;
        c[2] = n2;
        c[3] = n3;
        k0 += PHX_WEYL_A;
        k1 += PHX_WEYL_B;
    }
    out[0] = c[0];
    out[1] = c[1];
    out[2] = c[2];
    out[3] = c[3];
}

/* The 32-bit word of row t, column i (S2). */
uint32_t oracle_noise_word(uint64_t seed, uint64_t offset, int64_t t, int64_t i)
{
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    const uint32_t ctr[4] = {(uint32_t)(i / 4), (uint32_t)t, (uint32_t)offset,
                             (uint32_t)(offset >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(ctr, key, r);
    return r[i % 4];
}

/* The Gumbel variate of a word (S3), in float64. */
double oracle_gumbel_of_word(uint32_t r)
{
    const double v = ((double)r + 0.5) / 4294967296.0;
    const double e = -log1p(-v);
    return -log(e);
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: rows are independent, each row's arithmetic is done  */
/* by one thread in column order, so results do not depend on the threads.   */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *logits;
    int64_t V;
    int t0, t1;
    uint64_t seed, offset;
    double *H;
    int64_t *sample, *amax;
    double *best, *second;
} row_job;

/* [ENT] S1: -sum p ln p over one row, p = softmax(row), in float64. */
static double row_entropy(const float *l, int64_t V)
{
    double mx = -INFINITY;
    for (int64_t i = 0; i < V; i++)
        if ((double)l[i] > mx)
            mx = (double)l[i];
    double z = 0.0;
    for (int64_t i = 0; i < V; i++)
        z += exp((double)l[i] - mx);
    const double log_z = log(z);
    double h = 0.0;
    for (int64_t i = 0; i < V; i++) {
        if (isinf(l[i]) && l[i] < 0)
            continue;                     /* p_i = 0: contributes nothing */
        const double log_p = (double)l[i] - mx - log_z;
        h -= exp(log_p) * log_p;
    }
    return h;
}

static void *entropy_worker(void *arg)
{
    row_job *j = (row_job *)arg;
    for (int t = j->t0; t < j->t1; t++)
        j->H[t] = row_entropy(j->logits + (int64_t)t * j->V, j->V);
    return NULL;
}

/* [GUM] S4 for one row: the sample, the argmax, and the best and second-best
   perturbed scores (the tests use the gap to tell near-ties). */
static void *gumbel_worker(void *arg)
{
    row_job *j = (row_job *)arg;
    for (int t = j->t0; t < j->t1; t++) {
        const float *l = j->logits + (int64_t)t * j->V;
        int64_t s_idx = -1, a_idx = -1;
        double s_best = -INFINITY, s_second = -INFINITY, a_best = -INFINITY;
        for (int64_t i = 0; i < j->V; i++) {
            const double li = (double)l[i];
            if (a_idx < 0 || li > a_best) {
                a_best = li;
                a_idx = i;
            }
            const double score = li + oracle_gumbel_of_word(
                                          oracle_noise_word(j->seed, j->offset, t, i));
            if (s_idx < 0 || score > s_best) {
                s_second = s_best;
                s_best = score;
                s_idx = i;
            } else if (score > s_second) {
                s_second = score;
            }
        }
        j->sample[t] = s_idx;
        j->amax[t] = a_idx;
        j->best[t] = s_best;
        j->second[t] = s_second;
    }
    return NULL;
}

static void run_rows(void *(*fn)(void *), row_job proto, int M, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > M)
        nthreads = M > 0 ? M : 1;
    row_job *jobs = (row_job *)calloc((size_t)nthreads, sizeof(row_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    const int per = (M + nthreads - 1) / nthreads;
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = proto;
        jobs[i].t0 = i * per < M ? i * per : M;
        jobs[i].t1 = (i + 1) * per < M ? (i + 1) * per : M;
    }
    for (int i = 1; i < nthreads; i++)
        pthread_create(&th[i], NULL, fn, &jobs[i]);
    fn(&jobs[0]);
    for (int i = 1; i < nthreads; i++)
        pthread_join(th[i], NULL);
    free(jobs);
    free(th);
}

void oracle_entropy(const float *logits, int M, int64_t V, double *H, int nthreads)
{
    row_job p;
    memset(&p, 0, sizeof p);
    p.logits = logits;
    p.V = V;
    p.H = H;
    run_rows(entropy_worker, p, M, nthreads);
}

void oracle_gumbel_argmax(const float *logits, int M, int64_t V, uint64_t seed, uint64_t offset,
                          int64_t *sample, int64_t *amax, double *best, double *second,
                          int nthreads)
{
    row_job p;
    memset(&p, 0, sizeof p);
    p.logits = logits;
    p.V = V;
    p.seed = seed;
    p.offset = offset;
    p.sample = sample;
    p.amax = amax;
    p.best = best;
    p.second = second;
    run_rows(gumbel_worker, p, M, nthreads);
}
