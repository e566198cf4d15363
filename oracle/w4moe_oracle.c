/*
 * w4moe_oracle.c -- the float64 CPU oracle for the W4A16 routed
 * mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load this library.  It shares no
 * code, header, table or constant with the CUDA library, and neither side
 * includes or links the other.
 *
 * Sources (page title -- section):
 *   [CK] "diffusiongemma-26B-A4B-w4a16" -- Checkpoint format: each weight is
 *        a 4-bit unsigned code with an fp16 scale and an fp16 (asymmetric)
 *        zero point shared by a group of consecutive contraction elements;
 *        byte j of a packed row holds code 2j in its low nibble and code
 *        2j+1 in its high nibble; the group is 128 for gate_up and 64 for
 *        down, whose 704-wide contraction 128 does not divide.
 *   [BM] same page -- Benchmarks: quantisation is round-to-nearest min/max,
 *        no calibration.
 *   [CAP] "Inference: Making every denoising pass fast" -- The first
 *        constraint was capacity: a group g is rebuilt from integer q_i,
 *        scale s_g and zero point z_g (the formula itself did not survive
 *        extraction; read as w_i = s_g * (q_i - z_g)).
 *   [SP] same post -- Quantisation alone leaves a sparse execution problem:
 *        each token is routed to k = 8 of E = 128 experts and its output is
 *        the routing-weighted sum of those experts' outputs; the assignments
 *        are grouped by expert and padded to whole blocks before the GEMMs,
 *        and each token's k partial outputs are summed in one fixed order
 *        with no atomic adds.
 *   [GM] "dg-w4-kernels" -- Grouped MoE: alignment is sync-free, the
 *        activation is folded into the first GEMM's epilogue, the weighted
 *        combine is a fixed-order reduction.
 *   [DL] "dg-w4-kernels" -- W4A16: w4a16_linear(x, qw, scale, zero) equals
 *        F.linear(x, dequant(W)), groups of 128 along the contraction dim;
 *        "Inference: Making every denoising pass fast" -- Dense W4 everywhere:
 *        attention, the shared MLP and the LM head as dense W4A16 layers.
 *
 * Readings where the pages are silent (each is repeated at its function):
 *   R1 gated activation: h = gelu_tanh(gate) * up.
 *   R2 gate_up rows [0, m) are the gate, rows [m, 2m) the up projection.
 *   R3 scale s = (max - min) / 15 in fp32, stored fp16; a group whose fp16
 *      scale would be zero (constant group) uses s = 1.
 *   R4 zero point z = -min / s16 in fp32, stored as fp16 (fractional).
 *   R5 q = clamp(round_half_even(w / s16 + z16), 0, 15), in fp32, no FMA.
 *   R6 router: softmax in float64, top-k by probability (equivalently by
 *      logit) with ties to the lower expert index, slots ordered by
 *      descending probability, weights renormalised over the k selected and
 *      rounded once to fp32.
 *   R7 alignment pads with the sentinel A = M*k; block_expert is -1 past the
 *      last populated block; ids outside [0, E) are counted and skipped.
 *   R8 combine: out_t = sum over slots j = 0..k-1, in that order, of
 *      w[t,j] * y[t*k+j]; the weight is applied in the combine.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 and bfloat16, written from the format definitions.      */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);              /* subnormal: fr * 2^-24 */
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fr), ex - 25); /* (1 + fr/1024) * 2^(ex-15) */
    return sign ? -v : v;
}

/* Round a finite or infinite binary32 value to binary16, nearest-even. */
uint16_t oracle_f32_to_f16(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f))
        return 0x7e00;
    /* 65504 is the largest finite value; the rounding boundary to infinity is
     * halfway to the next power of two, 65520. */
    if (a >= 65520.0)
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    /* quantum of the binade that holds a (subnormal quantum is 2^-24) */
    int e;
    frexp(a, &e);              /* a = f * 2^e with f in [0.5, 1) */
    int ulp_exp = (e - 1) - 10;
    if (ulp_exp < -24)
        ulp_exp = -24;
    double r = nearbyint(ldexp(a, -ulp_exp)); /* exact scaling, then RNE */
    double v = ldexp(r, ulp_exp);
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -14))   /* subnormal result */
        return sign | (uint16_t)ldexp(v, 24);
    frexp(v, &e);
    int ex = (e - 1) + 15;
    int fr = (int)(ldexp(v, -(e - 1) + 10) - 1024.0);
    return sign | (uint16_t)(ex << 10) | (uint16_t)fr;
}

static float f16_to_f32(uint16_t h) { return (float)oracle_f16_to_f64(h); }

/* bfloat16 is the top half of a binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* [CK] nibble packing: byte j = q[2j] | q[2j+1] << 4                         */
/* ------------------------------------------------------------------------ */

void oracle_pack_codes(const uint8_t *codes, int64_t n, uint8_t *bytes)
{
    for (int64_t j = 0; j < n / 2; j++)
        bytes[j] = (uint8_t)((codes[2 * j] & 0xf) | ((codes[2 * j + 1] & 0xf) << 4));
}

void oracle_unpack_codes(const uint8_t *bytes, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; i++)
        codes[i] = (uint8_t)((bytes[i / 2] >> (4 * (i % 2))) & 0xf);
}

/* ------------------------------------------------------------------------ */
/* [CK][BM][CAP] quantize_w4: asymmetric uint4, min/max round-to-nearest.     */
/* W is [rows, K] fp32 row-major; group runs along K.                        */
/* Outputs: q [rows, K/2] packed, s16 and z16 [rows, K/group] (binary16 bits)*/
/* Returns 0, or 1 on a shape the format cannot hold.                        */
/* ------------------------------------------------------------------------ */
int oracle_quantize_w4(const float *W, int64_t rows, int64_t K, int group,
                       uint8_t *q, uint16_t *s16, uint16_t *z16)
{
    if (rows < 0 || K <= 0 || group <= 0 || group % 2 || K % group)
        return 1;
    int64_t G = K / group;
    uint8_t *codes = (uint8_t *)malloc((size_t)group);
    if (!codes)
        return 1;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t g = 0; g < G; g++) {
            const float *w = W + r * K + g * group;
            float lo = w[0], hi = w[0];
            for (int i = 1; i < group; i++) {
                if (w[i] < lo) lo = w[i];
                if (w[i] > hi) hi = w[i];
            }
            /* R3: scale in fp32, stored fp16; zero fp16 scale -> 1 */
            float s = (hi - lo) / 15.0f;
            uint16_t sh = oracle_f32_to_f16(s);
            if ((sh & 0x7fff) == 0)
                sh = 0x3c00;
            float sf = f16_to_f32(sh);
            /* R4: fractional zero point, -min / s16 in fp32 (+0 folds -0) */
            float zf = -lo / sf;
            zf = zf + 0.0f;
            uint16_t zh = oracle_f32_to_f16(zf);
            float zz = f16_to_f32(zh);
            /* R5: nearest code, half-even, clamped to the 4-bit range */
            for (int i = 0; i < group; i++) {
                float t = w[i] / sf;
                t = t + zz;
                float rq = nearbyintf(t);
                int qi = rq < 0.0f ? 0 : (rq > 15.0f ? 15 : (int)rq);
                codes[i] = (uint8_t)qi;
            }
            oracle_pack_codes(codes, group, q + r * (K / 2) + g * (group / 2));
            s16[r * G + g] = sh;
            z16[r * G + g] = zh;
        }
    }
    free(codes);
    return 0;
}

/* [CAP] w_hat = s_g * (q - z_g), in float64.  out is [rows, K]. */
void oracle_dequant_w4(const uint8_t *q, const uint16_t *s16, const uint16_t *z16,
                       int64_t rows, int64_t K, int group, double *out)
{
    int64_t G = K / group;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t k = 0; k < K; k++) {
            int code = (q[r * (K / 2) + k / 2] >> (4 * (k % 2))) & 0xf;
            double s = oracle_f16_to_f64(s16[r * G + k / group]);
            double z = oracle_f16_to_f64(z16[r * G + k / group]);
            out[r * K + k] = s * ((double)code - z);
        }
}

/* ------------------------------------------------------------------------ */
/* [SP] router: softmax over E logits, top-k, renormalise (R6).               */
/* ------------------------------------------------------------------------ */
int oracle_route(const float *logits, int M, int E, int k, int32_t *ids, float *weights)
{
    if (M < 0 || E <= 0 || k <= 0 || k > E)
        return 1;
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    if (!p || !taken) {
        free(p);
        free(taken);
        return 1;
    }
    for (int t = 0; t < M; t++) {
        const float *l = logits + (int64_t)t * E;
        double mx = l[0];
        for (int e = 1; e < E; e++)
            if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++) {
            p[e] = exp((double)l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < E; e++) {
            p[e] /= z;
            taken[e] = 0;
        }
        /* softmax is strictly increasing in the logit, so the k most
         * probable experts are the k largest logits; comparing the fp32
         * logits themselves keeps float64 rounding of p from merging two
         * distinct logits into a tie. */
        double sel = 0.0;
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;   /* strict '>' keeps the lower index on ties */
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
            sel += p[best];
        }
        for (int j = 0; j < k; j++)
            weights[(int64_t)t * k + j] = (float)(p[ids[(int64_t)t * k + j]] / sel);
    }
    free(p);
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [SP][GM] token-to-expert alignment (counting sort, stable, padded).        */
/* ------------------------------------------------------------------------ */
int64_t oracle_align_capacity(int M, int k, int E, int block_m)
{
    int64_t A = (int64_t)M * k;
    int64_t cap = A + (int64_t)E * (block_m - 1);
    return (cap + block_m - 1) / block_m * block_m;
}

/* ids [M*k] flat, a = t*k + j.  Outputs:
 *   sorted_ids [cap]        slot -> flat assignment index, pads hold A (R7)
 *   block_expert [cap/bm]   expert owning each block, -1 past the end
 *   expert_offsets [E+1]    padded start slot of each expert
 *   num_padded [1]          expert_offsets[E]
 * Returns the number of ids outside [0, E) (skipped), or -1 on bad args. */
int64_t oracle_moe_align(const int32_t *ids, int M, int k, int E, int block_m,
                         int32_t *sorted_ids, int32_t *block_expert,
                         int32_t *expert_offsets, int32_t *num_padded)
{
    if (M < 0 || k <= 0 || E <= 0 || block_m <= 0)
        return -1;
    int64_t A = (int64_t)M * k;
    int64_t cap = oracle_align_capacity(M, k, E, block_m);
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *fill = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!count || !fill) {
        free(count);
        free(fill);
        return -1;
    }
    int64_t bad = 0;
    for (int64_t a = 0; a < A; a++) {
        if (ids[a] < 0 || ids[a] >= E)
            bad++;
        else
            count[ids[a]]++;
    }
    /* padded exclusive prefix sum of ceil(c_e / bm) * bm */
    expert_offsets[0] = 0;
    for (int e = 0; e < E; e++) {
        int64_t padded = (count[e] + block_m - 1) / block_m * block_m;
        expert_offsets[e + 1] = (int32_t)(expert_offsets[e] + padded);
    }
    for (int64_t i = 0; i < cap; i++)
        sorted_ids[i] = (int32_t)A;
    /* stable placement: walk a in increasing order */
    for (int64_t a = 0; a < A; a++) {
        int e = ids[a];
        if (e < 0 || e >= E)
            continue;
        sorted_ids[expert_offsets[e] + fill[e]] = (int32_t)a;
        fill[e]++;
    }
    for (int64_t b = 0; b < cap / block_m; b++) {
        int64_t slot = b * block_m;
        int32_t owner = -1;
        for (int e = 0; e < E; e++)
            if (slot >= expert_offsets[e] && slot < expert_offsets[e + 1])
                owner = e;
        block_expert[b] = owner;
    }
    num_padded[0] = expert_offsets[E];
    free(count);
    free(fill);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Expert MLP (R1, R2) and the fixed-order combine (R8).                      */
/* ------------------------------------------------------------------------ */

/* R1: GELU with the tanh approximation, in float64. */
double oracle_gelu_tanh(double v)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
}

/* One dequantised dot product: sum_k (s_g * (q_k - z_g)) * a_k over a row. */
static double w4_row_dot(const uint8_t *qrow, const uint16_t *srow, const uint16_t *zrow,
                         int64_t K, int group, const double *a)
{
    double acc = 0.0;
    for (int64_t kk = 0; kk < K; kk++) {
        int code = (qrow[kk / 2] >> (4 * (kk % 2))) & 0xf;
        double s = oracle_f16_to_f64(srow[kk / group]);
        double z = oracle_f16_to_f64(zrow[kk / group]);
        acc += s * ((double)code - z) * a[kk];
    }
    return acc;
}

typedef struct {
    const uint16_t *x;
    int M, d, m, E, k;
    const uint8_t *gu_q;
    const uint16_t *gu_s, *gu_z;
    int gu_group;
    const uint8_t *dn_q;
    const uint16_t *dn_s, *dn_z;
    int dn_group;
    const int32_t *ids;
    double *h_all, *y_all;      /* [M*k, m], [M*k, d] */
    int tid, nthreads;
} layer_job;

/* Phase 1: every flat assignment a = t*k + j is independent; threads take
 * a = tid, tid + nthreads, ... and write h_a and y_a. */
static void *expert_worker(void *arg)
{
    layer_job *J = (layer_job *)arg;
    const int d = J->d, m = J->m, k = J->k;
    double *xr = (double *)malloc(sizeof(double) * (size_t)d);
    if (!xr)
        return NULL;
    const int64_t Ggu = d / J->gu_group, Gdn = m / J->dn_group;
    const int64_t A = (int64_t)J->M * k;
    for (int64_t a = J->tid; a < A; a += J->nthreads) {
        const int64_t t = a / k;
        double *h = J->h_all + a * m;
        double *y = J->y_all + a * d;
        int e = J->ids[a];
        if (e < 0 || e >= J->E) {                   /* R7: skipped */
            memset(h, 0, sizeof(double) * (size_t)m);
            memset(y, 0, sizeof(double) * (size_t)d);
            continue;
        }
        for (int c = 0; c < d; c++)
            xr[c] = oracle_bf16_to_f64(J->x[t * d + c]);
        /* gate_up: rows [0, m) gate, [m, 2m) up (R2) */
        const int64_t gu_rows = 2 * (int64_t)m;
        for (int i = 0; i < m; i++) {
            int64_t rg = (int64_t)e * gu_rows + i, ru = rg + m;
            double g = w4_row_dot(J->gu_q + rg * (d / 2), J->gu_s + rg * Ggu,
                                  J->gu_z + rg * Ggu, d, J->gu_group, xr);
            double u = w4_row_dot(J->gu_q + ru * (d / 2), J->gu_s + ru * Ggu,
                                  J->gu_z + ru * Ggu, d, J->gu_group, xr);
            h[i] = oracle_gelu_tanh(g) * u;   /* R1 */
        }
        /* down: d rows, contraction over m */
        for (int r = 0; r < d; r++) {
            int64_t rr = (int64_t)e * d + r;
            y[r] = w4_row_dot(J->dn_q + rr * (m / 2), J->dn_s + rr * Gdn,
                              J->dn_z + rr * Gdn, m, J->dn_group, h);
        }
    }
    free(xr);
    return NULL;
}

static void run_threads(void *(*fn)(void *), layer_job *jobs, int nthreads)
{
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, fn, &jobs[i]) != 0)
            break;
        started = i;
    }
    fn(&jobs[0]);
    for (int i = 1; i <= started; i++)
        pthread_join(th[i], NULL);
    for (int i = started + 1; i < nthreads; i++)   /* threads that failed to start */
        fn(&jobs[i]);
}

/* The whole layer in float64.
 *   x        [M, d] bf16 bits
 *   gu_q     [E, 2m, d/2], gu_s/gu_z [E, 2m, d/gu_group]
 *   dn_q     [E, d, m/2],  dn_s/dn_z [E, d, m/dn_group]
 *   ids, weights [M, k]
 *   h_out [M*k, m], y_out [M*k, d] (either may be NULL), out [M, d].
 * Assignments (t, j) are split over nthreads POSIX threads, each writing its
 * own h and y rows; the combine then runs token by token in slot order.  Every
 * value is produced by one fixed sequence of operations, so the result does
 * not depend on the thread count.  Returns 0, or 1 on bad arguments. */
int oracle_moe_layer(const uint16_t *x, int M, int d, int m, int E, int k,
                     const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z, int gu_group,
                     const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
                     const int32_t *ids, const float *weights, int nthreads,
                     double *h_out, double *y_out, double *out)
{
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0 || gu_group <= 0 || dn_group <= 0 ||
        d % gu_group || m % dn_group || d % 2 || m % 2)
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    const int64_t A = (int64_t)M * k;
    double *h_all = h_out ? h_out : (double *)malloc(sizeof(double) * (size_t)(A * m + 1));
    double *y_all = y_out ? y_out : (double *)malloc(sizeof(double) * (size_t)(A * d + 1));
    if (!h_all || !y_all) {
        if (!h_out) free(h_all);
        if (!y_out) free(y_all);
        return 1;
    }
    layer_job jobs[256];
    for (int i = 0; i < nthreads; i++) {
        layer_job J = {x, M, d, m, E, k, gu_q, gu_s, gu_z, gu_group, dn_q, dn_s, dn_z,
                       dn_group, ids, h_all, y_all, i, nthreads};
        jobs[i] = J;
    }
    run_threads(expert_worker, jobs, nthreads);
    /* Phase 2, R8: out_t = sum over slots j = 0..k-1, in that order */
    for (int64_t t = 0; t < M; t++) {
        for (int c = 0; c < d; c++) {
            double acc = 0.0;
            for (int j = 0; j < k; j++) {
                const int64_t a = t * k + j;
                if (ids[a] < 0 || ids[a] >= E)
                    continue;
                acc += (double)weights[a] * y_all[a * d + c];
            }
            out[t * d + c] = acc;
        }
    }
    if (!h_out) free(h_all);
    if (!y_out) free(y_all);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [DL] the dense W4A16 linear: y[t, n] = sum_k x[t, k] * deq(W)[n, k], in   */
/* float64, x given as bf16 bits.  Rows of y are split over POSIX threads;   */
/* every value is one fixed sequence of operations.                           */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *x;
    int M, K, N;
    const uint8_t *q;
    const uint16_t *s, *z;
    int group;
    double *y;
    int tid, nthreads;
} linear_job;

static void *linear_worker(void *arg)
{
    linear_job *J = (linear_job *)arg;
    double *xr = (double *)malloc(sizeof(double) * (size_t)J->K);
    if (!xr)
        return NULL;
    const int64_t G = J->K / J->group;
    for (int t = J->tid; t < J->M; t += J->nthreads) {
        for (int kk = 0; kk < J->K; kk++)
            xr[kk] = oracle_bf16_to_f64(J->x[(int64_t)t * J->K + kk]);
        for (int n = 0; n < J->N; n++)
            J->y[(int64_t)t * J->N + n] =
                w4_row_dot(J->q + (int64_t)n * (J->K / 2), J->s + (int64_t)n * G,
                           J->z + (int64_t)n * G, J->K, J->group, xr);
    }
    free(xr);
    return NULL;
}

int oracle_w4a16_linear(const uint16_t *x, int M, int K, int N, const uint8_t *q,
                        const uint16_t *s, const uint16_t *z, int group, int nthreads, double *y)
{
    if (M < 0 || K <= 0 || N <= 0 || group <= 0 || K % group || K % 2)
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    linear_job jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; i++) {
        linear_job J = {x, M, K, N, q, s, z, group, y, i, nthreads};
        jobs[i] = J;
    }
    int started = 0;
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&th[i], NULL, linear_worker, &jobs[i]) != 0)
            break;
        started = i;
    }
    linear_worker(&jobs[0]);
    for (int i = 1; i <= started; i++)
        pthread_join(th[i], NULL);
    for (int i = started + 1; i < nthreads; i++)
        linear_worker(&jobs[i]);
    return 0;
}
