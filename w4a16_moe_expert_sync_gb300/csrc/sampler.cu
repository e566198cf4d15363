// sampler.cu -- one streaming pass over vocabulary logits [M, V] fp32 that
// yields, per row, the entropy of Categorical(logits) in nats, a Gumbel-max
// sample and the plain argmax ("dg-w4-kernels" -- Sampler: fused_entropy in a
// single pass instead of the logsumexp/sub/exp/mul/sum chain;
// gumbel_argmax_sample draws from the same Categorical with Philox noise made
// inline, the argmax coming out of the same reduction).
//
// Layout of the work: the rows are laid end to end as quads (4 consecutive
// logits) and cut into equal spans, one per persistent 256-thread CTA (three
// per SM); a CTA reduces each row segment of its span to a partial
// (online-softmax state, best perturbed score, best logit), and a second
// launch merges each row's partials.  Every reduction runs in a fixed order,
// so results do not depend on scheduling (the spans depend on the SM count).
//
// Noise (Philox4x32-10, Salmon et al., SC 2011): key = (seed lo, seed hi);
// the quad q of row t uses counter (q, t, offset lo, offset hi) and its
// column 4q + j takes output word j.  A word r gives v = (r + 1/2) 2^-32,
// E = -ln(1 - v) and g = -ln E; the sample is argmax(logit + g), the argmax
// argmax(logit), ties to the lower column in both.
#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace w4 {

namespace {

constexpr int kSamplerThreads = 256;

// g = -ln(-ln(1 - v)) never exceeds 22.88 (v >= 2^-33); a quad whose largest
// logit is more than this below the running best cannot win and skips its noise.
constexpr float kGumbelBound = 23.0f;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The entropy state is kept in base 2: with y = l log2(e) and m the running
// max of y, s = sum 2^(y - m) and t = sum 2^(y - m) (y - m); then
// H = ln 2 (log2 s - t / s), whatever m is.
struct Partial {
    float m, s, t;        // base-2 max, sum 2^(y - m), sum 2^(y - m) (y - m)
    float best;           // best perturbed score
    int best_idx;
    float amax;           // best logit
    int amax_idx;
    int pad;
};

// The ten round keys of one (seed) key schedule: key + r * Weyl constants.
// Passed as a kernel parameter so that the key XOR reads them from the
// constant bank instead of recomputing them per call.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};

__device__ __forceinline__ uint64_t mul_wide(uint32_t a, uint32_t b)
{
    uint64_t p;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
    return p;
}

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              const PhiloxKeys &key, uint32_t out[4])
{
#pragma unroll
    for (int r = 0; r < 10; r++) {
        const uint64_t p0 = mul_wide(0xD2511F53u, c0);
        const uint64_t p1 = mul_wide(0xCD9E8D57u, c2);
        const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ key.k0[r];
        const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ key.k1[r];
        c0 = n0;
        c1 = static_cast<uint32_t>(p1);
        c2 = n2;
        c3 = static_cast<uint32_t>(p0);
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The Gumbel variate of a word r: v = (r + 1/2) 2^-32, g = -ln(-ln(1 - v)),
// computed two ways (|error| below ~2e-7 in both):
//  * v < 1/8: g = -ln v - P(v), P(v) ~ ln(-ln(1 - v) / v) = v/2 + 5v^2/24 + ...
//    as the polynomial v (c1 + v (c2 + v (c3 + v c4))), least-squares fitted
//    on [0, 1/8] (error 1.7e-8 in fp32), and one approximate log2 of v;
//  * v >= 1/8: g = -ln(-ln 2 log2(1 - v)) with 1 - v within 2^-25 of exact;
//    here g <= 2.014, so the path only runs for logits that can still win.
constexpr float kSmallV = 0.125f;
constexpr float kLargeBound = 2.02f;     // g < 2.0134 when v >= 1/8
constexpr float kP1 = 0.4999984585455972f, kP2 = 0.20844736943052908f;
constexpr float kP3 = 0.12235092648523167f, kP4 = 0.11096642997321587f;

__device__ __forceinline__ float word_to_v(uint32_t r)
{
    return fmaf(static_cast<float>(r), 0x1p-32f, 0x1p-33f);
}

__device__ __forceinline__ float gumbel_small(float v)
{
    const float p = v * fmaf(v, fmaf(v, fmaf(v, kP4, kP3), kP2), kP1);
    return fmaf(-kLn2, lg2_approx(v), -p);
}

// v is capped below 1 so that -ln(1 - v) stays finite
__device__ __forceinline__ float gumbel_large(float v)
{
    const float e = -kLn2 * lg2_approx(1.0f - fminf(v, 0x1.fffffep-1f));
    return -kLn2 * lg2_approx(e);
}

// (val, idx) pairs: the larger value wins, equal values go to the lower
// index, idx < 0 marks "none yet"
__device__ __forceinline__ bool pair_better(float bv, int bi, float av, int ai)
{
    return bi >= 0 && (ai < 0 || bv > av || (bv == av && bi < ai));
}

__device__ __forceinline__ void ent_merge(float &m, float &s, float &t, float m2, float s2, float t2)
{
    const float mn = fmaxf(m, m2);
    const float c1 = exp2f(m - mn), c2 = exp2f(m2 - mn);
    const float sn = c1 * s + c2 * s2;
    t = c1 * (t + (m - mn) * s) + c2 * (t2 + (m2 - mn) * s2);
    s = sn;
    m = mn;
}

__device__ __forceinline__ void partial_merge(Partial &a, const Partial &b)
{
    ent_merge(a.m, a.s, a.t, b.m, b.s, b.t);
    if (pair_better(b.best, b.best_idx, a.best, a.best_idx)) {
        a.best = b.best;
        a.best_idx = b.best_idx;
    }
    if (pair_better(b.amax, b.amax_idx, a.amax, a.amax_idx)) {
        a.amax = b.amax;
        a.amax_idx = b.amax_idx;
    }
}

__device__ __forceinline__ Partial shfl_partial(const Partial &p, int src_lane_xor)
{
    Partial q;
    const unsigned full = 0xffffffffu;
    q.m = __shfl_xor_sync(full, p.m, src_lane_xor);
    q.s = __shfl_xor_sync(full, p.s, src_lane_xor);
    q.t = __shfl_xor_sync(full, p.t, src_lane_xor);
    q.best = __shfl_xor_sync(full, p.best, src_lane_xor);
    q.best_idx = __shfl_xor_sync(full, p.best_idx, src_lane_xor);
    q.amax = __shfl_xor_sync(full, p.amax, src_lane_xor);
    q.amax_idx = __shfl_xor_sync(full, p.amax_idx, src_lane_xor);
    q.pad = 0;
    return q;
}

// Butterfly merge: every lane ends with the same value.  A lane's partner
// is the same for both lanes of a pair and the merge is applied with the
// lower lane's value first, so both lanes compute bit-identical results.
__device__ __forceinline__ void warp_merge(Partial &p, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Partial q = shfl_partial(p, o);
        if (lane & o) {
            Partial lo = q;
            partial_merge(lo, p);
            p = lo;
        } else {
            partial_merge(p, q);
        }
    }
}

__device__ __forceinline__ Partial empty_partial()
{
    Partial p;
    p.m = -FLT_MAX;
    p.s = 0.0f;
    p.t = 0.0f;
    p.best = -INFINITY;
    p.best_idx = -1;
    p.amax = -INFINITY;
    p.amax_idx = -1;
    p.pad = 0;
    return p;
}

constexpr int kBatch = 4;          // quads per thread per load batch (double-buffered)
constexpr int kMaxGrid = 2048;     // cap on the persistent grid (bounds the workspace)
constexpr int kMinSpan = kSamplerThreads * kBatch;   // quads per CTA at least

// One quad: logits l[0..3] of columns col0..col0+3 (-inf past the row's end).
template <bool ENT, bool SAMP>
__device__ __forceinline__ void process_quad(Partial &p, const float (&l)[4], int64_t q, int t,
                                             int col0, const PhiloxKeys &key, uint32_t off0,
                                             uint32_t off1)
{
    const float qm = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
    if constexpr (ENT) {
        const float qm2 = qm * kLog2e;
        if (qm2 > p.m) {           // rescale to the new maximum
            const float c1 = ex2_approx(p.m - qm2);
            p.t = c1 * fmaf(p.m - qm2, p.s, p.t);
            p.s *= c1;
            p.m = qm2;
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            // -inf logits (masked, or past the row's end) contribute 0
            const float y = fmaxf(fmaf(l[j], kLog2e, -p.m), -300.0f);
            const float e = ex2_approx(y);
            p.s += e;
            p.t = fmaf(e, y, p.t);
        }
    }
    // Selections compare strictly against the running best, so a -inf
    // logit (masked, or past the row's end) is never chosen and the
    // column of a new best is the quad's first holding it; a row with
    // no finite logit keeps index -1, resolved by the merge kernel.
    if (qm > p.amax) {
        const int jj = l[0] == qm ? 0 : l[1] == qm ? 1 : l[2] == qm ? 2 : 3;
        p.amax = qm;
        p.amax_idx = col0 + jj;
    }
    if constexpr (SAMP) {
        if (qm + kGumbelBound >= p.best) {
            uint32_t r[4];
            philox4x32_10(static_cast<uint32_t>(q), static_cast<uint32_t>(t), off0, off1, key, r);
            float v[4], sc[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                v[j] = word_to_v(r[j]);
                sc[j] = v[j] < kSmallV ? l[j] + gumbel_small(v[j]) : -INFINITY;
            }
            if (qm + kLargeBound >= p.best) {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    if (v[j] >= kSmallV)
                        sc[j] = l[j] + gumbel_large(v[j]);
            }
            const float qs = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            if (qs > p.best) {
                const int jj = sc[0] == qs ? 0 : sc[1] == qs ? 1 : sc[2] == qs ? 2 : 3;
                p.best = qs;
                p.best_idx = col0 + jj;
            }
        }
    }
}

template <bool VEC>
__device__ __forceinline__ void load_batch(const float *row, int64_t V, int64_t q, int64_t qend,
                                           float4 (&buf)[kBatch])
{
#pragma unroll
    for (int i = 0; i < kBatch; i++) {
        const int64_t qi = q + static_cast<int64_t>(i) * kSamplerThreads;
        if constexpr (VEC) {
            buf[i] = qi < qend ? __ldcs(reinterpret_cast<const float4 *>(row) + qi)
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        } else {
            const int64_t col = 4 * qi;
            const bool in = qi < qend;
            buf[i].x = in && col < V ? __ldcs(row + col) : -INFINITY;
            buf[i].y = in && col + 1 < V ? __ldcs(row + col + 1) : -INFINITY;
            buf[i].z = in && col + 2 < V ? __ldcs(row + col + 2) : -INFINITY;
            buf[i].w = in && col + 3 < V ? __ldcs(row + col + 3) : -INFINITY;
        }
    }
}

// Persistent CTAs: CTA b streams quads [b span, (b + 1) span) of the rows laid
// end to end (nq quads per row), each thread every 256th quad with the next
// batch in flight, and writes one partial per row segment it covers, for
// row t at slot b + t (distinct for every (b, t) since spans are contiguous).
template <bool VEC, bool ENT, bool SAMP>
__global__ void __launch_bounds__(kSamplerThreads, 3)
    sampler_partial_kernel(const float *__restrict__ logits, int64_t V, int64_t nq,
                           int64_t total_q, int64_t span, const __grid_constant__ PhiloxKeys key,
                           uint32_t off0, uint32_t off1, Partial *__restrict__ part)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t g_begin = static_cast<int64_t>(b) * span;
    const int64_t g_end = min(total_q, g_begin + span);
    __shared__ Partial wp[kSamplerThreads / 32];
    constexpr int64_t kStep = static_cast<int64_t>(kBatch) * kSamplerThreads;
    for (int64_t gs = g_begin; gs < g_end;) {
        const int t = static_cast<int>(gs / nq);
        const int64_t ge = min(g_end, static_cast<int64_t>(t + 1) * nq);
        const int64_t qa = gs - static_cast<int64_t>(t) * nq;
        const int64_t qb = ge - static_cast<int64_t>(t) * nq;
        const float *row = logits + static_cast<int64_t>(t) * V;
        Partial p = empty_partial();
        float4 cur[kBatch], nxt[kBatch];
        load_batch<VEC>(row, V, qa + tid, qb, cur);
        for (int64_t q = qa + tid; q < qb; q += kStep) {
            load_batch<VEC>(row, V, q + kStep, qb, nxt);
            if (q + (kBatch - 1) * kSamplerThreads < qb) {    // a whole batch: no checks
#pragma unroll
                for (int i = 0; i < kBatch; i++) {
                    const int64_t qi = q + static_cast<int64_t>(i) * kSamplerThreads;
                    const float l[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
                    process_quad<ENT, SAMP>(p, l, qi, t, static_cast<int>(4 * qi), key, off0,
                                            off1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kBatch; i++) {
                    const int64_t qi = q + static_cast<int64_t>(i) * kSamplerThreads;
                    if (qi < qb) {
                        const float l[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
                        process_quad<ENT, SAMP>(p, l, qi, t, static_cast<int>(4 * qi), key,
                                                off0, off1);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; i++)
                cur[i] = nxt[i];
        }
        // CTA reduction in a fixed order: butterfly in each warp, then warp 0
        // merges the warps' results in warp order
        warp_merge(p, lane);
        if (lane == 0)
            wp[warp] = p;
        __syncthreads();
        if (warp == 0) {
            Partial a = lane < kSamplerThreads / 32 ? wp[lane] : empty_partial();
            warp_merge(a, lane);
            if (lane == 0)
                part[b + t] = a;
        }
        __syncthreads();
        gs = ge;
    }
}

// One warp per row: the partials of the CTAs whose spans meet row t, lane i
// taking the i-th, i+32-th, ... of them, merged by butterfly (a fixed order).
__global__ void __launch_bounds__(256)
    sampler_finish_kernel(const Partial *__restrict__ part, int M, int64_t nq, int64_t span,
                          int grid, float *__restrict__ entropy, int64_t *__restrict__ sample,
                          int64_t *__restrict__ amax)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= M)
        return;
    const int b0 = static_cast<int>(static_cast<int64_t>(t) * nq / span);
    const int b1 = min(grid - 1, static_cast<int>((static_cast<int64_t>(t + 1) * nq - 1) / span));
    Partial p = empty_partial();
    for (int b = b0 + lane; b <= b1; b += 32)
        partial_merge(p, part[b + t]);
    warp_merge(p, lane);
    if (lane == 0) {
        if (entropy)
            entropy[t] = kLn2 * (log2f(p.s) - p.t / p.s);
        // a row with no finite logit: column 0 for both, as for ties
        if (sample)
            sample[t] = p.best_idx >= 0 ? p.best_idx : 0;
        if (amax)
            amax[t] = p.amax_idx >= 0 ? p.amax_idx : 0;
    }
}

struct SamplerGrid {
    int64_t nq, total_q, span;
    int grid;
};

template <bool VEC, bool ENT, bool SAMP>
cudaError_t launch_partial(const float *logits, int M, int64_t V, const SamplerGrid &g,
                           uint64_t seed, uint64_t offset, Partial *part, cudaStream_t stream)
{
    PhiloxKeys key;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; r++) {      // the schedule: the key bumped by the Weyl constants
        key.k0[r] = k0;
        key.k1[r] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return launch_pdl(sampler_partial_kernel<VEC, ENT, SAMP>, dim3(g.grid), dim3(kSamplerThreads),
                      0, stream, logits, V, g.nq, g.total_q, g.span, key,
                      static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32), part);
}

template <bool VEC>
cudaError_t launch_partial_any(bool ent, bool samp, const float *logits, int M, int64_t V,
                               const SamplerGrid &g, uint64_t seed, uint64_t offset, Partial *part,
                               cudaStream_t stream)
{
    if (ent && samp)
        return launch_partial<VEC, true, true>(logits, M, V, g, seed, offset, part, stream);
    if (ent)
        return launch_partial<VEC, true, false>(logits, M, V, g, seed, offset, part, stream);
    if (samp)
        return launch_partial<VEC, false, true>(logits, M, V, g, seed, offset, part, stream);
    return launch_partial<VEC, false, false>(logits, M, V, g, seed, offset, part, stream);
}

// Three resident CTAs per SM (the launch bounds guarantee the registers).
SamplerGrid sampler_grid(int M, int64_t V)
{
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0, n = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        num_sms = n > 0 ? n : 1;
    }
    SamplerGrid g;
    g.nq = (V + 3) / 4;
    g.total_q = static_cast<int64_t>(M) * g.nq;
    const int64_t slots = std::min<int64_t>(kMaxGrid, 3 * static_cast<int64_t>(num_sms));
    g.span = std::max<int64_t>(kMinSpan, (g.total_q + slots - 1) / slots);
    g.grid = static_cast<int>((g.total_q + g.span - 1) / g.span);
    return g;
}

}  // namespace

size_t sampler_workspace_bytes(int M, int64_t V)
{
    (void)V;
    return sizeof(Partial) * (static_cast<size_t>(kMaxGrid) + static_cast<size_t>(M));
}

cudaError_t launch_sampler(const float *logits, int M, int64_t V, uint64_t seed, uint64_t offset,
                           float *entropy, int64_t *sample, int64_t *amax, void *workspace,
                           cudaStream_t stream)
{
    if (M == 0)
        return cudaSuccess;
    const SamplerGrid g = sampler_grid(M, V);
    Partial *part = static_cast<Partial *>(workspace);
    const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    cudaError_t err = vec ? launch_partial_any<true>(entropy != nullptr, sample != nullptr, logits,
                                                     M, V, g, seed, offset, part, stream)
                          : launch_partial_any<false>(entropy != nullptr, sample != nullptr,
                                                      logits, M, V, g, seed, offset, part, stream);
    if (err != cudaSuccess)
        return err;
    return launch_pdl(sampler_finish_kernel, dim3((M + 7) / 8), dim3(256), 0, stream,
                      static_cast<const Partial *>(part), M, g.nq, g.span, g.grid, entropy,
                      sample, amax);
}

}  // namespace w4
