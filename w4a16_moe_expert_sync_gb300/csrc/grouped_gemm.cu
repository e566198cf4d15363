// grouped_gemm.cu -- grouped W4A16 expert GEMMs on the 5th-generation tensor
// cores (tcgen05) of sm_103a.
//
// What is computed ("dg-w4-kernels" -- Grouped MoE; "diffusiongemma-26B-A4B-
// w4a16" -- Checkpoint format; "Inference: Making every denoising pass fast"
// -- Quantisation alone leaves a sparse execution problem, The final best W4
// MoE kernel):
//   gate_up: for every expert e and every alignment slot of e,
//            [g | u] = x_t . deq(Wgu[e])^T, h[slot] = gelu_tanh(g) * u
//   down:    y[a] = h[slot(a)] . deq(Wdn[e])^T
// with deq(W) = s_g * (q - z_g) for uint4 codes q packed two per byte and fp16
// s, z per group along the contraction dim.
//
// Design (one persistent CTA per SM, 16 warps, static round-robin schedule):
//   * A work unit is (job, panel).  A job is one expert's slot range of at
//     most 256 slots; a panel is 128 weight rows (gate_up: 64 gate rows and
//     the matching 64 up rows; down: 128 output rows).  Every weight row of an
//     expert is streamed from HBM once per job, whatever the number of tokens.
//   * The MMA is "swap-AB": the 128 dequantised weight rows are the M = 128
//     operand and the expert's tokens are N (16..256).  The A operand lives in
//     tensor memory: dequant warps write fp16 weights straight from registers
//     with tcgen05.st, so the expanded weights never touch shared memory
//     bandwidth.  B (activations, fp16) is read by the tensor core from
//     shared memory in the 128-byte-swizzled K-major layout.  fp32
//     accumulators live in tensor memory (columns 256..511).
//   * Warp roles
//       warp 0      TMA producer: packed nibble tiles (128 rows x 128 B, two
//                   64-row boxes, SWIZZLE_128B, evict-first) into a 6-stage
//                   ring; the unit's fp16 scales/zeros by bulk copy into a
//                   double buffer.
//       warp 1      TMEM owner and single-thread tcgen05.mma issuer.
//       warps 2-7   activation producers: gather token rows (gate_up: x rows
//                   of the slots' tokens, bf16 -> fp16; down: h rows of the
//                   slots), write them swizzled into a 3-slot ring.
//       warps 8-15  dequant (two warps per TMEM lane quarter, one per half of
//                   each 256-wide K chunk) and then the epilogue.
//   * Dequantisation of 8 codes held in one 32-bit word costs 12 integer /
//     half2 instructions: the nibbles are ORed into the mantissa of the fp16
//     constant 1024 (exact integers 1024 + q and 1024 + 16q), the 1024 (or 64
//     after a 1/16 scale) is removed exactly, and one half2 FMA applies
//     q * s + (-z * s) with a single rounding.  Extracting nibbles this way
//     yields the pairs (q0,q4), (q1,q5), (q2,q6), (q3,q7), so the K order
//     inside every block of 8 is permuted to 0,4,1,5,2,6,3,7 for both
//     operands; the activation producers apply the same permutation when they
//     convert x (or h) to fp16, so the contraction is unchanged.
//   * Every output element is written once, by one thread, after a fixed
//     sequence of MMAs in increasing K: results are bit-identical run to run.
//   * Every pipeline wait has a time limit; on expiry the CTA raises
//     W4_DEV_PIPELINE_TIMEOUT, stops, drains its own copies and MMAs, frees
//     its tensor memory and exits.
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace w4 {

namespace {

constexpr int kThreads = 512;
constexpr int kStagesA = 6;                 // packed-weight stages
constexpr int kStagesB = 3;                 // activation stages
constexpr int kTileRows = 128;              // MMA M
constexpr int kChunkK = 256;                // K elements per weight stage
constexpr int kStageABytes = kTileRows * kChunkK / 2;   // 16 KB
constexpr int kStageBBytes = 32768;         // N x Kb x 2 B, N*Kb <= 16384
constexpr int kMaxN = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;           // accumulator columns [256, 512)
constexpr int kNumBThreads = 192;           // warps 2..7
constexpr int kNumDqThreads = 256;          // warps 8..15

struct GemmArgs {
    CUtensorMap tmap_w;                     // [E*R rows, K/2 bytes] uint8
    const uint16_t *act;
    const uint16_t *sc;
    const uint16_t *zp;
    const int32_t *sorted_ids;
    const int32_t *expert_offsets;
    void *out;
    int32_t *dev_status;
    int E, k, A, K, R, m_up, out_cols, group, G, n_panels, n_kchunks, sz_bytes, max_jobs;
};

struct SmemLayout {
    int off_b, off_sz, off_bar, off_misc, off_offs, off_jobs, total;
};

__host__ __device__ inline SmemLayout smem_layout(int sz_bytes, int E, int max_jobs)
{
    SmemLayout L;
    L.off_b = kStagesA * kStageABytes;
    L.off_sz = L.off_b + kStagesB * kStageBBytes;
    L.off_bar = L.off_sz + 2 * sz_bytes;
    L.off_bar = (L.off_bar + 7) & ~7;
    L.off_misc = L.off_bar + 8 * (2 * kStagesA + 2 * kStagesB + 4 + 4 + 3);
    L.off_offs = L.off_misc + 16;
    L.off_jobs = L.off_offs + 4 * (E + 1);
    L.total = L.off_jobs + 4 * max_jobs;
    return L;
}

struct Bars {
    uint64_t *a_full, *a_empty, *b_full, *b_empty, *t_full, *t_empty, *sz_full, *sz_empty;
    uint64_t *acc_full, *acc_empty, *drain;
};

__device__ __forceinline__ Bars carve_bars(uint8_t *base)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    Bars r;
    r.a_full = b;
    r.a_empty = r.a_full + kStagesA;
    r.b_full = r.a_empty + kStagesA;
    r.b_empty = r.b_full + kStagesB;
    r.t_full = r.b_empty + kStagesB;
    r.t_empty = r.t_full + 2;
    r.sz_full = r.t_empty + 2;
    r.sz_empty = r.sz_full + 2;
    r.acc_full = r.sz_empty + 2;
    r.acc_empty = r.acc_full + 1;
    r.drain = r.acc_empty + 1;
    return r;
}

struct Job {
    int e, start, n;
};

__device__ __forceinline__ Job decode_job(const int *jobs, const int *offs, int j)
{
    const int v = jobs[j];
    Job J;
    J.e = v & 0xffff;
    J.start = offs[J.e] + (v >> 16) * kMaxN;
    J.n = min(kMaxN, offs[J.e + 1] - J.start);
    return J;
}

// K elements held by one activation slot for a job of n tokens (multiple of 64).
__device__ __forceinline__ int slot_k(int n) { return 64 * (kMaxN / n); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// fp32 pair -> fp16x2 (lo in the low half), round to nearest, saturating.
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 uint4 codes (one 32-bit word, code i in bits 4i..4i+3) -> 4 fp16x2 words
// in the permuted K order (q0,q4) (q1,q5) (q2,q6) (q3,q7), each s*q + c.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 c2, uint32_t *o)
{
    const uint32_t kMagic = 0x64006400u;                // fp16 1024.0 twice
    const __half2 k1024 = u2h(kMagic);
    const __half2 kSixteenth = u2h(0x2C002C00u);        // 1/16
    const __half2 kMinus64 = u2h(0xD400D400u);          // -64
    const uint32_t w8 = w >> 8;
    const __half2 q04 = __hsub2(u2h((w & 0x000F000Fu) | kMagic), k1024);
    const __half2 q15 = __hfma2(u2h((w & 0x00F000F0u) | kMagic), kSixteenth, kMinus64);
    const __half2 q26 = __hsub2(u2h((w8 & 0x000F000Fu) | kMagic), k1024);
    const __half2 q37 = __hfma2(u2h((w8 & 0x00F000F0u) | kMagic), kSixteenth, kMinus64);
    o[0] = h2u(__hfma2(q04, s2, c2));
    o[1] = h2u(__hfma2(q15, s2, c2));
    o[2] = h2u(__hfma2(q26, s2, c2));
    o[3] = h2u(__hfma2(q37, s2, c2));
}

// 8 bf16 activations (x0..x7) -> fp16 in the permuted order.
__device__ __forceinline__ uint4 bf16x8_to_f16_perm(uint4 v)
{
    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xffff0000u);
    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xffff0000u);
    const float x4 = __uint_as_float(v.z << 16), x5 = __uint_as_float(v.z & 0xffff0000u);
    const float x6 = __uint_as_float(v.w << 16), x7 = __uint_as_float(v.w & 0xffff0000u);
    uint4 o;
    o.x = f16x2_sat(x0, x4);
    o.y = f16x2_sat(x1, x5);
    o.z = f16x2_sat(x2, x6);
    o.w = f16x2_sat(x3, x7);
    return o;
}

// 8 fp16 values (h0..h7) -> the permuted order, by byte permutes.
__device__ __forceinline__ uint4 f16x8_perm(uint4 v)
{
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);   // (h0, h4)
    o.y = __byte_perm(v.x, v.z, 0x7632);   // (h1, h5)
    o.z = __byte_perm(v.y, v.w, 0x5410);   // (h2, h6)
    o.w = __byte_perm(v.y, v.w, 0x7632);   // (h3, h7)
    return o;
}

__device__ __forceinline__ float gelu_tanh(float v)
{
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}

// bounded wait that ignores the abort flag (used only while draining)
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 200000000ull)
            return;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemLayout L = smem_layout(p.sz_bytes, p.E, p.max_jobs);
    uint8_t *stage_a = smem;
    uint8_t *stage_b = smem + L.off_b;
    uint8_t *sz_base = smem + L.off_sz;
    const Bars bar = carve_bars(smem + L.off_bar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    int *n_jobs_sm = reinterpret_cast<int *>(smem + L.off_misc + 8);
    int *offs = reinterpret_cast<int *>(smem + L.off_offs);
    int *jobs = reinterpret_cast<int *>(smem + L.off_jobs);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned full = 0xffffffffu;
    int32_t *status = p.dev_status;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < kStagesA; i++) {
            mbar_init(&bar.a_full[i], 1);
            mbar_init(&bar.a_empty[i], kNumDqThreads);
        }
        for (int i = 0; i < kStagesB; i++) {
            mbar_init(&bar.b_full[i], kNumBThreads);
            mbar_init(&bar.b_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar.t_full[i], kNumDqThreads);
            mbar_init(&bar.t_empty[i], 1);
            mbar_init(&bar.sz_full[i], 1);
            mbar_init(&bar.sz_empty[i], kNumDqThreads);
        }
        mbar_init(bar.acc_full, 1);
        mbar_init(bar.acc_empty, kNumDqThreads);
        mbar_init(bar.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0)
        prefetch_tmap(&p.tmap_w);
    for (int i = tid; i <= p.E; i += kThreads)
        offs[i] = __ldg(p.expert_offsets + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // job list: one job per expert and 256-slot chunk of its range
    if (warp == 0) {
        int base = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            int nj = 0;
            if (e < p.E)
                nj = (offs[e + 1] - offs[e] + kMaxN - 1) / kMaxN;
            int inc = nj;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(full, inc, o);
                if (lane >= o)
                    inc += v;
            }
            const int excl = base + inc - nj;
            for (int c = 0; c < nj; c++)
                if (excl + c < p.max_jobs)
                    jobs[excl + c] = e | (c << 16);
            base += __shfl_sync(full, inc, 31);
        }
        if (lane == 0) {
            *n_jobs_sm = min(base, p.max_jobs);
            if (base > p.max_jobs && status)
                atomicOr(status, kDevTooManyJobs);
        }
    }
    __syncthreads();

    const uint32_t tmem = *tmem_holder;
    const int n_units = *n_jobs_sm * p.n_panels;
    const int K = p.K;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int sa = 0, szb = 0;
            uint32_t ph_a = 0, ph_sz = 0;
            uint32_t issued_a = 0, issued_sz = 0;          // bit i: stage used
            uint32_t issue_ph_a = 0, issue_ph_sz = 0;       // phase of last issue
            const uint8_t *sc = reinterpret_cast<const uint8_t *>(p.sc);
            const uint8_t *zp = reinterpret_cast<const uint8_t *>(p.zp);
            const int rowbytes = p.G * 2;
            for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
                const Job J = decode_job(jobs, offs, u / p.n_panels);
                const int pnl = u % p.n_panels;
                const int row0 = J.e * p.R + pnl * (GATE_UP ? 64 : 128);
                const int row1 = GATE_UP ? row0 + p.m_up : row0 + 64;
                if (!mbar_wait(&bar.sz_empty[szb], ph_sz ^ 1, abort_flag, status,
                               kDevPipelineTimeout))
                    break;
                {
                    uint8_t *dst = sz_base + szb * p.sz_bytes;
                    const uint32_t hb = 64u * rowbytes;     // 64 rows of s (or z)
                    mbar_arrive_expect_tx(&bar.sz_full[szb], 4 * hb);
                    bulk_load(dst, sc + static_cast<int64_t>(row0) * rowbytes, hb,
                              &bar.sz_full[szb], pol);
                    bulk_load(dst + hb, sc + static_cast<int64_t>(row1) * rowbytes, hb,
                              &bar.sz_full[szb], pol);
                    bulk_load(dst + 2 * hb, zp + static_cast<int64_t>(row0) * rowbytes, hb,
                              &bar.sz_full[szb], pol);
                    bulk_load(dst + 3 * hb, zp + static_cast<int64_t>(row1) * rowbytes, hb,
                              &bar.sz_full[szb], pol);
                    issued_sz |= 1u << szb;
                    issue_ph_sz = (issue_ph_sz & ~(1u << szb)) | (ph_sz << szb);
                    szb ^= 1;
                    if (szb == 0)
                        ph_sz ^= 1;
                }
                bool ok = true;
                for (int kc = 0; kc < p.n_kchunks; kc++) {
                    if (!mbar_wait(&bar.a_empty[sa], ph_a ^ 1, abort_flag, status,
                                   kDevPipelineTimeout)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = stage_a + sa * kStageABytes;
                    mbar_arrive_expect_tx(&bar.a_full[sa], kStageABytes);
                    tma_load_2d(dst, &p.tmap_w, kc * 128, row0, &bar.a_full[sa], pol);
                    tma_load_2d(dst + kStageABytes / 2, &p.tmap_w, kc * 128, row1,
                                &bar.a_full[sa], pol);
                    issued_a |= 1u << sa;
                    issue_ph_a = (issue_ph_a & ~(1u << sa)) | (ph_a << sa);
                    if (++sa == kStagesA) {
                        sa = 0;
                        ph_a ^= 1;
                    }
                }
                if (!ok)
                    break;
            }
            if (*abort_flag) {   // let our own copies land before the CTA exits
                for (int i = 0; i < kStagesA; i++)
                    if (issued_a >> i & 1u)
                        drain_wait(&bar.a_full[i], issue_ph_a >> i & 1u);
                for (int i = 0; i < 2; i++)
                    if (issued_sz >> i & 1u)
                        drain_wait(&bar.sz_full[i], issue_ph_sz >> i & 1u);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int tb = 0, sb = 0;
            uint32_t ph_t = 0, ph_b = 0, ph_acc = 0;
            const uint32_t acc = tmem + kAccCol;
            const uint32_t b_base = smem_u32(stage_b);
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Job J = decode_job(jobs, offs, u / p.n_panels);
                const uint32_t idesc = idesc_f16_f32(kTileRows, J.n);
                const int kb_cap = slot_k(J.n);
                if (!mbar_wait(bar.acc_empty, ph_acc ^ 1, abort_flag, status,
                               kDevPipelineTimeout))
                    break;
                tc_fence_after();
                int kb = 0;   // K offset inside the current activation slot
                for (int kc = 0; kc < p.n_kchunks && ok; kc++) {
                    if (!mbar_wait(&bar.t_full[tb], ph_t, abort_flag, status,
                                   kDevPipelineTimeout)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int steps = min(16, (K - kc * kChunkK) / 16);
                    for (int ks = 0; ks < steps; ks++) {
                        const int kpos = kc * kChunkK + ks * 16;
                        if (kb == 0) {
                            if (!mbar_wait(&bar.b_full[sb], ph_b, abort_flag, status,
                                           kDevPipelineTimeout)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t baddr = b_base + sb * kStageBBytes +
                                               (kb >> 6) * (J.n * 128) + ((kb & 63) >> 4) * 32;
                        tc_mma_ts(acc, tmem + tb * 128 + ks * 8, sdesc_sw128(baddr), idesc,
                                  kpos > 0 ? 1u : 0u);
                        kb += 16;
                        if (kb == kb_cap || kpos + 16 == K) {
                            tc_commit(&bar.b_empty[sb]);
                            kb = 0;
                            if (++sb == kStagesB) {
                                sb = 0;
                                ph_b ^= 1;
                            }
                        }
                    }
                    if (!ok)
                        break;
                    tc_commit(&bar.t_empty[tb]);
                    tb ^= 1;
                    if (tb == 0)
                        ph_t ^= 1;
                }
                if (!ok)
                    break;
                tc_commit(bar.acc_full);
                ph_acc ^= 1;
            }
            // all MMAs issued by this thread complete before TMEM is freed
            tc_commit(bar.drain);
            drain_wait(bar.drain, 0);
        }
    } else if (warp < 8) {
        // ---------------------------------------------- activation producers
        const int bt = tid - 64;
        int sb = 0;
        uint32_t ph_b = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const int kb_cap = slot_k(J.n);
            for (int k_lo = 0; k_lo < K; k_lo += kb_cap) {
                if (!mbar_wait(&bar.b_empty[sb], ph_b ^ 1, abort_flag, status,
                               kDevPipelineTimeout)) {
                    ok = false;
                    break;
                }
                const int cpr = min(kb_cap, K - k_lo) >> 3;     // 16-byte chunks per row
                const int total = J.n * cpr;
                uint8_t *slot = stage_b + sb * kStageBBytes;
                const int cb_stride = J.n * 128;
                for (int i0 = bt; i0 < total; i0 += 4 * kNumBThreads) {
                    uint4 v[4];
                    int dst[4];
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const int i = i0 + r * kNumBThreads;
                        v[r] = make_uint4(0, 0, 0, 0);
                        dst[r] = -1;
                        if (i < total) {
                            const int row = i / cpr, c8 = i - row * cpr;
                            const int kk = k_lo + c8 * 8;
                            if constexpr (GATE_UP) {
                                const int a = __ldg(p.sorted_ids + J.start + row);
                                if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A)) {
                                    const int t = a / p.k;
                                    v[r] = __ldg(reinterpret_cast<const uint4 *>(
                                        p.act + static_cast<int64_t>(t) * K + kk));
                                }
                            } else {
                                v[r] = __ldg(reinterpret_cast<const uint4 *>(
                                    p.act + static_cast<int64_t>(J.start + row) * K + kk));
                            }
                            const int cb = c8 >> 3, cc = c8 & 7;
                            dst[r] = cb * cb_stride + (row >> 3) * 1024 + (row & 7) * 128 +
                                     ((cc ^ (row & 7)) << 4);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        if (dst[r] >= 0) {
                            const uint4 o = GATE_UP ? bf16x8_to_f16_perm(v[r]) : f16x8_perm(v[r]);
                            *reinterpret_cast<uint4 *>(slot + dst[r]) = o;
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&bar.b_full[sb]);
                if (++sb == kStagesB) {
                    sb = 0;
                    ph_b ^= 1;
                }
            }
        }
    } else {
        // ------------------------------------------------ dequant + epilogue
        const int q4 = warp & 3;            // TMEM lane quarter
        const int half = (warp - 8) >> 2;   // which 128-wide half of a K chunk
        const int row = GATE_UP ? (lane < 16 ? 16 * q4 + lane : 64 + 16 * q4 + (lane - 16))
                                : 32 * q4 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        int sa = 0, tb = 0, szb = 0;
        uint32_t ph_a = 0, ph_t = 0, ph_sz = 0, ph_acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const int pnl = u % p.n_panels;
            if (!mbar_wait(&bar.sz_full[szb], ph_sz, abort_flag, status, kDevPipelineTimeout))
                break;
            const __half *s_row =
                reinterpret_cast<const __half *>(sz_base + szb * p.sz_bytes) + row * p.G;
            const __half *z_row = s_row + kTileRows * p.G;
            for (int kc = 0; kc < p.n_kchunks; kc++) {
                if (!mbar_wait(&bar.a_full[sa], ph_a, abort_flag, status,
                               kDevPipelineTimeout)) {
                    ok = false;
                    break;
                }
                const uint8_t *rp = stage_a + sa * kStageABytes + row * 128;
                uint4 wv[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    const int chunk = half * 4 + c4;
                    wv[c4] = *reinterpret_cast<const uint4 *>(rp + ((chunk ^ (row & 7)) << 4));
                }
                mbar_arrive(&bar.a_empty[sa]);
                if (++sa == kStagesA) {
                    sa = 0;
                    ph_a ^= 1;
                }
                if (!mbar_wait(&bar.t_empty[tb], ph_t ^ 1, abort_flag, status,
                               kDevPipelineTimeout)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int k0 = kc * kChunkK + half * 128;
#pragma unroll
                for (int qq = 0; qq < 2; qq++) {
                    const int kq = k0 + qq * 64;
                    if (kq < K) {
                        const int g = kq / p.group;
                        const __half sh = s_row[g];
                        const __half ch =
                            __float2half_rn(-__half2float(z_row[g]) * __half2float(sh));
                        const __half2 s2 = __half2half2(sh), c2 = __half2half2(ch);
                        uint32_t o[32];
                        const uint32_t wq[8] = {wv[2 * qq].x,     wv[2 * qq].y,
                                                wv[2 * qq].z,     wv[2 * qq].w,
                                                wv[2 * qq + 1].x, wv[2 * qq + 1].y,
                                                wv[2 * qq + 1].z, wv[2 * qq + 1].w};
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            dequant_word(wq[j], s2, c2, &o[4 * j]);
                        tmem_st_32x32b_x32(tmem + lane_base + tb * 128 + half * 64 + qq * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.t_full[tb]);
                tb ^= 1;
                if (tb == 0)
                    ph_t ^= 1;
            }
            if (!ok)
                break;
            mbar_arrive(&bar.sz_empty[szb]);
            szb ^= 1;
            if (szb == 0)
                ph_sz ^= 1;

            // ------------------------------------------------------ epilogue
            if (!mbar_wait(bar.acc_full, ph_acc, abort_flag, status, kDevPipelineTimeout))
                break;
            ph_acc ^= 1;
            tc_fence_after();
            const int ncol = J.n >> 1;
            const int col0 = half * ncol;
            for (int c = 0; c < ncol; c += 8) {
                uint32_t v[8];
                tmem_ld_32x32b_x8(tmem + lane_base + kAccCol + col0 + c, v);
                if constexpr (GATE_UP) {
                    __half *hout = reinterpret_cast<__half *>(p.out);
                    const bool is_gate = lane < 16;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t send = is_gate ? v[4 + i] : v[i];
                        const uint32_t recv = __shfl_xor_sync(full, send, 16);
                        const float g = __uint_as_float(is_gate ? v[i] : recv);
                        const float uu = __uint_as_float(is_gate ? recv : v[4 + i]);
                        const float hv = gelu_tanh(g) * uu;
                        const int col = col0 + c + (is_gate ? i : 4 + i);
                        const int64_t slot = J.start + col;
                        const uint32_t hb = f16x2_sat(hv, 0.0f);
                        hout[slot * p.out_cols + pnl * 64 + 16 * q4 + (lane & 15)] =
                            __ushort_as_half(static_cast<unsigned short>(hb & 0xffffu));
                    }
                } else {
                    float *yout = reinterpret_cast<float *>(p.out);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int slot = J.start + col0 + c + i;
                        const int a = __ldg(p.sorted_ids + slot);
                        if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A))
                            yout[static_cast<int64_t>(a) * p.out_cols + pnl * 128 + 32 * q4 +
                                 lane] = __uint_as_float(v[i]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar.acc_empty);
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------- host
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

struct DeviceInfo {
    int sms = 0, smem_optin = 0;
    bool attr_set[2] = {false, false};
};

DeviceInfo &device_info(int dev)
{
    static DeviceInfo info[64];
    DeviceInfo &d = info[dev & 63];
    if (d.sms == 0) {
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return d;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem &q, cudaStream_t stream,
                                const char **why)
{
    *why = nullptr;
    const int G = q.K / q.group;
    GemmArgs a;
    a.act = q.act;
    a.sc = q.ws;
    a.zp = q.wz;
    a.sorted_ids = q.sorted_ids;
    a.expert_offsets = q.expert_offsets;
    a.out = q.out;
    a.dev_status = q.dev_status;
    a.E = q.E;
    a.k = q.k;
    a.A = q.M * q.k;
    a.K = q.K;
    a.R = q.R;
    a.m_up = q.gate_up ? q.R / 2 : 0;
    a.out_cols = q.out_cols;
    a.group = q.group;
    a.G = G;
    a.n_panels = q.gate_up ? (q.R / 2) / 64 : q.R / 128;
    a.n_kchunks = (q.K + kChunkK - 1) / kChunkK;
    a.sz_bytes = kTileRows * G * 2 * 2;
    a.max_jobs = q.E + static_cast<int>(q.cap / kMaxN) + 1;

    const SmemLayout L = smem_layout(a.sz_bytes, a.E, a.max_jobs);
    const size_t smem = static_cast<size_t>(L.total) + 1024;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    DeviceInfo &di = device_info(dev);
    if (smem > static_cast<size_t>(di.smem_optin)) {
        *why = "shared memory needed by the grouped GEMM exceeds the device limit "
               "(contraction dim or expert count too large)";
        return cudaErrorInvalidValue;
    }

    EncodeTiledFn encode = get_encode_fn();
    if (!encode) {
        *why = "driver entry point cuTensorMapEncodeTiled not available";
        return cudaErrorNotSupported;
    }
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(q.K / 2),
                                static_cast<cuuint64_t>(q.E) * static_cast<cuuint64_t>(q.R)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(q.K / 2)};
    const cuuint32_t box[2] = {128, 64};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult cr = encode(&a.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                               const_cast<uint8_t *>(q.wq), gdim, gstride, box, estride,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected the packed weight tensor";
        return cudaErrorInvalidValue;
    }

    auto kern = q.gate_up ? grouped_gemm_kernel<true> : grouped_gemm_kernel<false>;
    const int which = q.gate_up ? 1 : 0;
    if (!di.attr_set[which]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   di.smem_optin);
        if (err != cudaSuccess)
            return err;
        di.attr_set[which] = true;
    }
    kern<<<di.sms, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace w4
