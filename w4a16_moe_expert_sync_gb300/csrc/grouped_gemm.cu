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
// Design (one persistent CTA per SM, 24 warps, static round-robin schedule):
//   * A work unit is (job, panel).  A job is one expert's slot range of at
//     most 256 slots; a panel is 128 weight rows (gate_up: 64 gate rows and
//     the matching 64 up rows; down: 128 output rows).  Every weight row of an
//     expert is streamed from HBM once per job, whatever the number of tokens.
//   * The MMA is "swap-AB": the 128 dequantised weight rows are the M = 128
//     operand and the expert's tokens are N (16..256).  The A operand lives in
//     tensor memory: dequant warps write fp16 weights straight from registers
//     with tcgen05.st, so the expanded weights never cost shared-memory
//     bandwidth.  B (activations, fp16) is read by the tensor core from
//     shared memory in the 128-byte-swizzled K-major layout.
//   * Every asynchronous instruction (tcgen05.mma, a TMA copy) holds its
//     issuing thread for ~70-100 cycles on this part, while an MMA with
//     M=128, N=16, K=16 is only a few cycles of tensor work.  Issue is
//     therefore spread over warps: four MMA warps each own every fourth K
//     step of a chunk and their own fp32 accumulator in tensor memory
//     (columns 256..511; fewer issuers when N is large), summed in a fixed
//     order in the epilogue; three TMA warps share the activation tiles.
//   * Warp roles
//       warps 0-3   tcgen05.mma issuers (one lane each); warp 0 owns TMEM.
//       warp 4      TMA: packed nibble tiles (128 rows x 128 B as two 64-row
//                   boxes, SWIZZLE_128B, evict-first) into a 6-stage ring;
//                   the unit's fp16 scales/zeros by bulk copy (double buffer).
//       warps 5-7   TMA: 16-row activation tiles of the slot-ordered input
//                   (gate_up: the gathered activations xg; down: h) into a
//                   3-slot ring.
//       warps 8-23  dequant (four warps per TMEM lane quarter, each 64 of the
//                   256 contraction elements of a chunk), then the epilogue.
//   * Dequantisation of 8 codes held in one 32-bit word costs 13 integer /
//     half2 instructions: the nibbles are ORed into the mantissa of the fp16
//     constant 1024 (exact integers 1024 + q and 1024 + 16q), the 1024 (or 64
//     after a 1/16 scale) is removed exactly, and one half2 FMA applies
//     q * s + (-z * s) with a single rounding.  The codes come out in the
//     block order of korder.cuh; activations and h are stored in that order.
//   * Every output element is written once, by one thread, after a fixed
//     sequence of MMAs and a fixed-order accumulator sum: results are
//     bit-identical run to run.
//   * Every pipeline wait has a time limit; on expiry the CTA raises
//     W4_DEV_PIPELINE_TIMEOUT, stops, drains its own copies and MMAs, frees
//     its tensor memory and exits.
#include <cuda_fp16.h>

#include "korder.cuh"
#include "launch.h"
#include "ptx.cuh"

// Optional pipeline tracing (compile with -DW4_TRACE): CTA 0 records the
// SM clock at twelve points of its pipeline for its first 64 events of each;
// the host reads them with w4_trace_read().  Compiled out by default.
#ifdef W4_TRACE
__device__ unsigned long long g_w4_trace[12][64];
extern "C" int w4_trace_read(void *host)
{
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_w4_trace, sizeof(g_w4_trace)));
}
#define W4_TRACE_POINT(row, idx)                                                     \
    do {                                                                             \
        if (blockIdx.x == 0 && (idx) < 64) {                                         \
            unsigned long long c_;                                                   \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                       \
            g_w4_trace[row][idx] = c_;                                               \
        }                                                                            \
    } while (0)
#else
#define W4_TRACE_POINT(row, idx) ((void)0)
#endif

namespace w4 {

namespace {

constexpr int kNumMmaWarps = 4;             // warps 0-3: MMA issuers
constexpr int kWarpTmaW = 4;                // warp 4: weights + scales/zeros
constexpr int kFirstTmaBWarp = 5;           // warps 5-7: activations
constexpr int kNumTmaBWarps = 3;
constexpr int kFirstDqWarp = 8;             // warps 8-23: dequant + epilogue
constexpr int kNumDqWarps = 16;
constexpr int kNumWarps = kFirstDqWarp + kNumDqWarps;
constexpr int kThreads = 32 * kNumWarps;
constexpr int kStagesA = 6;                 // packed-weight stages
constexpr int kStagesB = 3;                 // activation stages
constexpr int kTileRows = 128;              // MMA M
constexpr int kChunkK = 256;                // K elements per weight stage
constexpr int kStageABytes = kTileRows * kChunkK / 2;   // 16 KB
constexpr int kStageBBytes = 32768;         // N x Kb x 2 B, N*Kb <= 16384
constexpr int kMaxN = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;           // accumulators in columns [256, 512)
// Barriers that many warps feed take one arrival per warp (after a
// __syncwarp), so a phase costs a handful of shared-memory atomics.

struct GemmArgs {
    CUtensorMap tmap_w;     // packed weights [E*R rows, K/2 bytes] u8, box 128 B x 64 rows
    CUtensorMap tmap_b;     // slot-ordered activations [cap, K] fp16 (gate_up: xg,
                            // down: h), box 64 x 16
    const uint16_t *sc;
    const uint16_t *zp;
    const int32_t *sorted_ids;
    const int32_t *expert_offsets;
    void *out;
    int32_t *dev_status;
    int M, E, k, A, K, R, m_up, out_cols, group, G, n_panels, n_kchunks, sz_bytes, max_jobs;
};

struct SmemLayout {
    int off_b, off_sz, off_bar, off_misc, off_offs, off_jobs, total;
};

constexpr int kNumBars = 2 * kStagesA + 2 * kStagesB + 4 + 4 + 2 + kNumMmaWarps;

__host__ __device__ inline SmemLayout smem_layout(int sz_bytes, int E, int max_jobs)
{
    SmemLayout L;
    L.off_b = kStagesA * kStageABytes;
    L.off_sz = L.off_b + kStagesB * kStageBBytes;
    L.off_bar = (L.off_sz + 2 * sz_bytes + 15) & ~15;
    L.off_misc = L.off_bar + 8 * kNumBars;
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

// MMA issuers (each with its own accumulator of n columns) for a job of n
// tokens: as many as fit in the 256 accumulator columns, at most four.
__device__ __forceinline__ int num_issuers(int n)
{
    return max(1, min(kNumMmaWarps, static_cast<int>(kAccCol) / n));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// 8 uint4 codes (one 32-bit word, code i in bits 4i..4i+3) -> 4 fp16x2 words
// in the block order (q0,q4) (q1,q5) (q2,q6) (q3,q7), each s*q + c.
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

__device__ __forceinline__ float gelu_tanh(float v)
{
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}

// Sum of `count` accumulators (column stride `stride`) over 8 columns of this
// thread's TMEM lane, in the fixed order 0, 1, ..., count-1.
__device__ __forceinline__ void tmem_sum_x8(uint32_t taddr, int stride, int count, float (&s)[8])
{
#pragma unroll
    for (int i = 0; i < 8; i++)
        s[i] = 0.0f;
    for (int a = 0; a < count; a += 4) {
        uint32_t r[32];
        const uint32_t t0 = taddr + a * stride;
        const uint32_t t1 = taddr + min(a + 1, count - 1) * stride;
        const uint32_t t2 = taddr + min(a + 2, count - 1) * stride;
        const uint32_t t3 = taddr + min(a + 3, count - 1) * stride;
        tmem_ld_4x_32x32b_x8(t0, t1, t2, t3, r);
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (a + j < count)
#pragma unroll
                for (int i = 0; i < 8; i++)
                    s[i] += __uint_as_float(r[8 * j + i]);
    }
}

// A bounded wait by one lane whose outcome the whole warp follows.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, bool leader,
                                          volatile int *abort_flag, int32_t *status)
{
    int ok = 1;
    if (leader)
        ok = mbar_wait(bar, parity, abort_flag, status, kDevPipelineTimeout) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// A bounded wait for a whole warp: lane 0 polls, the warp follows its
// outcome, and on success every lane observes the completed phase once
// itself (a single try_wait that succeeds) so each lane acquires the data.
__device__ __forceinline__ bool warp_all_wait(uint64_t *bar, uint32_t parity, int lane,
                                              volatile int *abort_flag, int32_t *status)
{
    int ok = 1;
    if (lane == 0)
        ok = mbar_wait(bar, parity, abort_flag, status, kDevPipelineTimeout) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok)
        mbar_try_wait(bar, parity);
    return ok != 0;
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
            mbar_init(&bar.a_empty[i], kNumDqWarps);
        }
        for (int i = 0; i < kStagesB; i++) {
            mbar_init(&bar.b_full[i], kNumTmaBWarps);
            mbar_init(&bar.b_empty[i], kNumMmaWarps);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar.t_full[i], kNumDqWarps);
            mbar_init(&bar.t_empty[i], kNumMmaWarps);
            mbar_init(&bar.sz_full[i], 1);
            mbar_init(&bar.sz_empty[i], kNumDqWarps);
        }
        mbar_init(bar.acc_full, kNumMmaWarps);
        mbar_init(bar.acc_empty, kNumDqWarps);
        for (int i = 0; i < kNumMmaWarps; i++)
            mbar_init(&bar.drain[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTmaW && lane == 0) {
        prefetch_tmap(&p.tmap_w);
        prefetch_tmap(&p.tmap_b);
    }
    for (int i = tid; i <= p.E; i += kThreads)
        offs[i] = __ldg(p.expert_offsets + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // job list: one job per expert and 256-slot chunk of its range
    if (warp == kWarpTmaW) {
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
    const bool leader = lane == 0;

    if (warp == kWarpTmaW) {
        // ------------------------------------------------- TMA: weights, s/z
        // The whole warp walks the schedule; lane 0 waits and issues, and the
        // result of each wait is broadcast so the warp stays converged.
        const uint64_t pol = l2_policy_evict_first();
        int sa = 0, szb = 0;
        uint32_t ph_a = 0, ph_sz = 0;
        uint32_t issued_a = 0, issued_sz = 0;          // bit i: stage used
        uint32_t issue_ph_a = 0, issue_ph_sz = 0;       // phase of last issue
        const uint8_t *sc = reinterpret_cast<const uint8_t *>(p.sc);
        const uint8_t *zp = reinterpret_cast<const uint8_t *>(p.zp);
        const int rowbytes = p.G * 2;
        int n_trace = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const int pnl = u % p.n_panels;
            const int row0 = J.e * p.R + pnl * (GATE_UP ? 64 : 128);
            const int row1 = GATE_UP ? row0 + p.m_up : row0 + 64;
            if (!warp_wait(&bar.sz_empty[szb], ph_sz ^ 1, leader, abort_flag, status))
                break;
            if (leader) {
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
            }
            issued_sz |= 1u << szb;
            issue_ph_sz = (issue_ph_sz & ~(1u << szb)) | (ph_sz << szb);
            szb ^= 1;
            if (szb == 0)
                ph_sz ^= 1;
            for (int kc = 0; kc < p.n_kchunks; kc++) {
                if (!warp_wait(&bar.a_empty[sa], ph_a ^ 1, leader, abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    W4_TRACE_POINT(0, n_trace);
                    uint8_t *dst = stage_a + sa * kStageABytes;
                    mbar_arrive_expect_tx(&bar.a_full[sa], kStageABytes);
                    tma_load_2d(dst, &p.tmap_w, kc * 128, row0, &bar.a_full[sa], pol);
                    tma_load_2d(dst + kStageABytes / 2, &p.tmap_w, kc * 128, row1,
                                &bar.a_full[sa], pol);
                }
                issued_a |= 1u << sa;
                issue_ph_a = (issue_ph_a & ~(1u << sa)) | (ph_a << sa);
                n_trace++;
                if (++sa == kStagesA) {
                    sa = 0;
                    ph_a ^= 1;
                }
            }
        }
        if (leader && *abort_flag) {   // let our own copies land before the CTA exits
            for (int i = 0; i < kStagesA; i++)
                if (issued_a >> i & 1u)
                    drain_wait(&bar.a_full[i], issue_ph_a >> i & 1u);
            for (int i = 0; i < 2; i++)
                if (issued_sz >> i & 1u)
                    drain_wait(&bar.sz_full[i], issue_ph_sz >> i & 1u);
        }
        __syncwarp();
    } else if (warp < kNumMmaWarps) {
        // ------------------------------------------------------- MMA issuers
        // MMA warp i issues the K steps i, i + nis, i + 2 nis, ... of every
        // chunk into its own accumulator (columns 256 + i*n).  Lane 0 waits,
        // issues and commits (a commit tracks its own thread's MMAs); every
        // MMA warp commits once per phase, active or not, so the barrier
        // counts stay fixed.
        const int mw = warp;
        int tb = 0, sb = 0;
        uint32_t ph_t = 0, ph_b = 0, ph_acc = 0;
        const uint32_t b_base = smem_u32(stage_b);
        int n_trace = 0, n_mma = 0, n_slot = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const uint32_t idesc = idesc_f16_f32(kTileRows, J.n);
            const int kb_cap = slot_k(J.n);
            const int nis = num_issuers(J.n);
            const bool active = mw < nis;
            const uint32_t acc_tmem = tmem + kAccCol + mw * J.n;
            if (!warp_wait(bar.acc_empty, ph_acc ^ 1, leader, abort_flag, status))
                break;
            tc_fence_after();
            int kb = 0;        // K offset inside the current activation slot
            int turn = 0;      // K step of the unit modulo nis
            bool first = true; // this issuer's first MMA of the unit
            for (int kc = 0; kc < p.n_kchunks && ok; kc++) {
                if (!warp_wait(&bar.t_full[tb], ph_t, leader, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader && mw == 0)
                    W4_TRACE_POINT(1, n_trace);
                const int steps = min(16, (K - kc * kChunkK) / 16);
                for (int ks = 0; ks < steps; ks++) {
                    const int kpos = kc * kChunkK + ks * 16;
                    if (kb == 0) {
                        if (!warp_wait(&bar.b_full[sb], ph_b, leader, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (leader && mw == 0)
                            W4_TRACE_POINT(10, n_slot);
                        n_slot++;
                    }
                    if (active && turn == mw) {
                        if (leader) {
                            const uint32_t baddr = b_base + sb * kStageBBytes +
                                                   (kb >> 6) * (J.n * 128) + ((kb & 63) >> 4) * 32;
                            if (mw == 0)
                                W4_TRACE_POINT(9, n_mma);
                            tc_mma_ts(acc_tmem, tmem + tb * 128 + ks * 8, sdesc_sw128(baddr), idesc,
                                      first ? 0u : 1u);
                            if (mw == 0)
                                W4_TRACE_POINT(8, n_mma);
                        }
                        n_mma++;
                        first = false;
                    }
                    if (++turn == nis)
                        turn = 0;
                    kb += 16;
                    if (kb == kb_cap || kpos + 16 == K) {
                        if (leader)
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
                if (leader) {
                    if (mw == 0)
                        W4_TRACE_POINT(2, n_trace);
                    tc_commit(&bar.t_empty[tb]);
                }
                n_trace++;
                tb ^= 1;
                if (tb == 0)
                    ph_t ^= 1;
            }
            if (!ok)
                break;
            if (leader)
                tc_commit(bar.acc_full);
            ph_acc ^= 1;
        }
        // all MMAs issued by this thread complete before TMEM is freed
        if (leader) {
            tc_commit(&bar.drain[mw]);
            drain_wait(&bar.drain[mw], 0);
        }
        __syncwarp();
    } else if (warp < kFirstTmaBWarp + kNumTmaBWarps) {
        // --------------------------------------------------- TMA: activations
        // The three activation warps split the 16-row x 64-column tiles of
        // every slot round-robin; each arrives once per slot with the bytes
        // it issued.
        const int bw = warp - kFirstTmaBWarp;
        int sb = 0;
        uint32_t ph_b = 0;
        uint32_t issued_b = 0, issue_ph_b = 0;
        int n_trace = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const int kb_cap = slot_k(J.n);
            const int row_groups = J.n / 16;
            for (int k_lo = 0; k_lo < K; k_lo += kb_cap) {
                if (!warp_wait(&bar.b_empty[sb], ph_b ^ 1, leader, abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    if (bw == 0)
                        W4_TRACE_POINT(3, n_trace);
                    const int kcnt = min(kb_cap, K - k_lo);
                    const int tiles = (kcnt / 64) * row_groups;
                    const int mine = tiles > bw ? (tiles - bw + kNumTmaBWarps - 1) / kNumTmaBWarps : 0;
                    uint8_t *slot = stage_b + sb * kStageBBytes;
                    mbar_arrive_expect_tx(&bar.b_full[sb], static_cast<uint32_t>(mine * 2048));
                    for (int i = bw; i < tiles; i += kNumTmaBWarps) {
                        const int cb = i / row_groups, rg = i - cb * row_groups;
                        tma_load_2d_nohint(slot + cb * (J.n * 128) + rg * 2048, &p.tmap_b,
                                           k_lo + cb * 64, J.start + rg * 16, &bar.b_full[sb]);
                    }
                    if (bw == 0)
                        W4_TRACE_POINT(4, n_trace);
                }
                issued_b |= 1u << sb;
                issue_ph_b = (issue_ph_b & ~(1u << sb)) | (ph_b << sb);
                n_trace++;
                if (++sb == kStagesB) {
                    sb = 0;
                    ph_b ^= 1;
                }
            }
        }
        if (leader && *abort_flag)
            for (int i = 0; i < kStagesB; i++)
                if (issued_b >> i & 1u)
                    drain_wait(&bar.b_full[i], issue_ph_b >> i & 1u);
        __syncwarp();
    } else if (warp >= kFirstDqWarp) {
        // ------------------------------------------------ dequant + epilogue
        const int q4 = warp & 3;                      // TMEM lane quarter
        const int sub = (warp - kFirstDqWarp) >> 2;   // 64-wide slice of a K chunk
        const int row = GATE_UP ? (lane < 16 ? 16 * q4 + lane : 64 + 16 * q4 + (lane - 16))
                                : 32 * q4 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        int sa = 0, tb = 0, szb = 0;
        int n_trace = 0;
        uint32_t ph_a = 0, ph_t = 0, ph_sz = 0, ph_acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Job J = decode_job(jobs, offs, u / p.n_panels);
            const int pnl = u % p.n_panels;
            if (!warp_all_wait(&bar.sz_full[szb], ph_sz, lane, abort_flag, status))
                break;
            const __half *s_row =
                reinterpret_cast<const __half *>(sz_base + szb * p.sz_bytes) + row * p.G;
            const __half *z_row = s_row + kTileRows * p.G;
            for (int kc = 0; kc < p.n_kchunks; kc++) {
                if (!warp_all_wait(&bar.a_full[sa], ph_a, lane, abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (tid == 32 * kFirstDqWarp)
                    W4_TRACE_POINT(5, n_trace);
                const uint8_t *rp = stage_a + sa * kStageABytes + row * 128;
                const uint4 w0 = *reinterpret_cast<const uint4 *>(
                    rp + (((2 * sub) ^ (row & 7)) << 4));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(
                    rp + (((2 * sub + 1) ^ (row & 7)) << 4));
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bar.a_empty[sa]);
                if (++sa == kStagesA) {
                    sa = 0;
                    ph_a ^= 1;
                }
                if (!warp_all_wait(&bar.t_empty[tb], ph_t ^ 1, lane, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tid == 32 * kFirstDqWarp)
                    W4_TRACE_POINT(6, n_trace);
                const int kq = kc * kChunkK + sub * 64;
                if (kq < K) {
                    const int g = kq / p.group;
                    const __half sh = s_row[g];
                    const __half ch = __float2half_rn(-__half2float(z_row[g]) * __half2float(sh));
                    const __half2 s2 = __half2half2(sh), c2 = __half2half2(ch);
                    uint32_t o[32];
                    const uint32_t wq[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        dequant_word(wq[j], s2, c2, &o[4 * j]);
                    if (tid == 32 * kFirstDqWarp)
                        W4_TRACE_POINT(11, n_trace);
                    tmem_st_32x32b_x32(tmem + lane_base + tb * 128 + sub * 32, o);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (tid == 32 * kFirstDqWarp)
                    W4_TRACE_POINT(7, n_trace);
                n_trace++;
                if (lane == 0)
                    mbar_arrive(&bar.t_full[tb]);
                tb ^= 1;
                if (tb == 0)
                    ph_t ^= 1;
            }
            if (!ok)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar.sz_empty[szb]);
            szb ^= 1;
            if (szb == 0)
                ph_sz ^= 1;

            // ------------------------------------------------------ epilogue
            if (!warp_all_wait(bar.acc_full, ph_acc, lane, abort_flag, status))
                break;
            ph_acc ^= 1;
            tc_fence_after();
            const int nis = num_issuers(J.n);
            for (int c = sub * 8; c < J.n; c += 32) {
                float v[8];
                tmem_sum_x8(tmem + lane_base + kAccCol + c, J.n, nis, v);
                if constexpr (GATE_UP) {
                    // lanes 0-15 hold gate rows, lanes 16-31 the matching up
                    // rows: the gate lane finishes columns c..c+3, the up lane
                    // columns c+4..c+7
                    __half *hout = reinterpret_cast<__half *>(p.out);
                    const bool is_gate = lane < 16;
                    const int il = 16 * q4 + (lane & 15);   // intermediate index in panel
                    const int pos = pnl * 64 + (il & ~7) + korder_pos(il & 7);
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float send = is_gate ? v[4 + i] : v[i];
                        const float recv = __shfl_xor_sync(full, send, 16);
                        const float g = is_gate ? v[i] : recv;
                        const float uu = is_gate ? recv : v[4 + i];
                        const float hv = gelu_tanh(g) * uu;
                        const int64_t slot = J.start + c + (is_gate ? i : 4 + i);
                        hout[slot * p.out_cols + pos] =
                            __ushort_as_half(static_cast<unsigned short>(f16x2_sat(hv, 0.0f)));
                    }
                } else {
                    float *yout = reinterpret_cast<float *>(p.out);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int a = __ldg(p.sorted_ids + J.start + c + i);
                        if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A))
                            yout[static_cast<int64_t>(a) * p.out_cols + pnl * 128 + 32 * q4 +
                                 lane] = v[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar.acc_empty);
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
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

bool encode_2d(EncodeTiledFn encode, CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
               uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
               uint32_t box_outer)
{
    const cuuint64_t gdim[2] = {inner, outer};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, dtype, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem &q, cudaStream_t stream,
                                const char **why)
{
    *why = nullptr;
    const int G = q.K / q.group;
    GemmArgs a;
    a.sc = q.ws;
    a.zp = q.wz;
    a.sorted_ids = q.sorted_ids;
    a.expert_offsets = q.expert_offsets;
    a.out = q.out;
    a.dev_status = q.dev_status;
    a.M = q.M;
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
    // packed weights: rows of K/2 bytes, boxes of 128 B x 64 rows
    if (!encode_2d(encode, &a.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, q.wq, q.K / 2,
                   static_cast<uint64_t>(q.E) * q.R, q.K / 2, 128, 64)) {
        *why = "cuTensorMapEncodeTiled rejected the packed weight tensor";
        return cudaErrorInvalidValue;
    }
    // slot-ordered activations [cap, K] fp16 (gate_up: xg, down: h): 16-row tiles
    if (!encode_2d(encode, &a.tmap_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.act, q.K,
                   static_cast<uint64_t>(q.cap), static_cast<uint64_t>(q.K) * 2, 64, 16)) {
        *why = "cuTensorMapEncodeTiled rejected the activation tensor";
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
