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
// s, z per group of `group` elements along the contraction dim.
//
// Dequantisation.  Eight codes sit in one 32-bit word; ORing a masked pair
// of nibbles into the mantissa of fp16 1024.0 gives 1024 + q (or 1024 + 16q
// for the high nibbles) exactly; one HADD2 (or HFMA2 by 1/16) leaves q, and
// one HFMA2 makes q * s + c with c = fp16(-z * s), a single rounding of the
// product.  Per word that is one shift and four LOP3 on the integer pipe and
// eight fp16 operations on the FMA pipe, which issue in parallel.
//
// Design (one persistent CTA per SM, 26 warps, static round-robin schedule):
//   * A work unit is (job, panel).  A job is at most 32 consecutive slots of
//     one expert; a panel is 128 weight rows (gate_up: 64 gate rows and the
//     matching 64 up rows; down: 128 output rows).
//   * Swap-AB: the 128 weight rows are the M = 128 operand, in tensor memory
//     (written with tcgen05.st), the job's tokens are N (16 or 32).  B, the
//     activations, is read by the tensor core from shared memory in the
//     128-byte-swizzled K-major layout; one 3-D TMA copy fills a 32 KB slot.
//   * A tcgen05.mma holds its issuing thread for ~100 cycles on this part
//     whatever its size, so four issuer warps share the work: the unit's
//     64-element sub-chunks go round-robin to them, each into its own fp32
//     accumulator; the epilogue adds the four in a fixed order.
//   * Warp roles
//       warps 0-3   tcgen05.mma issuers (one lane each).
//       warps 4-7   epilogue (one TMEM lane quarter each).
//       warps 8-23  dequant: four per lane quarter, one 64-code sub-chunk of
//                   each 256-code chunk each (warps 8 + 4 i + q feed issuer i).
//       warp 24     TMA: packed codes (128 rows x 256 codes per stage, two
//                   64-row boxes, evict-first), per unit the scales, zeros
//                   and activation group sums (bulk copies).
//       warp 25     TMA: activation slots.
//   * Tensor memory: columns 0-255 eight A sub-chunk buffers (64 codes, 32
//     columns each), two per issuer, so every buffer has one producer group
//     (the dequant warps of one half) and one consumer, both in order;
//     columns 256-511 two sets of four 32-column accumulators, alternating
//     per unit, so a unit's epilogue overlaps the next unit's MMAs.
//   * Every barrier wait is at most one phase ahead of the barrier (each
//     waiter waits on every phase of its barriers in order), which is what
//     makes the parity waits exact.
//   * Every output element is written once, by one thread, after a fixed
//     sequence of MMAs and fixed-order sums: results are bit-identical run to
//     run.
//   * Every pipeline wait has a time limit; on expiry the CTA raises
//     W4_DEV_PIPELINE_TIMEOUT, stops, drains its own copies and MMAs, frees
//     its tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "korder.cuh"
#include "launch.h"
#include "ptx.cuh"

// Optional pipeline tracing (compile with -DW4_TRACE): CTA 0 records the SM
// clock at sixteen points of its pipeline for its first 128 events of each;
// the host reads them with w4_trace_read().  Compiled out by default.
#ifdef W4_TRACE
__device__ unsigned long long g_w4_trace[16][128];
extern "C" int w4_trace_read(void *host)
{
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_w4_trace, sizeof(g_w4_trace)));
}
#define W4_TRACE_POINT(row, idx)                                                     \
    do {                                                                             \
        if (blockIdx.x == 0 && (idx) < 128) {                                        \
            unsigned long long c_;                                                   \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                       \
            g_w4_trace[row][idx] = c_;                                               \
        }                                                                            \
    } while (0)
// First pipeline wait in the grid that ran out: block, warp, lane, barrier
// index, parity, clock.
__device__ unsigned long long g_w4_timeout[8];
extern "C" int w4_timeout_read(void *host)
{
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_w4_timeout, sizeof(g_w4_timeout)));
}
extern "C" int w4_timeout_reset(void)
{
    unsigned long long z[8] = {};
    return static_cast<int>(cudaMemcpyToSymbol(g_w4_timeout, z, sizeof(z)));
}
// Per block and warp: the wait each warp gave up on (shared address | parity << 31).
__device__ unsigned int g_w4_gaveup[256][32];
extern "C" int w4_gaveup_read(void *host)
{
    return static_cast<int>(cudaMemcpyFromSymbol(host, g_w4_gaveup, sizeof(g_w4_gaveup)));
}
#define W4_TIMEOUT_RECORD(bar, parity, status)                                              \
    do {                                                                                    \
        if (blockIdx.x < 256)                                                               \
            g_w4_gaveup[blockIdx.x][threadIdx.x >> 5] =                                     \
                w4::smem_u32(bar) | (static_cast<unsigned>(parity) << 31);                  \
        if ((status) && (*(volatile int32_t *)(status) & 2) &&                              \
            atomicCAS(&g_w4_timeout[0], 0ull, 1ull) == 0ull) {                              \
            g_w4_timeout[1] = blockIdx.x;                                                   \
            g_w4_timeout[2] = threadIdx.x >> 5;                                             \
            g_w4_timeout[3] = threadIdx.x & 31;                                             \
            g_w4_timeout[4] = w4::smem_u32(bar);                                              \
            g_w4_timeout[5] = (parity);                                                     \
            unsigned long long c_;                                                          \
            asm volatile("mov.u64 %0, %%clock64;" : "=l"(c_));                              \
            g_w4_timeout[6] = c_;                                                           \
        }                                                                                   \
    } while (0)
#else
#define W4_TRACE_POINT(row, idx) ((void)0)
#define W4_TIMEOUT_RECORD(bar, parity, status) ((void)0)
#endif

namespace w4 {

namespace {

constexpr int kIssuers = 4;                 // warps 0-3
constexpr int kFirstEpiWarp = 4;            // warps 4-7
constexpr int kNumEpiWarps = 4;
constexpr int kFirstDqWarp = 8;             // warps 8-15
constexpr int kNumDqWarps = 16;            // warps 8-23
constexpr int kWarpTmaW = 24;
constexpr int kWarpTmaB = 25;
constexpr int kNumWarps = 26;
constexpr int kThreads = 32 * kNumWarps;
constexpr int kStagesW = 5;                 // packed-code stages
constexpr int kStagesB = 3;                 // activation slots
constexpr int kStagesSZ = 3;                // per-unit scales, zeros, group sums
constexpr int kTileRows = 128;              // MMA M
constexpr int kChunkK = 256;                // codes per row per stage
constexpr int kSubK = 64;                   // codes per A sub-chunk
constexpr int kMaxSubBufs = 12;             // A buffers in tensor memory (kIssuers x BUFS)
constexpr int kStageWBytes = kTileRows * kChunkK / 2;   // 16 KB
constexpr int kStageBBytes = 32768;
constexpr int kResSlotBytes = kStagesB * kStageBBytes / 2;   // resident mode: 2 x 48 KB
constexpr int kMaxN = 32;                   // slots per job
constexpr uint32_t kTmemCols = 512;
// Tensor memory: A buffer b at column 32 b (b = issuer + kIssuers * slot), then
// the accumulators acc[set][issuer] at acc_col<BUFS> + 128 set + 32 issuer.
// BUFS = 3 A buffers per issuer leave room for one accumulator set, BUFS = 2
// for two (the next unit's MMAs need not wait for the epilogue).
template <int BUFS>
__host__ __device__ constexpr int acc_sets() { return BUFS >= 3 ? 1 : 2; }
template <int BUFS>
__host__ __device__ constexpr uint32_t acc_col() { return 32u * kIssuers * BUFS; }
static_assert(acc_col<3>() + 128u * acc_sets<3>() <= kTmemCols, "tensor memory budget");
static_assert(acc_col<2>() + 128u * acc_sets<2>() <= kTmemCols, "tensor memory budget");
constexpr int kBufsGateUp = 2;
constexpr int kBufsDown = 2;

struct GemmArgs {
    CUtensorMap tmap_w;       // packed codes u8 [E*R rows, K/2 B], box 128 B x 64 rows, SW128
    CUtensorMap tmap_b[2];    // activations [cap, K] fp16 as {64, cap, K/64}, box {64, 16(i+1), kcols}
    const uint16_t *sc;       // [E*R, G] fp16
    const uint16_t *zp;       // [E*R, G] fp16
    const int32_t *sorted_ids;
    const int32_t *expert_offsets;
    void *out;
    int32_t *dev_status;
    int E, A, K, R, m_up, out_cols, group, group_shift, G, n_panels, n_kchunks, n_sub;
    int early_schedule;       // the schedule may be read before the grid-dependency wait
    int out_bf16;             // plain epilogue: bf16 rows instead of fp32
};

constexpr int kNumBars = 2 * kStagesW + 2 * kStagesB + 2 * kMaxSubBufs + 2 + 2 + 2 * kStagesSZ + kIssuers;

struct Bars {
    uint64_t *w_full, *w_empty, *b_full, *b_empty, *a_full, *a_empty, *acc_full, *acc_empty,
        *sz_full, *sz_empty, *drain;
};

__device__ __forceinline__ Bars carve_bars(uint8_t *base)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    Bars r;
    r.w_full = b;
    r.w_empty = r.w_full + kStagesW;
    r.b_full = r.w_empty + kStagesW;
    r.b_empty = r.b_full + kStagesB;
    r.a_full = r.b_empty + kStagesB;
    r.a_empty = r.a_full + kMaxSubBufs;
    r.acc_full = r.a_empty + kMaxSubBufs;
    r.acc_empty = r.acc_full + 2;
    r.sz_full = r.acc_empty + 2;
    r.sz_empty = r.sz_full + kStagesSZ;
    r.drain = r.sz_empty + kStagesSZ;
    return r;
}

struct SmemLayout {
    int off_b, off_sz, off_bar, off_misc, off_offs, off_jp;
    int sz_stride, total;
};

// One sz stage: s [128 rows][G] fp16, then z [128][G] fp16.
__host__ __device__ inline SmemLayout smem_layout(int G, int E)
{
    SmemLayout L;
    L.off_b = kStagesW * kStageWBytes;
    L.sz_stride = ((kTileRows * G * 2 * 2) + 127) & ~127;
    L.off_sz = L.off_b + kStagesB * kStageBBytes;
    L.off_bar = L.off_sz + kStagesSZ * L.sz_stride;
    L.off_misc = L.off_bar + kNumBars * 8;
    L.off_offs = L.off_misc + 16;
    L.off_jp = L.off_offs + (E + 1) * 4;
    L.total = L.off_jp + (E + 1) * 4;
    return L;
}

struct Job {
    int e, start, n;
};

// Job j of the schedule: the expert whose job range holds j (jp = exclusive
// prefix of jobs per expert) and its j - jp[e]-th block of kMaxN slots.
__device__ __forceinline__ Job decode_job(const int *jp, const int *offs, int E, int j)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (jp[mid] <= j)
            lo = mid;
        else
            hi = mid - 1;
    }
    Job J;
    J.e = lo;
    J.start = offs[lo] + (j - jp[lo]) * kMaxN;
    J.n = min(kMaxN, offs[lo + 1] - J.start);
    return J;
}

// 64-code column blocks per activation slot for a job of n slots (32 KB).
__host__ __device__ constexpr int b_kcols(int n) { return n == 16 ? 16 : 8; }

// Resident mode: the activation block of a full job (kMaxN slots x K) fits
// one of two 48 KB slots and is loaded once per job, not once per unit.
__host__ __device__ constexpr bool b_fits_resident(int K)
{
    return K / 64 <= 256 && static_cast<int64_t>(K) * 2 * kMaxN <= kResSlotBytes;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// (a & MASK) | magic in one LOP3, the mask an immediate and the magic
// constant in a register (two immediates would cost a second LOP3).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t magic)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "r"(magic));
    return r;
}

// 8 codes (one word, code i in bits 4i..4i+3) -> 4 words of fp16 pairs
// q * s + c in the block order (q0,q4) (q1,q5) (q2,q6) (q3,q7).  `magic` holds
// fp16 1024.0 twice.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 c2, uint32_t magic,
                                             uint32_t *o)
{
    const __half2 k1024 = u2h(magic);
    const __half2 kSixteenth = u2h(0x2C002C00u);           // 1/16
    const __half2 kMinus64 = u2h(0xD400D400u);             // -64
    const uint32_t w8 = w >> 8;
    const __half2 q04 = __hsub2(u2h(and_or<0x000F000Fu>(w, magic)), k1024);
    const __half2 q15 = __hfma2(u2h(and_or<0x00F000F0u>(w, magic)), kSixteenth, kMinus64);
    const __half2 q26 = __hsub2(u2h(and_or<0x000F000Fu>(w8, magic)), k1024);
    const __half2 q37 = __hfma2(u2h(and_or<0x00F000F0u>(w8, magic)), kSixteenth, kMinus64);
    o[0] = h2u(__hfma2(q04, s2, c2));
    o[1] = h2u(__hfma2(q15, s2, c2));
    o[2] = h2u(__hfma2(q26, s2, c2));
    o[3] = h2u(__hfma2(q37, s2, c2));
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

__device__ __forceinline__ float lds_half_as_float(uint32_t saddr)
{
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(saddr));
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float gelu_tanh(float v)
{
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}

// A bounded wait by every lane of a warp (each lane observes the phase
// itself, which gives it acquire ordering); the vote keeps the warp's
// control flow uniform if the wait ever times out.
__device__ __forceinline__ bool warp_all_wait(uint64_t *bar, uint32_t parity, int lane,
                                              volatile int *abort_flag, int32_t *status)
{
    const bool ok = mbar_wait_warp(bar, parity, abort_flag, status, kDevPipelineTimeout);
    if (!ok && lane == 0)
        W4_TIMEOUT_RECORD(bar, parity, status);
    return ok;
}

__device__ __forceinline__ bool lane_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, status, kDevPipelineTimeout);
    if (!ok)
        W4_TIMEOUT_RECORD(bar, parity, status);
    return ok;
}

// bounded wait that ignores the abort flag (used only while draining)
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 200000000ull)
            return;
}

// Tile row (0..127 of the stage) held by lane `lane` of a warp of TMEM lane
// quarter q4.  gate_up pairs gate row i with up row i in lanes l and l + 16.
template <bool GATE_UP>
__device__ __forceinline__ int tile_row(int q4, int lane)
{
    if constexpr (GATE_UP)
        return lane < 16 ? 16 * q4 + lane : 64 + 16 * q4 + (lane - 16);
    else
        return 32 * q4 + lane;
}

// RESIDENT: each job's activations are loaded once into one of two 48 KB
// slots (contraction dim <= 768); otherwise they stream through 32 KB slots.
template <bool GATE_UP, int BUFS, bool RESIDENT>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs p)
{
    constexpr int kSets = acc_sets<BUFS>();
    constexpr uint32_t kAccCol = acc_col<BUFS>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemLayout L = smem_layout(p.G, p.E);
    uint8_t *stage_w = smem;
    uint8_t *stage_b = smem + L.off_b;
    uint8_t *sz_base = smem + L.off_sz;
    const Bars bar = carve_bars(smem + L.off_bar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    int *offs = reinterpret_cast<int *>(smem + L.off_offs);
    int *jp = reinterpret_cast<int *>(smem + L.off_jp);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned full = 0xffffffffu;
    int32_t *status = p.dev_status;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < kStagesW; i++) {
            mbar_init(&bar.w_full[i], 1);
            mbar_init(&bar.w_empty[i], kNumDqWarps);
        }
        for (int i = 0; i < kStagesB; i++) {
            mbar_init(&bar.b_full[i], 1);
            mbar_init(&bar.b_empty[i], kIssuers);
        }
        for (int i = 0; i < kMaxSubBufs; i++) {
            mbar_init(&bar.a_full[i], 4);            // the four lane quarters
            mbar_init(&bar.a_empty[i], 1);           // the issuer's commit
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar.acc_full[i], kIssuers);
            mbar_init(&bar.acc_empty[i], kNumEpiWarps);
        }
        for (int i = 0; i < kStagesSZ; i++) {
            mbar_init(&bar.sz_full[i], 1);
            mbar_init(&bar.sz_empty[i], kNumDqWarps);
        }
        for (int i = 0; i < kIssuers; i++)
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
        prefetch_tmap(&p.tmap_b[0]);
        prefetch_tmap(&p.tmap_b[1]);
    }
    // everything above touched only this CTA; from here on the inputs of the
    // preceding kernels are read (the schedule possibly early, see GemmArgs)
    if (!p.early_schedule) {
        pdl_wait();
        pdl_trigger();
    }
    for (int i = tid; i <= p.E; i += kThreads)
        offs[i] = __ldg(p.expert_offsets + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // jobs per expert (ceil(slots / kMaxN)), exclusive prefix in jp[0..E]
    if (warp == kFirstEpiWarp) {
        int base = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            const int nj = e < p.E ? (offs[e + 1] - offs[e] + kMaxN - 1) / kMaxN : 0;
            int inc = nj;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(full, inc, o);
                if (lane >= o)
                    inc += v;
            }
            if (e < p.E)
                jp[e] = base + inc - nj;
            base += __shfl_sync(full, inc, 31);
        }
        if (lane == 0)
            jp[p.E] = base;
    }
    __syncthreads();

    const uint32_t tmem = *tmem_holder;
    const int n_units = jp[p.E] * p.n_panels;
    const int K = p.K;

    if (warp < kIssuers) {
        // ------------------------------------------------------- MMA issuers
        // Each issuer warp runs this loop converged (every value in it is
        // warp-uniform) and one elected lane issues each tcgen05 instruction,
        // which costs the warp far fewer cycles than issuing from a lone lane.
        {
            const int me = warp;
            const uint32_t b_base = smem_u32(stage_b);
            uint32_t b_seq = 0, n_unit = 0;
            uint32_t a_slot = 0, a_ph = 0;   // this issuer's next A buffer and its phase
            int n_tr = 0;
            int cur_job = -1;       // resident mode: the job whose activations are held
            uint32_t res_slot = 0;
            bool ok = true;
            // One 64-code sub-chunk: wait for its A buffer, four K=16 MMAs, and
            // hand the buffer back when they complete.
            auto issue = [&](uint32_t d_tmem, uint64_t bdesc, uint32_t idesc, bool first) -> bool {
                const int buf = me + kIssuers * a_slot;
                if (!warp_all_wait(&bar.a_full[buf], a_ph, lane, abort_flag, status))
                    return false;
                if (++a_slot == BUFS) {
                    a_slot = 0;
                    a_ph ^= 1;
                }
                tc_fence_after();
                if (me == 0 && lane == 0)
                    W4_TRACE_POINT(5, n_tr);
                const uint32_t a_tmem = tmem + buf * 32;
                // K steps of 16: +32 B in the swizzled row (+2 in the
                // descriptor's address field), +8 columns of A
                tc_mma_ts_elect(d_tmem, a_tmem, bdesc, idesc, first ? 0u : 1u);
                tc_mma_ts_elect(d_tmem, a_tmem + 8, bdesc + 2, idesc, 1u);
                tc_mma_ts_elect(d_tmem, a_tmem + 16, bdesc + 4, idesc, 1u);
                tc_mma_ts_elect(d_tmem, a_tmem + 24, bdesc + 6, idesc, 1u);
                tc_commit_elect(&bar.a_empty[buf]);
                if (me == 0 && lane == 0)
                    W4_TRACE_POINT(6, n_tr);
                n_tr++;
                return true;
            };
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, n_unit++) {
                const int job = u / p.n_panels;
                const Job J = decode_job(jp, offs, p.E, job);
                const uint32_t idesc = idesc_f16_f32(kTileRows, J.n);
                const uint32_t col_bytes = static_cast<uint32_t>(J.n) * 128;
                const int set = kSets == 1 ? 0 : (n_unit & 1);
                const uint32_t acc_ph = (kSets == 1 ? n_unit : n_unit >> 1) & 1;
                if (!warp_all_wait(&bar.acc_empty[set], acc_ph ^ 1, lane, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + kAccCol + set * 128 + me * 32;
                if constexpr (RESIDENT) {
                    // the job's activations stay in one slot for all its units
                    if (job != cur_job) {
                        if (cur_job >= 0)
                            tc_commit_elect(&bar.b_empty[res_slot]);
                        res_slot = b_seq & 1;
                        if (!warp_all_wait(&bar.b_full[res_slot], (b_seq >> 1) & 1, lane, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        b_seq++;
                        cur_job = job;
                    }
                    const uint32_t b_slot = b_base + res_slot * kResSlotBytes;
                    for (int j = me; j < p.n_sub; j += kIssuers) {
                        if (!issue(d_tmem, sdesc_sw128(b_slot + static_cast<uint32_t>(j) * col_bytes),
                                   idesc, j == me)) {
                            ok = false;
                            break;
                        }
                    }
                } else {
                    const int kb_cap = 64 * b_kcols(J.n);
                    const int n_bslots = (K + kb_cap - 1) / kb_cap;
                    bool first = true;
                    for (int t = 0; t < n_bslots && ok; t++) {
                        const int sb = (b_seq + t) % kStagesB;
                        if (!warp_all_wait(&bar.b_full[sb], ((b_seq + t) / kStagesB) & 1, lane, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t b_slot = b_base + sb * kStageBBytes;
                        const int j0 = t * (kb_cap / kSubK);
                        const int j1 = min(p.n_sub, j0 + kb_cap / kSubK);
                        // my sub-chunks in this slot: j = me (mod kIssuers); sub-chunk
                        // j - j0 of the slot is its (j - j0)-th 64-wide column block
                        for (int j = j0 + ((me - j0) % kIssuers + kIssuers) % kIssuers; j < j1;
                             j += kIssuers) {
                            if (!issue(d_tmem,
                                       sdesc_sw128(b_slot + static_cast<uint32_t>(j - j0) * col_bytes),
                                       idesc, first)) {
                                ok = false;
                                break;
                            }
                            first = false;
                        }
                        if (!ok)
                            break;
                        tc_commit_elect(&bar.b_empty[sb]);
                    }
                    b_seq += n_bslots;
                }
                if (!ok)
                    break;
                tc_commit_elect(&bar.acc_full[set]);
            }
            // every MMA of this warp completes before tensor memory is freed
            tc_commit_elect(&bar.drain[me]);
            drain_wait(&bar.drain[me], 0);
        }
        __syncwarp();
    } else if (warp == kWarpTmaW) {
        // ----------------------------------- TMA: codes, scales/zeros, sums
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int sa = 0, szb = 0, n_tr = 0;
            uint32_t ph_a = 0, ph_sz = 0;
            uint32_t issued_a = 0, issue_ph_a = 0, issued_sz = 0, issue_ph_sz = 0;
            const uint32_t hb = 64u * p.G * 2;          // 64 rows of s (or z)
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Job J = decode_job(jp, offs, p.E, u / p.n_panels);
                const int pnl = u % p.n_panels;
                const int row0 = J.e * p.R + pnl * (GATE_UP ? 64 : 128);
                const int row1 = GATE_UP ? row0 + p.m_up : row0 + 64;
                if (!lane_wait(&bar.sz_empty[szb], ph_sz ^ 1, abort_flag, status))
                    break;
                {
                    uint8_t *dst = sz_base + szb * L.sz_stride;
                    mbar_arrive_expect_tx(&bar.sz_full[szb], 4 * hb);
                    bulk_load(dst, p.sc + static_cast<int64_t>(row0) * p.G, hb, &bar.sz_full[szb],
                              pol);
                    bulk_load(dst + hb, p.sc + static_cast<int64_t>(row1) * p.G, hb,
                              &bar.sz_full[szb], pol);
                    bulk_load(dst + 2 * hb, p.zp + static_cast<int64_t>(row0) * p.G, hb,
                              &bar.sz_full[szb], pol);
                    bulk_load(dst + 3 * hb, p.zp + static_cast<int64_t>(row1) * p.G, hb,
                              &bar.sz_full[szb], pol);
                }
                issued_sz |= 1u << szb;
                issue_ph_sz = (issue_ph_sz & ~(1u << szb)) | (ph_sz << szb);
                if (++szb == kStagesSZ) {
                    szb = 0;
                    ph_sz ^= 1;
                }
                for (int kc = 0; kc < p.n_kchunks; kc++) {
                    if (!lane_wait(&bar.w_empty[sa], ph_a ^ 1, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    W4_TRACE_POINT(0, n_tr);
                    n_tr++;
                    uint8_t *dst = stage_w + sa * kStageWBytes;
                    mbar_arrive_expect_tx(&bar.w_full[sa], kStageWBytes);
                    tma_load_2d(dst, &p.tmap_w, kc * 128, row0, &bar.w_full[sa], pol);
                    tma_load_2d(dst + kStageWBytes / 2, &p.tmap_w, kc * 128, row1, &bar.w_full[sa],
                                pol);
                    issued_a |= 1u << sa;
                    issue_ph_a = (issue_ph_a & ~(1u << sa)) | (ph_a << sa);
                    if (++sa == kStagesW) {
                        sa = 0;
                        ph_a ^= 1;
                    }
                }
            }
            if (*abort_flag) {   // let our own copies land before the CTA exits
                for (int i = 0; i < kStagesW; i++)
                    if (issued_a >> i & 1u)
                        drain_wait(&bar.w_full[i], issue_ph_a >> i & 1u);
                for (int i = 0; i < kStagesSZ; i++)
                    if (issued_sz >> i & 1u)
                        drain_wait(&bar.sz_full[i], issue_ph_sz >> i & 1u);
            }
        }
        __syncwarp();
    } else if (warp == kWarpTmaB) {
        // --------------------------------------------------- TMA: activations
        if (p.early_schedule && lane == 0) {
            // the activations are the preceding kernel's output
            pdl_wait();
            pdl_trigger();
        }
        if (lane == 0) {
            int sb = 0, n_tr = 0;
            uint32_t ph_b = 0, issued_b = 0, issue_ph_b = 0;
            bool ok = true;
            if constexpr (RESIDENT) {
                // one load per job into slot b_seq & 1, once the issuers have
                // released that slot's previous job
                int cur_job = -1;
                uint32_t b_seq = 0;
                for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                    const int job = u / p.n_panels;
                    if (job == cur_job)
                        continue;
                    cur_job = job;
                    const Job J = decode_job(jp, offs, p.E, job);
                    const int s = b_seq & 1;
                    const uint32_t ph = (b_seq >> 1) & 1;
                    if (!lane_wait(&bar.b_empty[s], ph ^ 1, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    W4_TRACE_POINT(1, n_tr);
                    n_tr++;
                    mbar_arrive_expect_tx(&bar.b_full[s],
                                          static_cast<uint32_t>(J.n) * 128 * p.n_sub);
                    tma_load_3d(stage_b + s * kResSlotBytes, &p.tmap_b[J.n / 16 - 1], 0, J.start,
                                0, &bar.b_full[s]);
                    issued_b |= 1u << s;
                    issue_ph_b = (issue_ph_b & ~(1u << s)) | (ph << s);
                    b_seq++;
                }
            } else {
                for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                    const Job J = decode_job(jp, offs, p.E, u / p.n_panels);
                    const CUtensorMap *map = &p.tmap_b[J.n / 16 - 1];
                    const int kcols = b_kcols(J.n);
                    const uint32_t bytes = static_cast<uint32_t>(J.n) * 128 * kcols;
                    for (int k_lo = 0; k_lo < K; k_lo += 64 * kcols) {
                        if (!lane_wait(&bar.b_empty[sb], ph_b ^ 1, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        W4_TRACE_POINT(1, n_tr);
                        n_tr++;
                        mbar_arrive_expect_tx(&bar.b_full[sb], bytes);
                        tma_load_3d(stage_b + sb * kStageBBytes, map, 0, J.start, k_lo / 64,
                                    &bar.b_full[sb]);
                        issued_b |= 1u << sb;
                        issue_ph_b = (issue_ph_b & ~(1u << sb)) | (ph_b << sb);
                        if (++sb == kStagesB) {
                            sb = 0;
                            ph_b ^= 1;
                        }
                    }
                }
            }
            if (*abort_flag)
                for (int i = 0; i < kStagesB; i++)
                    if (issued_b >> i & 1u)
                        drain_wait(&bar.b_full[i], issue_ph_b >> i & 1u);
        }
        __syncwarp();
    } else if (warp >= kFirstDqWarp && warp < kFirstDqWarp + kNumDqWarps) {
        // ---------------------------------------------------------- dequant
        // Warp (q4, sub) expands sub-chunk sub of every chunk for its 32 rows:
        // sub-chunk j = 4 kc + sub goes to issuer sub, into that issuer's
        // buffers sub and sub + 4, alternating.
        const int q4 = warp & 3;
        const int sub = (warp - kFirstDqWarp) >> 2;
        const int row = tile_row<GATE_UP>(q4, lane);
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        int sa = 0, szb = 0, n_tr = 0;
        uint32_t ph_a = 0, ph_sz = 0, n_unit = 0;
        uint32_t a_slot = 0, a_ph = 0;   // next A buffer of issuer `sub`, and its phase
        const uint32_t stage_w_s = smem_u32(stage_w), sz_base_s = smem_u32(sz_base);
        const uint32_t code_off0 = static_cast<uint32_t>(row * 128 + (((2 * sub) ^ (row & 7)) << 4));
        const uint32_t code_off1 =
            static_cast<uint32_t>(row * 128 + (((2 * sub + 1) ^ (row & 7)) << 4));
        uint32_t magic;   // fp16 1024.0 twice, kept in a register
        asm("mov.b32 %0, 0x64006400;" : "=r"(magic));
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, n_unit++) {
            if (!warp_all_wait(&bar.sz_full[szb], ph_sz, lane, abort_flag, status))
                break;
            const uint32_t s_addr = sz_base_s + szb * L.sz_stride + 2 * row * p.G;
            for (int kc = 0; kc < p.n_kchunks; kc++) {
                if (!warp_all_wait(&bar.w_full[sa], ph_a, lane, abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (warp == kFirstDqWarp && lane == 0)
                    W4_TRACE_POINT(2, n_tr);
                const int j = kc * (kChunkK / kSubK) + sub;   // sub-chunk in unit
                const bool mine = j < p.n_sub;
                const uint32_t rp = stage_w_s + sa * kStageWBytes;
                uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
                float sf = 0.0f, zf = 0.0f;
                if (mine) {
                    w0 = lds128(rp + code_off0);
                    w1 = lds128(rp + code_off1);
                    const uint32_t g = static_cast<uint32_t>(j * kSubK) >> p.group_shift;
                    sf = lds_half_as_float(s_addr + 2 * g);
                    zf = lds_half_as_float(s_addr + 2 * (kTileRows * p.G + g));
                }
                __syncwarp();
                mbar_arrive_elect(&bar.w_empty[sa]);
                if (++sa == kStagesW) {
                    sa = 0;
                    ph_a ^= 1;
                }
                if (!mine)
                    continue;
                const int buf = sub + kIssuers * a_slot;
                if (!warp_all_wait(&bar.a_empty[buf], a_ph ^ 1, lane, abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (++a_slot == BUFS) {
                    a_slot = 0;
                    a_ph ^= 1;
                }
                if (warp == kFirstDqWarp && lane == 0)
                    W4_TRACE_POINT(4, n_tr);
                tc_fence_after();
                const __half2 s2 = __float2half2_rn(sf);
                const __half2 c2 = __float2half2_rn(-zf * sf);
                uint32_t o[32];
                dequant_word(w0.x, s2, c2, magic, &o[0]);
                dequant_word(w0.y, s2, c2, magic, &o[4]);
                dequant_word(w0.z, s2, c2, magic, &o[8]);
                dequant_word(w0.w, s2, c2, magic, &o[12]);
                dequant_word(w1.x, s2, c2, magic, &o[16]);
                dequant_word(w1.y, s2, c2, magic, &o[20]);
                dequant_word(w1.z, s2, c2, magic, &o[24]);
                dequant_word(w1.w, s2, c2, magic, &o[28]);
                if (warp == kFirstDqWarp && lane == 0)
                    W4_TRACE_POINT(8, n_tr);
                tmem_st_32x32b_x32(tmem + lane_base + buf * 32, o);
                tmem_wait_st();
                if (warp == kFirstDqWarp && lane == 0)
                    W4_TRACE_POINT(14, n_tr);
                tc_fence_before();
                __syncwarp();
                mbar_arrive_elect(&bar.a_full[buf]);
                if (warp == kFirstDqWarp && lane == 0)
                    W4_TRACE_POINT(3, n_tr);
                n_tr++;
            }
            if (!ok)
                break;
            __syncwarp();
            mbar_arrive_elect(&bar.sz_empty[szb]);
            if (++szb == kStagesSZ) {
                szb = 0;
                ph_sz ^= 1;
            }
        }
    } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + kNumEpiWarps) {
        // ---------------------------------------------------------- epilogue
        const int q4 = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        const int n_acc = min(kIssuers, p.n_sub);
        // gate_up: lanes 0-15 hold gate rows, lanes 16-31 the matching up rows;
        // the gate lane finishes even slots, the up lane odd ones
        const bool is_gate = lane < 16;
        const int il = 16 * q4 + (lane & 15);     // intermediate index in the panel
        uint32_t n_unit = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, n_unit++) {
            const Job J = decode_job(jp, offs, p.E, u / p.n_panels);
            const int pnl = u % p.n_panels;
            const int set = kSets == 1 ? 0 : (n_unit & 1);
            const uint32_t acc_ph = (kSets == 1 ? n_unit : n_unit >> 1) & 1;
            // down: the assignment of every slot of the job, fetched early
            int my_a = -1;
            if constexpr (!GATE_UP)
                my_a = lane < J.n ? __ldg(p.sorted_ids + J.start + lane) : -1;
            if (!warp_all_wait(&bar.acc_full[set], acc_ph, lane, abort_flag, status))
                break;
            if (warp == kFirstEpiWarp && lane == 0)
                W4_TRACE_POINT(10, n_unit);
            tc_fence_after();
            // Per block of 8 slots: the issuers' accumulators, added in a fixed
            // order (issuers without a sub-chunk in this unit never wrote
            // theirs), then the outputs.  The set goes back to the issuers as
            // soon as its last block is in registers.
            const uint32_t acc = tmem + lane_base + kAccCol + set * 128;
            const int n_blk = J.n / 8;
#pragma unroll
            for (int b = 0; b < kMaxN / 8; b++) {
                if (b >= n_blk)
                    break;
                float v[8];
                {
                    uint32_t r[32];
                    tmem_ld_4x_32x32b_x8(acc + 8 * b, acc + 32 + 8 * b, acc + 64 + 8 * b,
                                         acc + 96 + 8 * b, r);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        float t = __uint_as_float(r[i]);
                        if (n_acc > 1)
                            t += __uint_as_float(r[8 + i]);
                        if (n_acc > 2)
                            t += __uint_as_float(r[16 + i]);
                        if (n_acc > 3)
                            t += __uint_as_float(r[24 + i]);
                        v[i] = t;
                    }
                }
                if (b == n_blk - 1) {
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_elect(&bar.acc_empty[set]);
                }
                if constexpr (GATE_UP) {
                    __half *hout = reinterpret_cast<__half *>(p.out);
                    const int pos = pnl * 64 + (il & ~7) + korder_pos(il & 7);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const float send = is_gate ? v[i + 1] : v[i];
                        const float recv = __shfl_xor_sync(full, send, 16);
                        const float gv = is_gate ? v[i] : recv;
                        const float uv = is_gate ? recv : v[i + 1];
                        const int64_t slot = J.start + 8 * b + i + (is_gate ? 0 : 1);
                        hout[slot * p.out_cols + pos] = __ushort_as_half(
                            static_cast<uint16_t>(f16x2_sat(gelu_tanh(gv) * uv, 0.0f)));
                    }
                } else {
                    const int col = pnl * 128 + 32 * q4 + lane;
                    if (p.out_bf16) {
                        uint16_t *bout = reinterpret_cast<uint16_t *>(p.out);
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const int a = __shfl_sync(full, my_a, 8 * b + i);
                            if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A))
                                bout[static_cast<int64_t>(a) * p.out_cols + col] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
                        }
                    } else {
                        float *yout = reinterpret_cast<float *>(p.out);
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const int a = __shfl_sync(full, my_a, 8 * b + i);
                            if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A))
                                yout[static_cast<int64_t>(a) * p.out_cols + col] = v[i];
                        }
                    }
                }
            }
            if (warp == kFirstEpiWarp && lane == 0)
                W4_TRACE_POINT(11, n_unit);
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
    bool attr_set[3] = {false, false, false};
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

// Activations [cap, K] fp16 viewed as {64 elements, cap rows, K/64 column
// blocks} (strides 2K bytes and 128 bytes), so that one box
// {64, rows, kcols} lands in shared memory as kcols consecutive
// [rows x 128 B] swizzled blocks, the K-major layout the MMA reads.
bool encode_act(EncodeTiledFn encode, CUtensorMap *map, const void *base, int64_t cap, int K,
                int rows, int kcols)
{
    const cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(cap),
                                static_cast<cuuint64_t>(K / 64)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(kcols)};
    const cuuint32_t estride[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), gdim, gstride,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem &q, cudaStream_t stream,
                                const char **why)
{
    *why = nullptr;
    if (q.K % q.group != 0 || q.K % 64 != 0 || (q.group != 64 && q.group != 128)) {
        *why = "contraction dim must be a multiple of the group (64 or 128) and of 64";
        return cudaErrorInvalidValue;
    }
    GemmArgs a;
    a.sc = q.ws;
    a.zp = q.wz;
    a.sorted_ids = q.sorted_ids;
    a.expert_offsets = q.expert_offsets;
    a.out = q.out;
    a.dev_status = q.dev_status;
    a.E = q.E;
    a.A = q.M * q.k;
    a.K = q.K;
    a.R = q.R;
    a.m_up = q.gate_up ? q.R / 2 : 0;
    a.out_cols = q.out_cols;
    a.group = q.group;
    a.group_shift = q.group == 128 ? 7 : 6;
    a.G = q.K / q.group;
    a.n_panels = q.gate_up ? (q.R / 2) / 64 : q.R / 128;
    a.n_kchunks = (q.K + kChunkK - 1) / kChunkK;
    a.n_sub = q.K / kSubK;
    a.early_schedule = q.early_schedule ? 1 : 0;
    a.out_bf16 = q.out_bf16 ? 1 : 0;
    const bool resident = !q.gate_up && b_fits_resident(q.K);

    const SmemLayout L = smem_layout(a.G, a.E);
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
    // packed codes: rows of K/2 bytes, boxes of 128 B x 64 rows
    if (!encode_2d(encode, &a.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, q.wq, q.K / 2,
                   static_cast<uint64_t>(q.E) * q.R, q.K / 2, 128, 64)) {
        *why = "cuTensorMapEncodeTiled rejected the packed weight tensor";
        return cudaErrorInvalidValue;
    }
    for (int i = 0; i < 2; i++) {
        const int rows = 16 * (i + 1);
        const int kcols = resident ? q.K / 64 : b_kcols(rows);
        if (!encode_act(encode, &a.tmap_b[i], q.act, q.cap, q.K, rows, kcols)) {
            *why = "cuTensorMapEncodeTiled rejected the activation tensor";
            return cudaErrorInvalidValue;
        }
    }

    auto kern = q.gate_up ? grouped_gemm_kernel<true, kBufsGateUp, false>
                : resident ? grouped_gemm_kernel<false, kBufsDown, true>
                           : grouped_gemm_kernel<false, kBufsDown, false>;
    const int which = q.gate_up ? 2 : (resident ? 1 : 0);
    if (!di.attr_set[which]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   di.smem_optin);
        if (err != cudaSuccess)
            return err;
        di.attr_set[which] = true;
    }
    return launch_pdl(kern, dim3(di.sms), dim3(kThreads), smem, stream, a);
}

}  // namespace w4
