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
// Dequantisation.  Eight codes sit in one 32-bit word (code i in bits
// 4i..4i+3).  ANDing the word with 0x000F000F leaves codes 0 and 4 as the
// bit patterns of two fp16 subnormals, q * 2^-24, exactly; 0x00F000F0 leaves
// codes 1 and 5 as 16 q * 2^-24 (still subnormal: the first 10 bits of an
// fp16 are its mantissa); the word shifted right by 8 gives codes 2, 6 and
// 3, 7 the same way.  One HFMA2 per pair then forms
//     A = q * S + C,  S = s * 2^(24 - c),  C = fp16(-s * z * 2^-c)
// (S / 16 for the 16 q pairs): the product q * s * 2^-c is exact inside the
// fused operation and A is rounded once, i.e. A = 2^-c * fp16(q s + fp16(-z s))
// wherever that value is an fp16 normal.  c is a power-of-two exponent per
// weight row, chosen from the row's largest scale so that every S of the row
// is a finite fp16 (S <= 65504 needs s * 2^(24 - c) below 2^16); the epilogue
// multiplies the row's fp32 accumulator by 2^c, which is exact.  So a weight
// costs 5/8 integer and 4/8 fp16 operations: one shift and four LOP3 plus
// four HFMA2 per eight codes.
//
// Group-constant correction.  Rounding C to fp16 leaves an error that is the
// same for every weight of the group, so it adds up over the group as
// (C_exact - C) * (sum of the group's activations) instead of averaging out.
// The activation rows therefore end in a 64-column block of group sums (the
// gather writes one per group of 128 of x, gate_up's epilogue one per
// quarter of each group of 64 of h) and every unit ends with a correction
// sub-chunk: per row the low parts C_lo = fp16(C_exact - C) (exact in fp32
// before that rounding) as the A operand, one to four K = 16 MMAs against the
// sum block.  The dequantised weight is then exact to its own fp16 rounding.
//
// Design (one persistent CTA of 28 warps per SM, static round-robin schedule):
//   * A work unit is (job, panel).  A job is at most 32 consecutive slots of
//     one expert (64 in big-job mode, when the experts average 64 or more
//     slots); a panel is 128 weight rows (gate_up: 64 gate rows and the
//     matching 64 up rows; down: 128 output rows).
//   * Swap-AB: the 128 weight rows are the M = 128 operand, in tensor memory
//     (written with tcgen05.st), the job's tokens are N (16 or 32; up to 64
//     in big-job mode).  B, the
//     activations, is read by the tensor core from shared memory in the
//     128-byte-swizzled K-major layout; 3-D TMA copies fill its slots (or, for
//     down, one copy per job fills a resident slot).
//   * Codes arrive by TMA in stages of 128 rows x 256 codes (two 64-row
//     boxes), evict-first in L2.  A stage is four 64-code slices (the unit's
//     blocks 4 kc .. 4 kc + 3).  Ring r (two 32-column A buffers in tensor
//     memory, taken in turn) takes slice r of every stage; four dequant
//     warps per ring (one per lane quarter) expand it.
//   * Four issuer warps: issuer r issues each of ring r's fills as four
//     K = 16 MMAs and the commit that frees the buffer, in one issue block,
//     into its own fp32 accumulator ("chain").  The epilogue adds the chains
//     in a fixed order.  Two accumulator sets alternate per unit, so a
//     unit's epilogue overlaps the next unit's MMAs.  The unit's correction
//     goes, after that ring's last block, to the ring with one block fewer
//     (blocks % 4), or to ring unit % 4 when the rings have as many.  In
//     big-job mode issuers 0 and 1 take rings r and r + 2 each, into two
//     chains of 64 columns, and issuers 2-3 idle.
//   * Warp roles
//       warps 0-3   tcgen05.mma issuers (converged, one elected lane issues);
//                   warp 0 also allocates tensor memory
//       warps 4-7   epilogue (one TMEM lane quarter each)
//       warps 8-23  dequant (warp 8 + 4 r + q: lane quarter q, ring r)
//       warp 24     TMA: per unit the scales and zeros, and the code stages
//                   of parity 0 of the CTA's stage sequence
//       warp 27     TMA: the code stages of parity 1
//       warp 25     TMA: activation slots
//       warp 26     gate_up: sets the counters of the combine folded into
//                   down (combine_fold.cuh); in down, after its last unit,
//                   every warp of the CTA counts the CTA's y panels and
//                   combines the (token, panel) pairs it completed
//   * Tensor memory (512 columns): A buffers at 32 (2 r + b), accumulators
//     at 256 + 128 set + 32 chain (big jobs: + 64 chain).
//   * Every barrier has one producer group and one consumer group that take
//     its phases in order, so a waiter is never two phases ahead and parity
//     waits are exact (tests/test_grouped_pipeline_protocol.py models it).
//   * Every output element is written once, by one thread, after a fixed
//     sequence of MMAs: results are bit-identical run to run.
//   * Every pipeline wait has a time limit; on expiry the CTA raises
//     W4_DEV_PIPELINE_TIMEOUT, stops, drains its own copies and MMAs, frees
//     its tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "checks.cuh"
#include "combine_fold.cuh"
#include "korder.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4 {

namespace {

constexpr int kNumIssuers = 4;              // warps 0-3: issuer r takes ring r
constexpr int kWarpAlloc = 0;               // tensor-memory allocation (an issuer)
constexpr int kWarpTmaW = 24;              // scales/zeros and parity-0 code stages
constexpr int kWarpTmaW1 = 27;             // parity-1 code stages
constexpr int kWarpTmaB = 25;
constexpr int kFirstEpiWarp = 4;
constexpr int kNumEpiWarps = 4;
constexpr int kFirstDqWarp = 8;
constexpr int kNumDqWarps = 16;            // warp 8 + 4 r + q: lane quarter q, ring r
constexpr int kWarpComb = 26;               // gate_up: sets the folded combine's counters
constexpr int kNumWarps = 28;
constexpr int kThreads = 32 * kNumWarps;
// Ring r takes slice r (codes 64 r .. 64 r + 63) of every stage into its
// two A buffers in turn: all sixteen dequant warps work on every stage, so a
// stage is free as soon as each has read its slice, and a ring's four warps
// fill one buffer while the tensor core reads the other.
constexpr int kRings = 4;
constexpr int kRingBufs = 2;                // A buffers per ring
constexpr int kStagesW = 6;                 // packed-code stages
constexpr int kStagesB = 3;                 // streamed activation slots
constexpr int kMaxStagesSZ = 3;             // per-unit scales and zeros
constexpr int kTileRows = 128;              // MMA M
constexpr int kChunkK = 256;                // codes per row per stage
constexpr int kSliceK = 64;                 // codes per fill (one A buffer)
constexpr int kFillCols = kSliceK / 2;      // TMEM columns per A buffer
constexpr int kStageWBytes = kTileRows * kChunkK / 2;   // 16 KB
constexpr int kStageBBytes = 32768;
constexpr int kResSlotBytes = kStagesB * kStageBBytes / 2;   // resident mode: 2 x 48 KB
constexpr int kMaxN = 32;                   // slots per job
// Big-job mode (many tokens per expert): jobs of up to 64 slots, so each
// weight panel is dequantised once per 64 tokens; its accumulators take
// twice the columns, so two issuers take two rings each and keep two
// chains.  Activations always stream in this mode.
constexpr int kMaxNBig = 64;
template <bool BIGN> struct JobShape {
    static constexpr int kMaxN = BIGN ? kMaxNBig : ::w4::kMaxN;
    static constexpr int kIssuers = BIGN ? 2 : 4;   // issuers with MMAs (= chains)
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = kRings * kRingBufs * kFillCols;  // 256
// Accumulators: one per issuer ("chain" i of issuer i), at kAccCol + 128 set
// + 32 i, the set alternating per unit.
constexpr int kChains = kNumIssuers;
// Row scales 2^c handed from the dequant warps to the epilogue, one table
// per unit for the last eight units.  The ring-0 dequant warps write unit n's
// after claiming the buffer of its block 0, i.e. after the MMAs of ring 0's
// fill two fills earlier; every unit gives ring 0 at least one fill (block
// 0), so those MMAs belong to unit n - 2 or later and waited for the
// epilogue of unit n - 4 to release its accumulators, which it does after
// reading its table: the table of unit n - 8 is free.
constexpr int kRowScaleSets = 8;
// The (token, panel) combines a down CTA completes, kept until its last unit
// (a longer list is combined as it overflows).
constexpr int kCombListCap = 1024;
static_assert(kAccCol + 2 * kChains * kMaxN <= kTmemCols, "tensor memory budget");
static_assert(kAccCol + 2 * JobShape<true>::kIssuers * kMaxNBig <= kTmemCols,
              "tensor memory budget (big jobs)");
static_assert(kStagesW % 2 == 0, "a dequant warp must see every phase of its stage slots");

struct GemmArgs {
    CUtensorMap tmap_w;       // packed codes u8 [E*R rows, K/2 B], box 128 B x 64 rows, SW128
    CUtensorMap tmap_b[4];    // activations [cap, K] fp16 as {64, cap, K/64}, box {64, 16(i+1), kcols}
    const uint16_t *sc;       // [E*R, G] fp16
    const uint16_t *zp;       // [E*R, G] fp16
    const int32_t *sorted_ids;
    const int32_t *expert_offsets;
    void *out;
    int32_t *dev_status;
    int E, A, K, R, m_up, out_cols, group_shift, G, n_panels, n_kchunks, n_blocks, n_sz;
    int n_corr_mma;           // K = 16 MMAs of the group-constant correction
    int h_stride;             // gate_up: row length of h (m + 64: values, then group sums)
    int h_groups;             // gate_up: groups of 64 along m (the down GEMM's groups)
    int acc_mask[4];          // issuers (accumulators) with MMAs in the CTA's unit n,
                              // by n % 4 (the correction's ring may rotate)
    int early_schedule;       // the schedule may be read before the grid-dependency wait
    // The layer's combine, folded into the down GEMM (comb_cnt non-null):
    // counters [M][d/128 panels][4 lane quarters], set by the gate_up launch
    // before it (to k minus the token's valid assignments; it also zeroes
    // the out rows of tokens with none) and counted up by the down
    // epilogue; the warp that completes a counter writes those 32 columns
    // of out.
    const int32_t *topk_ids;  // [M, k]
    const float *topk_w;      // [M, k]
    int32_t *comb_cnt;
    uint16_t *comb_out;       // [M, d] bf16
    int M, k, comb_d;
    int64_t cap;              // alignment slots (rows of xg / h)
    // test hooks: the pipeline wait limit (ns), and whether the first unit's
    // scale/zero copy is withheld (so that the waits run out)
    uint64_t wait_ns;
    int test_withhold_sz;
};

constexpr int kNumBars = 2 * kStagesW + 2 * kStagesB + 2 * kRings * kRingBufs + 2 + 2 +
                         2 * kMaxStagesSZ + kNumIssuers;

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
    r.a_empty = r.a_full + kRings * kRingBufs;
    r.acc_full = r.a_empty + kRings * kRingBufs;
    r.acc_empty = r.acc_full + 2;
    r.sz_full = r.acc_empty + 2;
    r.sz_empty = r.sz_full + kMaxStagesSZ;
    r.drain = r.sz_empty + kMaxStagesSZ;
    return r;
}

struct SmemLayout {
    int off_b, off_sz, off_bar, off_misc, off_offs, off_jp, off_rs, off_cl;
    int sz_stride, total;
};

// Scale/zero stages: s [128 rows][G] fp16, then z [128][G] fp16.  Three
// stages when a unit's are small (down), two otherwise (gate_up: a unit is 11
// code stages, so the copy of the next unit's scales is never waited for).
__host__ __device__ inline int sz_stages(int G) { return G > 16 ? 2 : 3; }

__host__ __device__ inline SmemLayout smem_layout(int G, int E, bool gate_up)
{
    SmemLayout L;
    L.off_b = kStagesW * kStageWBytes;
    L.sz_stride = ((kTileRows * G * 2 * 2) + 127) & ~127;
    L.off_sz = L.off_b + kStagesB * kStageBBytes;
    L.off_bar = L.off_sz + sz_stages(G) * L.sz_stride;
    L.off_misc = L.off_bar + kNumBars * 8;
    L.off_offs = L.off_misc + 16;
    L.off_jp = L.off_offs + (E + 1) * 4;
    L.off_rs = (L.off_jp + (E + 1) * 4 + 15) & ~15;
    L.off_cl = L.off_rs + kRowScaleSets * kTileRows * 4;
    // down: the combine list (its count in the misc words)
    L.total = L.off_cl + (gate_up ? 0 : kCombListCap * 4);
    return L;
}

struct Job {
    int e, start, n;
};

// Job j of the schedule: the expert whose job range holds j (jp = exclusive
// prefix of jobs per expert) and its j - jp[e]-th block of maxn slots.
__device__ __forceinline__ Job decode_job(const int *jp, const int *offs, int E, int j,
                                          int maxn = kMaxN)
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
    J.start = offs[lo] + (j - jp[lo]) * maxn;
    J.n = min(maxn, offs[lo + 1] - J.start);
    return J;
}

// 64-code column blocks per streamed activation slot for a job of n slots.
__host__ __device__ constexpr int b_kcols(int n) { return kStageBBytes / (n * 128); }

// Resident mode: the activation block of a full job (kMaxN slots x K) fits
// one of two 48 KB slots and is loaded once per job, not once per unit.
__host__ __device__ constexpr bool b_fits_resident(int K)
{
    return static_cast<int64_t>(K + 64) * 2 * kMaxN <= kResSlotBytes;   // with the sums block
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// 8 codes (one word) -> 4 words of fp16 pairs A = q * S + C in the block
// order (q0,q4) (q1,q5) (q2,q6) (q3,q7); the codes enter as fp16 subnormals
// (q or 16 q times 2^-24), S16 = S / 16 serves the 16 q pairs.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 S, __half2 S16, __half2 C,
                                             uint32_t *o)
{
    const uint32_t w8 = w >> 8;
    o[0] = h2u(__hfma2(u2h(w & 0x000F000Fu), S, C));
    o[1] = h2u(__hfma2(u2h(w & 0x00F000F0u), S16, C));
    o[2] = h2u(__hfma2(u2h(w8 & 0x000F000Fu), S, C));
    o[3] = h2u(__hfma2(u2h(w8 & 0x00F000F0u), S16, C));
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t saddr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr)
{
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(saddr));
    return h;
}

// The row exponent c from the largest |scale| bit pattern of the row (for
// non-negative fp16 values the bit patterns order like the values): with f
// the biased exponent of that scale, c = max(f, 1) - 6 makes every scale of
// the row times 2^(24 - c) an fp16 of exponent at most 15, i.e. <= 65504.
__device__ __forceinline__ int row_exponent(uint32_t smax_bits)
{
    const int f = min(static_cast<int>(smax_bits >> 10), 30);
    return max(f, 1) - 6;
}

// The largest |scale| bit pattern among the G scales of a row in shared
// memory at s_addr: a 16-bit load up to the first 4-byte boundary, then two
// scales per 32-bit load with a packed 16-bit max, then the odd last one.
__device__ __forceinline__ uint32_t row_smax(uint32_t s_addr, int G)
{
    uint32_t smax = 0;
    if (s_addr & 2u) {
        smax = lds_u16(s_addr) & 0x7FFFu;
        s_addr += 2;
        G--;
    }
    uint32_t m2 = 0;
#pragma unroll 2
    for (int i = 0; i < (G >> 1); i++)
        m2 = __vmaxu2(m2, lds_u32(s_addr + 4 * i) & 0x7FFF7FFFu);
    smax = max(smax, max(m2 & 0xFFFFu, m2 >> 16));
    if (G & 1)
        smax = max(smax, lds_u16(s_addr + 2 * (G - 1)) & 0x7FFFu);
    return smax;
}

__device__ __forceinline__ float exp2i(int e)   // 2^e for -126 <= e <= 127, exact
{
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// The dequant constants of one group: S, S / 16 and C (see dequant_word).
struct GroupK {
    __half2 S, S16, C;
};

__device__ __forceinline__ GroupK group_consts(uint32_t s_bits, uint32_t z_bits, float scale_s,
                                               float scale_c)
{
    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(s_bits)));
    const float z = __half2float(__ushort_as_half(static_cast<unsigned short>(z_bits)));
    GroupK g;
    // power-of-two scalings of an fp16 value: exact
    g.S = __float2half2_rn(s * scale_s);
    g.S16 = __float2half2_rn(s * scale_s * 0.0625f);
    // s * z is exact in fp32 (two 11-bit significands); one rounding to fp16
    g.C = __float2half2_rn(-(s * z) * scale_c);
    return g;
}

// gelu_tanh(v) = 0.5 v (1 + tanh(u)), u = sqrt(2/pi) (v + 0.044715 v^3),
// evaluated as v / (1 + e^(-2u)) (the same function: 1 + tanh(u) =
// 2 / (1 + e^(-2u))) with the fast exponential and division, a relative
// error of a few units of fp32 against the fp16 rounding of h that
// follows; e^(-2u) = inf for large negative v gives the limit -0.
__device__ __forceinline__ float gelu_tanh(float v)
{
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    const float u = c * fmaf(0.044715f * v, v * v, v);
    return __fdividef(v, 1.0f + __expf(-2.0f * u));
}

// A bounded wait by every lane of a warp (each lane observes the phase
// itself, which gives it acquire ordering); the vote keeps the warp's
// control flow uniform if the wait ever times out.
// What a pipeline wait needs besides its barrier: the CTA's abort flag, the
// device status word and the time limit (one second unless a test shortens it).
struct WaitCtx {
    volatile int *abort_flag;
    int32_t *status;
    uint64_t limit_ns;
};

__device__ __forceinline__ bool warp_all_wait(uint64_t *bar, uint32_t parity, const WaitCtx &wc)
{
    return mbar_wait_warp(bar, parity, wc.abort_flag, wc.status, kDevPipelineTimeout,
                          wc.limit_ns);
}

__device__ __forceinline__ bool warp_all_wait_a(uint32_t bar, uint32_t parity, const WaitCtx &wc)
{
    return mbar_wait_warp_a(bar, parity, wc.abort_flag, wc.status, kDevPipelineTimeout,
                            wc.limit_ns);
}

__device__ __forceinline__ bool lane_wait(uint64_t *bar, uint32_t parity, const WaitCtx &wc)
{
    return mbar_wait(bar, parity, wc.abort_flag, wc.status, kDevPipelineTimeout, wc.limit_ns);
}

// bounded wait that ignores the abort flag (used only while draining)
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 200000000ull)
            return;
}

// The ring of the unit's 64-code block j (slice j % 4 of stage j / 4).
__host__ __device__ __forceinline__ int block_ring(int j) { return j & (kRings - 1); }

// The ring that carries the correction fill of the CTA's unit n (after the
// ring's last block of the unit).  When the block count is not a multiple of
// four, the ring the next block would go to: it has one block fewer than
// ring 0, so the correction evens the rings' fills out (down at m = 704: 11
// blocks, rings 3/3/3/2).  Otherwise every ring has as many blocks, and the
// correction turns by one per unit, so that over four units every ring takes
// one.
__host__ __device__ __forceinline__ int corr_ring(int n_unit, int n_blocks)
{
    const int rest = n_blocks & (kRings - 1);
    return rest ? rest : (n_unit & (kRings - 1));
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

// ------------------------------------------------- the combine, folded in
// out[t, pnl*128 .. +128] = bf16(sum over j = 0..k-1 in order of w_j y_j) by
// one warp (four columns per lane): the fp32 chain acc = fma(w_j, y_j, acc)
// from 0 over the token's valid assignments, rounded once, as the standalone
// combine computes it, so the result does not depend on which CTA completed
// the counter.  The y rows of all k assignments are loaded at once (rows of
// invalid ids are loaded but unused); y is read from L2 (written in this
// launch by other CTAs).
__device__ __forceinline__ void combine_panel(const GemmArgs &p, int t, int pnl, int lane)
{
    const unsigned full = 0xffffffffu;
    const int col = pnl * 128 + 4 * lane;
    const float *y = reinterpret_cast<const float *>(p.out);
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int j0 = 0; j0 < p.k; j0 += 8) {
        // ids and weights of 8 assignments on lanes 0-7, their y rows on all
        const int jl = j0 + (lane & 7);
        const int64_t aj = static_cast<int64_t>(t) * p.k + jl;
        const int e = jl < p.k ? __ldg(p.topk_ids + aj) : -1;
        const float wv = jl < p.k ? __ldg(p.topk_w + aj) : 0.0f;
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; u++)
            v[u] = j0 + u < p.k ? __ldcg(reinterpret_cast<const float4 *>(
                                      y + (static_cast<int64_t>(t) * p.k + j0 + u) * p.comb_d +
                                      col))
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const unsigned vmask = __ballot_sync(full, e >= 0 && e < p.E) & 0xFFu;
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const float wj = __shfl_sync(full, wv, u);
            if (vmask >> u & 1u) {
                a0 = fmaf(wj, v[u].x, a0);
                a1 = fmaf(wj, v[u].y, a1);
                a2 = fmaf(wj, v[u].z, a2);
                a3 = fmaf(wj, v[u].w, a3);
            }
        }
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a2, a3);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t *>(&lo);
    pk.y = *reinterpret_cast<const uint32_t *>(&hi);
    if (W4_IN_BOUNDS(t < p.M && col + 4 <= p.comb_d, p.dev_status))
        *reinterpret_cast<uint2 *>(p.comb_out + static_cast<int64_t>(t) * p.comb_d + col) = pk;
}

// (down, after the CTA's last unit and a fence that released its y stores)
// One arrival per valid slot of unit (J, pnl) on its token's counter of
// panel pnl (lane i for slot i); a warp that completed counters acquires
// the other CTAs' y stores with an acquire-release fence.  Completed
// (token, panel) pairs go to the CTA's list (or, past its capacity, are
// combined here).
__device__ __forceinline__ void combine_count(const GemmArgs &p, const Job &J, int pnl, int lane,
                                              int *list, int *count)
{
    const unsigned full = 0xffffffffu;
    for (int base = 0; base < J.n; base += 32) {   // the job's slots, 32 at a time
        int t = -1;
        bool last = false;
        if (base + lane < J.n) {
            const int a = __ldg(p.sorted_ids + J.start + base + lane);
            if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A)) {
                t = a / p.k;
                last = atomicAdd(p.comb_cnt + fold_counter_index(t, p.n_panels, pnl), 1) ==
                       p.k - 1;
            }
        }
        unsigned done = __ballot_sync(full, last);
        if (!done)
            continue;
        fence_acq_rel_gpu();
        int slot = 0;
        if (lane == 0)
            slot = atomicAdd(count, __popc(done));
        slot = __shfl_sync(full, slot, 0);
        while (done) {
            const int src = __ffs(done) - 1;
            done &= done - 1;
            const int tt = __shfl_sync(full, t, src);
            if (slot < kCombListCap) {
                if (lane == 0)
                    list[slot] = tt * p.n_panels + pnl;
            } else {
                combine_panel(p, tt, pnl, lane);
            }
            slot++;
        }
    }
}

// RESIDENT: each job's activations are loaded once into one of two 48 KB
// slots (contraction dim <= 768); otherwise they stream through 32 KB slots.
template <bool GATE_UP, bool RESIDENT, bool BIGN>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs p)
{
    constexpr int kJobN = JobShape<BIGN>::kMaxN;         // slots per job
    constexpr int kIss = JobShape<BIGN>::kIssuers;       // issuers with MMAs, chains
    static_assert(!(BIGN && RESIDENT), "big jobs stream their activations");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemLayout L = smem_layout(p.G, p.E, GATE_UP);
    uint8_t *stage_w = smem;
    uint8_t *stage_b = smem + L.off_b;
    uint8_t *sz_base = smem + L.off_sz;
    const Bars bar = carve_bars(smem + L.off_bar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    int *offs = reinterpret_cast<int *>(smem + L.off_offs);
    // 2^c per weight row for the last kRowScaleSets units (dequant -> epilogue)
    float *row_scale = reinterpret_cast<float *>(smem + L.off_rs);
    int *comb_list = reinterpret_cast<int *>(smem + L.off_cl);
    int *comb_count = reinterpret_cast<int *>(smem + L.off_misc) + 2;
    int *jp = reinterpret_cast<int *>(smem + L.off_jp);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned full = 0xffffffffu;
    int32_t *status = p.dev_status;
    const WaitCtx wc{abort_flag, status, p.wait_ns};
    const int n_sz = p.n_sz;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < kStagesW; i++) {
            mbar_init(&bar.w_full[i], 1);
            mbar_init(&bar.w_empty[i], kNumDqWarps);   // every dequant warp
        }
        for (int i = 0; i < kStagesB; i++) {
            mbar_init(&bar.b_full[i], 1);
            mbar_init(&bar.b_empty[i], kIss);   // every active issuer's commit
        }
        for (int i = 0; i < kRings * kRingBufs; i++) {
            mbar_init(&bar.a_full[i], 4);            // the ring's four lane quarters
            mbar_init(&bar.a_empty[i], 1);           // the ring's issuer's commit
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar.acc_full[i], kIss);
            mbar_init(&bar.acc_empty[i], kNumEpiWarps);
        }
        for (int i = 0; i < kMaxStagesSZ; i++) {
            mbar_init(&bar.sz_full[i], 1);
            mbar_init(&bar.sz_empty[i], kNumDqWarps);
        }
        for (int i = 0; i < kNumIssuers; i++)
            mbar_init(&bar.drain[i], 1);
        *abort_flag = 0;
        *comb_count = 0;
        fence_mbar_init();
    }
    if (warp == kWarpAlloc) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTmaW && lane == 0) {
        prefetch_tmap(&p.tmap_w);
        for (int i = 0; i < kJobN / 16; i++)
            prefetch_tmap(&p.tmap_b[i]);
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

    // jobs per expert (ceil(slots / kJobN)), exclusive prefix in jp[0..E]
    if (warp == kFirstEpiWarp) {
        int base = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            const int nj = e < p.E ? (offs[e + 1] - offs[e] + kJobN - 1) / kJobN : 0;
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
    const int n_blocks = p.n_blocks;     // 64-code blocks along K

    if (warp < kIss) {
        // ------------------------------------------------------ MMA issuers
        // Issuer r takes the fills of ring r in order: the unit's blocks j
        // with block_ring(j) == r, four K = 16 MMAs and the commit that frees
        // the buffer as one issue block each, then the correction when r is
        // the unit's correction ring, into its own accumulator.  Four issuers,
        // one per SM sub-partition.  (Big jobs: issuer r takes rings r and
        // r + 2, blocks with j % 2 == r, into its one chain.)  The warp runs
        // this loop converged (every value in it is warp-uniform, kept in
        // registers) and one elected lane issues each tcgen05 instruction.
        const int me = warp;
        const uint32_t b_base = smem_u32(stage_b);
        uint32_t b_seq = 0, n_unit = 0;
        // fills so far of ring me (low half) and, big jobs, ring me + 2 (high
        // half): buffer fill % kRingBufs
        uint32_t fills = 0;
        int cur_job = -1;       // resident mode: the job whose activations are held
        uint32_t res_slot = 0;
        bool ok = true;
        bool started = false;   // has this unit's first MMA gone (accumulate from then on)?
        // Block j (j == n_blocks: the correction): wait for the ring's next
        // buffer, issue its MMAs (four; n_corr_mma for the correction) with B
        // at the descriptor bdesc of the block's 64-code column block, and
        // release the buffer.
        auto issue = [&](int j, int ring, uint32_t d_tmem, uint64_t bdesc, uint32_t idesc) -> bool {
            const int n_mma = j == n_blocks ? p.n_corr_mma : 4;
            const int sh = ring == me ? 0 : 16;
            const uint32_t fill = (fills >> sh) & 0xFFFFu;
            const int buf = ring * kRingBufs + static_cast<int>(fill % kRingBufs);
            const uint32_t a_tmem = tmem + static_cast<uint32_t>(buf) * kFillCols;
            if (!warp_all_wait(&bar.a_full[buf], (fill / kRingBufs) & 1, wc))
                return false;
            fills = (fills & ~(0xFFFFu << sh)) | (((fill + 1) & 0xFFFFu) << sh);
            tc_fence_after();
            // K steps of 16: +32 B in the swizzled row (+2 in the descriptor's
            // address field), +8 columns of A
            tc_mma4_ts_commit_elect(d_tmem, a_tmem, bdesc, bdesc + 2, bdesc + 4, bdesc + 6, idesc,
                                    n_mma, started ? 1u : 0u, &bar.a_empty[buf]);
            started = true;
            return true;
        };
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, n_unit++) {
            const int job = u / p.n_panels;
            const Job J = decode_job(jp, offs, p.E, job, kJobN);
            const uint32_t idesc = idesc_f16_f32(kTileRows, J.n);
            const uint32_t col_bytes = static_cast<uint32_t>(J.n) * 128;
            const int set = n_unit & 1;
            const uint32_t acc_ph = (n_unit >> 1) & 1;
            const int corr = corr_ring(static_cast<int>(n_unit), n_blocks);
            if (!warp_all_wait(&bar.acc_empty[set], acc_ph ^ 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + kAccCol + set * (kIss * kJobN) + me * kJobN;
            started = false;
            if constexpr (RESIDENT) {
                // the job's activations stay in one slot for all its units
                if (job != cur_job) {
                    if (cur_job >= 0)
                        tc_commit_elect(&bar.b_empty[res_slot]);
                    res_slot = b_seq & 1;
                    if (!warp_all_wait(&bar.b_full[res_slot], (b_seq >> 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    b_seq++;
                    cur_job = job;
                }
                const uint32_t b_slot = b_base + res_slot * kResSlotBytes;
                for (int j = me; j < n_blocks && ok; j += kRings)
                    if (!issue(j, j & (kRings - 1), d_tmem,
                               sdesc_sw128(b_slot + static_cast<uint32_t>(j) * col_bytes), idesc))
                        ok = false;
                // the correction reads block n_blocks (the group sums)
                if (ok && me == corr &&
                    !issue(n_blocks, corr, d_tmem,
                           sdesc_sw128(b_slot + static_cast<uint32_t>(n_blocks) * col_bytes),
                           idesc))
                    ok = false;
            } else {
                const int kcols = b_kcols(J.n);
                // the last slot holds column block n_blocks, the group sums
                const int n_bslots = n_blocks / kcols + 1;
                for (int t = 0; t < n_bslots && ok; t++) {
                    const int sb = (b_seq + t) % kStagesB;
                    if (!warp_all_wait(&bar.b_full[sb], ((b_seq + t) / kStagesB) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_slot = b_base + sb * kStageBBytes;
                    const int j0 = t * kcols;
                    const int j1 = min(n_blocks, j0 + kcols);
                    for (int j = j0; j < j1 && ok; j++)
                        if (block_ring(j) % kIss == me &&
                            !issue(j, block_ring(j), d_tmem,
                                   sdesc_sw128(b_slot + static_cast<uint32_t>(j - j0) * col_bytes),
                                   idesc))
                            ok = false;
                    if (ok && t == n_bslots - 1 && corr % kIss == me) {
                        const uint32_t blk = static_cast<uint32_t>(n_blocks - t * kcols);
                        if (!issue(n_blocks, corr, d_tmem, sdesc_sw128(b_slot + blk * col_bytes),
                                   idesc))
                            ok = false;
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
        __syncwarp();
    } else if (warp < kNumIssuers) {
        // big jobs: issuers 2-3 idle
    } else if (warp == kWarpTmaW || warp == kWarpTmaW1) {
        // ------------------------------------------- TMA: codes, scales/zeros
        // Two producer threads, one per parity gp of the CTA's stage sequence:
        // stage g goes to slot g % kStagesW, so a parity owns every other
        // slot and each thread waits only on its own slots' releases.  The
        // parity-0 thread also issues each unit's scales and zeros before the
        // unit's stages.
        if (lane == 0) {
            const int gp = warp == kWarpTmaW ? 0 : 1;
            const uint64_t pol = l2_policy_evict_first();
            const uint32_t hb = 64u * p.G * 2;          // 64 rows of s (or z)
            uint32_t issued_a = 0, issue_ph_a = 0, issued_sz = 0, issue_ph_sz = 0;
            bool ok = true;
            int n_unit = 0;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, n_unit++) {
                const Job J = decode_job(jp, offs, p.E, u / p.n_panels, kJobN);
                const int pnl = u % p.n_panels;
                const int row0 = J.e * p.R + pnl * (GATE_UP ? 64 : 128);
                const int row1 = GATE_UP ? row0 + p.m_up : row0 + 64;
                if (gp == 0 && !(p.test_withhold_sz && n_unit == 0)) {
                    const int szb = n_unit % n_sz;
                    const uint32_t ph = (n_unit / n_sz) & 1;
                    if (!lane_wait(&bar.sz_empty[szb], ph ^ 1, wc))
                        break;
                    uint8_t *dst = sz_base + szb * L.sz_stride;
                    mbar_arrive_expect_tx(&bar.sz_full[szb], 4 * hb);
                    bulk_load_nohint(dst, p.sc + static_cast<int64_t>(row0) * p.G, hb,
                                     &bar.sz_full[szb]);
                    bulk_load_nohint(dst + hb, p.sc + static_cast<int64_t>(row1) * p.G, hb,
                                     &bar.sz_full[szb]);
                    bulk_load_nohint(dst + 2 * hb, p.zp + static_cast<int64_t>(row0) * p.G, hb,
                                     &bar.sz_full[szb]);
                    bulk_load_nohint(dst + 3 * hb, p.zp + static_cast<int64_t>(row1) * p.G, hb,
                                     &bar.sz_full[szb]);
                    issued_sz |= 1u << szb;
                    issue_ph_sz = (issue_ph_sz & ~(1u << szb)) | (ph << szb);
                }
                const int gs0 = n_unit * p.n_kchunks;
                for (int kc = (gs0 & 1) == gp ? 0 : 1; kc < p.n_kchunks; kc += 2) {
                    const int g = gs0 + kc;
                    const int sa = g % kStagesW;
                    const uint32_t ph = (g / kStagesW) & 1;
                    if (!lane_wait(&bar.w_empty[sa], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = stage_w + sa * kStageWBytes;
                    mbar_arrive_expect_tx(&bar.w_full[sa], kStageWBytes);
                    tma_load_2d(dst, &p.tmap_w, kc * 128, row0, &bar.w_full[sa], pol);
                    tma_load_2d(dst + kStageWBytes / 2, &p.tmap_w, kc * 128, row1,
                                &bar.w_full[sa], pol);
                    issued_a |= 1u << sa;
                    issue_ph_a = (issue_ph_a & ~(1u << sa)) | (ph << sa);
                }
            }
            if (*abort_flag) {   // let our own copies land before the CTA exits
                for (int i = 0; i < kStagesW; i++)
                    if (issued_a >> i & 1u)
                        drain_wait(&bar.w_full[i], issue_ph_a >> i & 1u);
                for (int i = 0; i < n_sz; i++)
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
            int sb = 0;
            uint32_t ph_b = 0, issued_b = 0, issue_ph_b = 0;
            bool ok = true;
            if constexpr (RESIDENT) {
                // one load per job into slot b_seq & 1, once the issuer has
                // released that slot's previous job
                int cur_job = -1;
                uint32_t b_seq = 0;
                for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                    const int job = u / p.n_panels;
                    if (job == cur_job)
                        continue;
                    cur_job = job;
                    const Job J = decode_job(jp, offs, p.E, job, kJobN);
                    const int s = b_seq & 1;
                    const uint32_t ph = (b_seq >> 1) & 1;
                    if (!lane_wait(&bar.b_empty[s], ph ^ 1, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar.b_full[s],
                                          static_cast<uint32_t>(J.n) * 128 * (K / 64 + 1));
                    tma_load_3d(stage_b + s * kResSlotBytes, &p.tmap_b[J.n / 16 - 1], 0, J.start,
                                0, &bar.b_full[s]);
                    issued_b |= 1u << s;
                    issue_ph_b = (issue_ph_b & ~(1u << s)) | (ph << s);
                    b_seq++;
                }
            } else {
                for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                    const Job J = decode_job(jp, offs, p.E, u / p.n_panels, kJobN);
                    const CUtensorMap *map = &p.tmap_b[J.n / 16 - 1];
                    const int kcols = b_kcols(J.n);
                    const uint32_t bytes = static_cast<uint32_t>(J.n) * 128 * kcols;
                    // column blocks 0 .. K / 64, the last one the group sums
                    for (int k_lo = 0; k_lo <= K; k_lo += 64 * kcols) {
                        if (!lane_wait(&bar.b_empty[sb], ph_b ^ 1, wc)) {
                            ok = false;
                            break;
                        }
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
        // Warp (q4, r): for every stage, expands slice r (codes 64 r ..
        // 64 r + 63, block 4 kc + r of the unit) for its 32 rows into ring
        // r's next A buffer.  A slice past K (a last stage of fewer than 256
        // codes) is skipped, but the stage is still waited for and released,
        // so the stage's arrival count is every dequant warp.
        const int q4 = warp & 3;
        const int r = (warp - kFirstDqWarp) >> 2;
        const int row = tile_row<GATE_UP>(q4, lane);
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        const int n_blocks = p.n_blocks;
        int szb = 0;
        uint32_t ph_sz = 0, n_unit = 0;
        const uint32_t sz_base_s = smem_u32(sz_base);
        // The running state, in registers: the next code stage slot `sa`
        // (its shared address, its barriers' addresses, its phase) and the
        // ring's next buffer `fb` (its TMEM column, its barriers, its phase).
        const uint32_t w_full0 = smem_u32(bar.w_full), w_empty0 = smem_u32(bar.w_empty);
        const uint32_t a_full0 = smem_u32(bar.a_full + r * kRingBufs);
        const uint32_t a_empty0 = smem_u32(bar.a_empty + r * kRingBufs);
        const uint32_t a_col_ring = tmem + lane_base + static_cast<uint32_t>(r * kRingBufs * kFillCols);
        int sa = 0;
        uint32_t ph_w = 0, fb = 0, ph_a = 0;
        // this warp's slice of a row: 16-byte chunks 2 r, 2 r + 1, swizzled
        const uint32_t sw = static_cast<uint32_t>(row & 7);
        const uint32_t code0 = smem_u32(stage_w) + static_cast<uint32_t>(row * 128) +
                               (((2u * r) ^ sw) << 4);
        const uint32_t code1 = smem_u32(stage_w) + static_cast<uint32_t>(row * 128) +
                               (((2u * r + 1) ^ sw) << 4);
        // the group index advances by 256 codes per stage
        const uint32_t g_step = 2u * (static_cast<uint32_t>(kChunkK) >> p.group_shift);
        // claim the ring's next buffer (the MMAs of two fills ago in it
        // complete); hand it over once written
        auto claim = [&]() -> bool {
            if (!warp_all_wait_a(a_empty0 + 8 * fb, ph_a ^ 1, wc))
                return false;
            tc_fence_after();
            return true;
        };
        auto hand_over = [&]() {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elect_a(a_full0 + 8 * fb);
            fb ^= 1;
            ph_a ^= fb ^ 1;    // the phase turns after buffer 1
        };
        // wait for the stage in slot sa; release it after the loads
        auto stage_wait = [&]() -> bool { return warp_all_wait_a(w_full0 + 8 * sa, ph_w, wc); };
        auto stage_release = [&]() {
            __syncwarp();
            mbar_arrive_elect_a(w_empty0 + 8 * sa);
            if (++sa == kStagesW) {
                sa = 0;
                ph_w ^= 1;
            }
        };
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, n_unit++) {
            if (!warp_all_wait(&bar.sz_full[szb], ph_sz, wc))
                break;
            const uint32_t s_addr = sz_base_s + szb * L.sz_stride + 2 * row * p.G;
            const uint32_t z_addr = s_addr + 2 * kTileRows * p.G;
            const int c = row_exponent(row_smax(s_addr, p.G));
            const float scale_s = exp2i(24 - c), scale_c = exp2i(-c);
            // stages 0 .. n_my - 1 hold a block of this ring (4 kc + r < n_blocks)
            const int n_my = (n_blocks - r + 3) >> 2;
            uint32_t g_off = 2u * ((static_cast<uint32_t>(r) * kSliceK) >> p.group_shift);
            for (int kc = 0; kc < n_my; kc++, g_off += g_step) {
                // the block's group constants before the codes arrive
                const GroupK k0 = group_consts(lds_u16(s_addr + g_off), lds_u16(z_addr + g_off),
                                               scale_s, scale_c);
                if (!stage_wait()) {
                    ok = false;
                    break;
                }
                const uint32_t so = static_cast<uint32_t>(sa * kStageWBytes);
                const uint4 v0 = lds128(code0 + so), v1 = lds128(code1 + so);
                stage_release();
                uint32_t o[16];
                dequant_word(v0.x, k0.S, k0.S16, k0.C, &o[0]);
                dequant_word(v0.y, k0.S, k0.S16, k0.C, &o[4]);
                dequant_word(v0.z, k0.S, k0.S16, k0.C, &o[8]);
                dequant_word(v0.w, k0.S, k0.S16, k0.C, &o[12]);
                if (!claim()) {
                    ok = false;
                    break;
                }
                if (kc == 0 && r == 0)   // block 0
                    row_scale[(n_unit & (kRowScaleSets - 1)) * kTileRows + row] = exp2i(c);
                const uint32_t a_col0 = a_col_ring + fb * kFillCols;
                // o is read by each store at issue and is free again after it
                tmem_st_32x32b_x16(a_col0, o);
                dequant_word(v1.x, k0.S, k0.S16, k0.C, &o[0]);
                dequant_word(v1.y, k0.S, k0.S16, k0.C, &o[4]);
                dequant_word(v1.z, k0.S, k0.S16, k0.C, &o[8]);
                dequant_word(v1.w, k0.S, k0.S16, k0.C, &o[12]);
                tmem_st_32x32b_x16(a_col0 + 16, o);
                hand_over();
            }
            // the unit's last stage when it holds no block of this ring
            for (int kc = n_my; kc < p.n_kchunks && ok; kc++) {
                if (!stage_wait()) {
                    ok = false;
                    break;
                }
                stage_release();
            }
            if (!ok)
                break;
            // the correction: a fill of ring corr_ring, after its last block
            if (r == corr_ring(static_cast<int>(n_unit), n_blocks)) {
                // The correction fill: C = -s z 2^-c rounded to fp16 (the
                // constant of every dequantised weight of the group) leaves
                // the part C_lo = fp16(C_exact - C).  The activations carry
                // one (xg) or four (h) sum columns per group, so contraction
                // index k of the correction belongs to group k or k / 4;
                // column i of MMA step t holds k = 16 t + 2 i, 16 t + 2 i + 1;
                // zero past the last group.
                // gate_up: word i of step t holds groups 16 t + 2 i, + 1;
                // down (four sum columns per group): both halves of words
                // 2 i' and 2 i' + 1 of step t hold group 4 t + i'
                constexpr int kRep = GATE_UP ? 1 : 4;
                if (!claim())
                    break;
                const uint32_t a_col0 = a_col_ring + fb * kFillCols;
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    if (t >= p.n_corr_mma)
                        break;
                    // the step's groups: all loads first (independent), then the math
                    constexpr int kNg = 16 / kRep;
                    uint32_t sb[kNg], zb[kNg];
#pragma unroll
                    for (int gi = 0; gi < kNg; gi++) {
                        const int g = kNg * t + gi;
                        sb[gi] = g < p.G ? lds_u16(s_addr + 2 * g) : 0u;
                        zb[gi] = g < p.G ? lds_u16(z_addr + 2 * g) : 0u;
                    }
                    uint32_t cw[8];
#pragma unroll
                    for (int gi = 0; gi < kNg; gi++) {
                        const float sv = __half2float(__ushort_as_half(static_cast<unsigned short>(sb[gi])));
                        const float zv = __half2float(__ushort_as_half(static_cast<unsigned short>(zb[gi])));
                        const float cx = -(sv * zv) * scale_c;          // exact
                        const float chi = __half2float(__float2half_rn(cx));
                        // cx - chi is exact; zero past the last group (s = z = 0)
                        const uint32_t lo = __half_as_ushort(__float2half_rn(cx - chi));
                        if constexpr (kRep == 1) {
                            if (gi & 1)
                                cw[gi >> 1] |= lo << 16;
                            else
                                cw[gi >> 1] = lo;
                        } else {
                            cw[2 * gi] = cw[2 * gi + 1] = lo | (lo << 16);
                        }
                    }
                    tmem_st_32x32b_x8(a_col0 + 8 * t, cw);
                }
                hand_over();
            }
            __syncwarp();
            mbar_arrive_elect(&bar.sz_empty[szb]);
            if (++szb == n_sz) {
                szb = 0;
                ph_sz ^= 1;
            }
        }
    } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + kNumEpiWarps) {
        // ---------------------------------------------------------- epilogue
        const int q4 = warp & 3;
        const int row = tile_row<GATE_UP>(q4, lane);
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        // gate_up: lanes 0-15 hold gate rows, lanes 16-31 the matching up rows;
        // the gate lane finishes even slots, the up lane odd ones
        const bool is_gate = lane < 16;
        const int il = 16 * q4 + (lane & 15);     // intermediate index in the panel
        uint32_t n_unit = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, n_unit++) {
            const Job J = decode_job(jp, offs, p.E, u / p.n_panels, kJobN);
            const int pnl = u % p.n_panels;
            const int set = n_unit & 1;
            const uint32_t acc_ph = (n_unit >> 1) & 1;
            // the assignment of every slot of the job, fetched early (gate_up:
            // padding slots get zero rows; down: rows go to y by assignment)
            const int my_a = lane < J.n ? __ldg(p.sorted_ids + J.start + lane) : -1;
            // big jobs: slots 32 .. 63
            const int my_a2 =
                BIGN && lane + 32 < J.n ? __ldg(p.sorted_ids + J.start + 32 + lane) : -1;
            if (!warp_all_wait(&bar.acc_full[set], acc_ph, wc))
                break;
            tc_fence_after();
            // 2^c of this lane's weight row, published by the dequant warps
            const float factor = row_scale[(n_unit & (kRowScaleSets - 1)) * kTileRows + row];
            const int mask = p.acc_mask[n_unit & 3];
            uint16_t *hout = reinterpret_cast<uint16_t *>(p.out);
            float *yout = reinterpret_cast<float *>(p.out);
            const int pos = pnl * 64 + (il & ~7) + korder_pos(il & 7);    // gate_up
            bool range = false;
            // passes of 16 slots (one for a 16-slot job)
#pragma unroll 1
            for (int half = 0; half < kJobN / 16; half++) {
                if (half * 16 >= J.n)
                    break;
                float v[16];
                {
                    // the accumulators that received MMAs, added in a fixed order
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        v[i] = 0.0f;
#pragma unroll
                    for (int c = 0; c < kIss; c++) {
                        if (!(mask >> c & 1))
                            continue;
                        uint32_t rr[16];
                        tmem_ld_32x32b_x16(tmem + lane_base + kAccCol + set * (kIss * kJobN) +
                                               c * kJobN + 16 * half,
                                           rr);
#pragma unroll
                        for (int i = 0; i < 16; i++)
                            v[i] += __uint_as_float(rr[i]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        v[i] *= factor;
                }
                if (half * 16 + 16 >= J.n) {   // the set's last read: hand it back
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_elect(&bar.acc_empty[set]);
                }
                if constexpr (GATE_UP) {
                    // h of this panel: 64 intermediates = group pnl of the down
                    // GEMM's contraction; this warp holds 16 of them and also
                    // writes their sum (of the fp16 values) to sum column
                    // 4 pnl + q4 of the row, the down GEMM's correction input
                    uint32_t pk[4];   // this lane's fp16 h of slot pairs 2 j, 2 j + 1
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const float send = is_gate ? v[i + 1] : v[i];
                        const float recv = __shfl_xor_sync(full, send, 16);
                        const float gv = is_gate ? v[i] : recv;
                        const float uv = is_gate ? recv : v[i + 1];
                        const int si = 16 * half + i + (is_gate ? 0 : 1);
                        const int a = __shfl_sync(full, half < 2 ? my_a : my_a2, si & 31);
                        const bool real = static_cast<unsigned>(a) < static_cast<unsigned>(p.A);
                        const float hv = gelu_tanh(gv) * uv;
                        range |= real && !(fabsf(hv) <= 65504.0f);
                        const uint16_t hq = real ? static_cast<uint16_t>(f16x2_sat(hv, 0.0f)) : 0;
                        uint16_t *hrow = hout + (J.start + si) * static_cast<int64_t>(p.h_stride);
                        if (W4_IN_BOUNDS(J.start + si < p.cap, status) &&
                            W4_IN_BOUNDS(pos < p.h_stride, status))
                            hrow[pos] = hq;
                        if (i & 2)
                            pk[i >> 2] |= static_cast<uint32_t>(hq) << 16;
                        else
                            pk[i >> 2] = hq;
                    }
                    // The eight slots' sums over the 16 lanes of each half of
                    // the warp (lanes 0-15 the even slots, 16-31 the odd
                    // ones): a butterfly that keeps half of the values at each
                    // step, pairing lanes by xor 8, 4, 2, 1 (the same fixed
                    // tree for every slot); lanes 2 m and 2 m + 1 of a half
                    // end with the sum of its pair m.
                    const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
                    float s4[4], s2[2];
#pragma unroll
                    for (int w2 = 0; w2 < 2; w2++) {
                        const __half2 kh = u2h(b3 ? pk[w2 + 2] : pk[w2]);
                        const __half2 rh = u2h(__shfl_xor_sync(full, b3 ? pk[w2] : pk[w2 + 2], 8));
                        s4[2 * w2] = __low2float(kh) + __low2float(rh);
                        s4[2 * w2 + 1] = __high2float(kh) + __high2float(rh);
                    }
#pragma unroll
                    for (int m = 0; m < 2; m++)
                        s2[m] = (b2 ? s4[m + 2] : s4[m]) +
                                __shfl_xor_sync(full, b2 ? s4[m] : s4[m + 2], 4);
                    float sum = (b1 ? s2[1] : s2[0]) + __shfl_xor_sync(full, b1 ? s2[0] : s2[1], 2);
                    sum += __shfl_xor_sync(full, sum, 1);
                    const int si = 16 * half + 2 * ((lane >> 1) & 7) + (is_gate ? 0 : 1);
                    if ((lane & 1) == 0 && si < J.n && W4_IN_BOUNDS(J.start + si < p.cap, status)) {
                        uint16_t *hrow = hout + (J.start + si) * static_cast<int64_t>(p.h_stride);
                        range |= !(fabsf(sum) <= 65504.0f);
                        if (W4_IN_BOUNDS(p.out_cols + 4 * pnl + q4 < p.h_stride, status))
                            hrow[p.out_cols + 4 * pnl + q4] = static_cast<uint16_t>(f16x2_sat(sum, 0.0f));
                        if (pnl == 0)   // sum columns past the last group, read by the
                                        // correction's last MMA step: zero
                            for (int c = 4 * p.h_groups + q4; c < 16 * ((p.h_groups + 3) / 4); c += 4)
                                if (W4_IN_BOUNDS(p.out_cols + c < p.h_stride, status))
                                    hrow[p.out_cols + c] = 0;
                    }
                } else {
                    const int col = pnl * 128 + row;
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int a = __shfl_sync(full, half < 2 ? my_a : my_a2, (16 * half + i) & 31);
                        if (static_cast<unsigned>(a) < static_cast<unsigned>(p.A) &&
                            W4_IN_BOUNDS(col < p.out_cols, status))
                            yout[static_cast<int64_t>(a) * p.out_cols + col] = v[i];
                    }
                }
            }
            if constexpr (GATE_UP) {
                if (__any_sync(full, range) && lane == 0 && status)
                    atomicOr(status, kDevFp16Range);
            }
        }
    } else if (warp == kWarpComb && p.comb_cnt) {
        // ------------------------------------ the folded combine's counters
        if constexpr (GATE_UP) {
            // set before the down launch that counts them
            for (int t = blockIdx.x; t < p.M; t += gridDim.x)
                fold_prepare_token(t, lane, p.topk_ids, p.k, p.E, p.comb_d, p.comb_cnt,
                                   p.comb_out);
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpAlloc) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (!GATE_UP) {
        if (p.comb_cnt && !*abort_flag) {
            if (p.early_schedule)
                pdl_wait();        // the counters are the preceding kernel's output
            // Every y store of this CTA is done (the barrier above); each
            // thread's fence then releases them to the CTA that completes a
            // counter.  One arrival per valid slot of each of the CTA's
            // units on its token's counter of the unit's panel (a warp per
            // unit, a lane per slot); completed (token, panel) pairs go to the
            // CTA's list (or are combined at once past its capacity).
            fence_acq_rel_gpu();
            for (int n = warp; n * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x) < n_units;
                 n += kNumWarps) {
                const int u = static_cast<int>(blockIdx.x) + n * static_cast<int>(gridDim.x);
                const Job J = decode_job(jp, offs, p.E, u / p.n_panels, kJobN);
                combine_count(p, J, u % p.n_panels, lane, comb_list, comb_count);
            }
            __syncthreads();
            // the CTA's completed combines, one (token, panel) per warp at a time
            const int n = min(*comb_count, kCombListCap);
            for (int i = warp; i < n; i += kNumWarps)
                combine_panel(p, comb_list[i] / p.n_panels, comb_list[i] % p.n_panels, lane);
        }
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
    bool attr_set[5] = {false, false, false, false, false};
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

bool grouped_gemm_fits(bool gate_up, int K, int group, int E)
{
    if (group <= 0 || K % group != 0)
        return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    const SmemLayout L = smem_layout(K / group, E, gate_up);
    return static_cast<size_t>(L.total) + 1024 <= static_cast<size_t>(device_info(dev).smem_optin);
}

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
    a.group_shift = q.group == 128 ? 7 : 6;
    a.G = q.K / q.group;
    a.n_panels = q.gate_up ? (q.R / 2) / 64 : q.R / 128;
    a.n_kchunks = (q.K + kChunkK - 1) / kChunkK;
    a.n_blocks = q.K / kSliceK;     // K is a multiple of the group, 64 or 128
    a.n_sz = sz_stages(a.G);
    // the activation rows end in one 64-column block of group sums: xg one
    // per group of 128, h one per quarter (16 intermediates) of each group of 64
    const int corr_rep = q.gate_up ? 1 : 4;
    if (a.G * corr_rep > 64) {
        *why = q.gate_up ? "gate_up contraction dim too large for its group sums (d <= 8192)"
                         : "down contraction dim too large for its group sums (m <= 1024)";
        return cudaErrorInvalidValue;
    }
    a.n_corr_mma = (a.G * corr_rep + 15) / 16;
    // Big jobs when the batch gives the experts 64 or more slots on average.
    const bool bign = static_cast<int64_t>(q.M) * q.k >= static_cast<int64_t>(kMaxNBig) * q.E;
    const int n_iss = bign ? JobShape<true>::kIssuers : JobShape<false>::kIssuers;
    // the accumulators (issuers) that receive MMAs in the CTA's unit n, by
    // n % 4
    for (int n = 0; n < 4; n++) {
        a.acc_mask[n] = 1 << (corr_ring(n, a.n_blocks) % n_iss);
        for (int j = 0; j < a.n_blocks; j++)
            a.acc_mask[n] |= 1 << (block_ring(j) % n_iss);
    }
    a.h_stride = q.gate_up ? q.R / 2 + 64 : 0;
    a.h_groups = q.gate_up ? (q.R / 2) / 64 : 0;
    a.early_schedule = q.early_schedule ? 1 : 0;
    a.topk_ids = q.topk_ids;
    a.topk_w = q.topk_w;
    a.comb_cnt = q.comb_cnt;
    a.comb_out = q.comb_out;
    a.M = q.M;
    a.k = q.k;
    a.comb_d = q.comb_d;
    a.cap = q.cap;
    a.wait_ns = q.wait_ns;
    a.test_withhold_sz = q.test_withhold_sz ? 1 : 0;
    const bool resident = !q.gate_up && !bign && b_fits_resident(q.K);

    const SmemLayout L = smem_layout(a.G, a.E, q.gate_up);
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
    for (int i = 0; i < (bign ? kMaxNBig : kMaxN) / 16; i++) {
        const int rows = 16 * (i + 1);
        const int kcols = resident ? q.K / 64 + 1 : b_kcols(rows);
        if (!encode_act(encode, &a.tmap_b[i], q.act, q.cap, q.K + 64, rows, kcols)) {
            *why = "cuTensorMapEncodeTiled rejected the activation tensor";
            return cudaErrorInvalidValue;
        }
    }

    auto kern = q.gate_up ? (bign ? grouped_gemm_kernel<true, false, true>
                                  : grouped_gemm_kernel<true, false, false>)
                : resident ? grouped_gemm_kernel<false, true, false>
                : bign     ? grouped_gemm_kernel<false, false, true>
                           : grouped_gemm_kernel<false, false, false>;
    const int which = q.gate_up ? (bign ? 4 : 2) : resident ? 1 : bign ? 3 : 0;
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
