// dense_gemm.cu -- the dense W4A16 GEMM: y[t, n] = sum_k x[t, k] deq(W)[n, k]
// ("dg-w4-kernels" -- W4A16: w4a16_linear reads packed nibbles and
// dequantises inline, equal to F.linear(x, dequant(W)); "Inference: Making
// every denoising pass fast" -- Dense W4 everywhere: QKV and LM-head tiles at
// 256 rows).
//
// Each 128-row panel of W is dequantised once per 64-code step into shared
// memory (fp16, the 128-byte-swizzled K-major layout the tensor cores read)
// and multiplied against up to 256 token rows at once: D[128 x 256] +=
// A[128 x 16] B[256 x 16]^T, tcgen05 kind::f16, fp32 accumulators in tensor
// memory.  The token rows come from the identity gather (fp16, the GEMMs'
// block order) by TMA.  Narrow outputs split the contraction dim so that the
// grid covers the GPU; the splits' fp32 partial sums are added in split order
// by a second launch.
//
// Warps: 0 TMA producer of packed codes (16 KB stages of 128-byte rows: four
// 64-code steps) and scales/zeros, 14 TMA producer of token tiles, 1 MMA
// issuer, 2-5 epilogue (tensor-memory lane quarter = warp & 3), 6-13
// dequantisation in four groups of two warps: group g expands step g of
// every code stage into its own A stage, so four steps are dequantised at
// once (thread = two rows of the step).  Every
// pipeline wait is bounded (~1 s), after which the kernel sets the timeout
// bit of dev_status, drains its own copies and MMAs, frees tensor memory and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "korder.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4 {

namespace {

constexpr int kDNumWarps = 15;
constexpr int kDThreads = 32 * kDNumWarps;
constexpr int kDWarpProd = 0;
constexpr int kDWarpProdB = 14;
constexpr int kDWarpMma = 1;
constexpr int kDFirstEpi = 2;
constexpr int kDNumEpi = 4;
constexpr int kDFirstDq = 6;
constexpr int kDNumDq = 8;
constexpr int kDRows = 128;       // weight rows per panel (MMA M)
constexpr int kDChunk = 64;       // codes per row per step: one 128-byte fp16 row of A
constexpr int kDMaxTok = 256;     // token rows per pass (MMA N)
constexpr int kDGroups = 4;        // dequantisation groups = A stages
constexpr int kDGroupWarps = kDNumDq / kDGroups;
constexpr int kDWChunk = 256;      // codes per row per code stage: one 128-byte row
constexpr int kDStagesA = kDGroups;
// each code stage holds one step per group, and every group waits on every
// code stage, so no barrier can run two phases ahead of a waiting warp
static_assert(kDWChunk / kDChunk == kDGroups, "stage counts");
constexpr int kDWBytes = kDRows * kDWChunk / 2;       // 16 KB of packed codes
constexpr int kDABytes = kDRows * kDChunk * 2;        // 16 KB of fp16
constexpr int kDMaxG = 32;                            // groups per weight row staged
constexpr int kDZOff = kDRows * kDMaxG * 2;           // z after s in a buffer
constexpr int kDSZBytes = 2 * kDZOff;                 // 16 KB per buffer
constexpr int kDSZBufs = 1;                           // scale/zero buffers (units in flight)
constexpr uint32_t kDTmemCols = 512;                  // two 256-column accumulators
constexpr int kDMaxSplits = 8;

// Shared-memory configurations, from the 1024-byte-aligned base: SW code
// stages (16 KB), SB token stages of BROWS rows (BROWS x 128 B), four A stages.
// Up to 256 token rows: 3 + 3 stages.  Up to 64 rows the token tiles are
// small and the room goes to code stages (7), which keeps more weight bytes
// in flight when the weights, not the tokens, set the pace.
template <int SW, int SB, int BROWS>
struct DCfg {
    static constexpr int kStagesW = SW, kStagesB = SB, kBRows = BROWS;
    static constexpr int kBBytes = BROWS * kDChunk * 2;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kDStagesA * kDABytes;
    static constexpr int kOffW = kOffB + kStagesB * kBBytes;
    static constexpr int kOffSZ = kOffW + kStagesW * kDWBytes;
    static constexpr int kOffBar = kOffSZ + kDSZBufs * kDSZBytes;
    static constexpr int kNumBars = 2 * SW + 2 * kDStagesA + 2 * SB + 2 + 2 + 2 * kDSZBufs + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr size_t kSmemLaunch = kOffMisc + 16 + 1024;
    static_assert(kSmemLaunch <= 227 * 1024, "shared memory budget");
    static_assert(kOffB % 1024 == 0 && kOffW % 1024 == 0 && kBBytes % 1024 == 0,
                  "swizzled tiles need 1024-byte alignment");
};
using DCfgLarge = DCfg<3, 3, kDMaxTok>;
using DCfgSmall = DCfg<7, 4, 64>;

struct DenseArgs {
    CUtensorMap tmap_w;   // q [N rows, K/2 bytes] u8, box {128 B, 128 rows}, 128-byte swizzle
    CUtensorMap tmap_b;   // xg [Mpad rows, K] fp16, box {64, box_rows}, 128-byte swizzle
    const uint16_t *sc;   // [N, G] fp16
    const uint16_t *zp;   // [N, G] fp16
    void *out;            // y [M, N] bf16, or fp32 partial sums [splits, M, N]
    int32_t *dev_status;
    int M, N, K, G, group_shift, box_rows;
    int n_panels, n_tiles, splits, chunks_per_split, n_kchunks, n_units;
};

struct DBars {
    uint64_t *w_full, *w_empty, *a_full, *a_empty, *b_full, *b_empty, *acc_full, *acc_empty,
        *sz_full, *sz_empty, *drain;
};

template <class C>
__device__ __forceinline__ DBars carve_dbars(uint8_t *base)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    DBars r;
    r.w_full = b;
    r.w_empty = r.w_full + C::kStagesW;
    r.a_full = r.w_empty + C::kStagesW;
    r.a_empty = r.a_full + kDStagesA;
    r.b_full = r.a_empty + kDStagesA;
    r.b_empty = r.b_full + C::kStagesB;
    r.acc_full = r.b_empty + C::kStagesB;
    r.acc_empty = r.acc_full + 2;
    r.sz_full = r.acc_empty + 2;
    r.sz_empty = r.sz_full + kDSZBufs;
    r.drain = r.sz_empty + kDSZBufs;
    return r;
}

struct DUnit {
    int panel, tile, split, kc0, kc1, t0, nt, ntp;
};

__device__ __forceinline__ DUnit decode_unit(const DenseArgs &p, int u)
{
    DUnit d;
    d.panel = u % p.n_panels;
    const int r = u / p.n_panels;
    d.tile = r % p.n_tiles;
    d.split = r / p.n_tiles;
    d.kc0 = d.split * p.chunks_per_split;
    d.kc1 = min(p.n_kchunks, d.kc0 + p.chunks_per_split);
    d.t0 = d.tile * kDMaxTok;
    d.nt = min(kDMaxTok, p.M - d.t0);
    d.ntp = (d.nt + 15) & ~15;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one elected lane of a
// converged warp.
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128_d(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

__device__ __forceinline__ float lds_f16(uint32_t saddr)
{
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(saddr));
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// (a & MASK) | magic in one LOP3
template <uint32_t MASK>
__device__ __forceinline__ uint32_t mask_or(uint32_t a, uint32_t magic)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "r"(magic));
    return r;
}

// 8 codes of one word -> 4 words of fp16 pairs q * s + c, in the block order
// (q0,q4) (q1,q5) (q2,q6) (q3,q7): the same arithmetic as the grouped GEMMs
// (q exact through the fp16 1024 + q trick, one fused rounding of q s + c).
__device__ __forceinline__ void dequant8(uint32_t w, __half2 s2, __half2 c2, uint32_t magic,
                                         uint32_t &o0, uint32_t &o1, uint32_t &o2, uint32_t &o3)
{
    const __half2 k1024 = as_h2(magic);
    const __half2 kSixteenth = as_h2(0x2C002C00u);
    const __half2 kMinus64 = as_h2(0xD400D400u);
    const uint32_t w8 = w >> 8;
    const __half2 q04 = __hsub2(as_h2(mask_or<0x000F000Fu>(w, magic)), k1024);
    const __half2 q15 = __hfma2(as_h2(mask_or<0x00F000F0u>(w, magic)), kSixteenth, kMinus64);
    const __half2 q26 = __hsub2(as_h2(mask_or<0x000F000Fu>(w8, magic)), k1024);
    const __half2 q37 = __hfma2(as_h2(mask_or<0x00F000F0u>(w8, magic)), kSixteenth, kMinus64);
    o0 = as_u32(__hfma2(q04, s2, c2));
    o1 = as_u32(__hfma2(q15, s2, c2));
    o2 = as_u32(__hfma2(q26, s2, c2));
    o3 = as_u32(__hfma2(q37, s2, c2));
}

__device__ __forceinline__ bool d_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            int32_t *status)
{
    return mbar_wait_warp(bar, parity, abort_flag, status, kDevPipelineTimeout);
}

__device__ __forceinline__ bool d_lane_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            int32_t *status)
{
    return mbar_wait(bar, parity, abort_flag, status, kDevPipelineTimeout);
}

// bounded wait that ignores the abort flag (draining only)
__device__ __forceinline__ void d_drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 200000000ull)
            return;
}

template <class C>
__global__ void __launch_bounds__(kDThreads, 1) dense_gemm_kernel(const __grid_constant__ DenseArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const DBars bar = carve_dbars<C>(smem + C::kOffBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *status = p.dev_status;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < C::kStagesW; i++) {
            mbar_init(&bar.w_full[i], 1);
            mbar_init(&bar.w_empty[i], kDNumDq);
        }
        for (int i = 0; i < kDStagesA; i++) {
            mbar_init(&bar.a_full[i], kDGroupWarps);
            mbar_init(&bar.a_empty[i], 1);
        }
        for (int i = 0; i < C::kStagesB; i++) {
            mbar_init(&bar.b_full[i], 1);
            mbar_init(&bar.b_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar.acc_full[i], 1);
            mbar_init(&bar.acc_empty[i], kDNumEpi);
        }
        for (int i = 0; i < kDSZBufs; i++) {
            mbar_init(&bar.sz_full[i], 1);
            mbar_init(&bar.sz_empty[i], kDNumDq);
        }
        mbar_init(&bar.drain[0], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, kDTmemCols);
        tmem_relinquish();
    }
    if (warp == kDWarpProd && lane == 0)
        prefetch_tmap(&p.tmap_w);
    if (warp == kDWarpProdB && lane == 0)
        prefetch_tmap(&p.tmap_b);
    // only this CTA's memory was touched so far; from here the inputs of the
    // preceding launch (the gathered rows) are read
    pdl_wait();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == kDWarpProd) {
        // ------------------------------------- TMA producer: codes, scales
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int sw = 0, szb = 0;
            uint32_t ph_w = 0, ph_sz = 0;
            // stages with a copy issued, and the parity that copy completes
            uint32_t w_iss = 0, w_par = 0, sz_iss = 0, sz_par = 0;
            const uint32_t szbytes = static_cast<uint32_t>(kDRows * p.G * 2);
            bool ok = true;
            for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
                const DUnit d = decode_unit(p, u);
                if (!d_lane_wait(&bar.sz_empty[szb], ph_sz ^ 1, abort_flag, status))
                    break;
                uint8_t *dst = smem + C::kOffSZ + szb * kDSZBytes;
                mbar_arrive_expect_tx(&bar.sz_full[szb], 2 * szbytes);
                bulk_load(dst, p.sc + static_cast<int64_t>(d.panel) * kDRows * p.G, szbytes,
                          &bar.sz_full[szb], pol);
                bulk_load(dst + kDZOff, p.zp + static_cast<int64_t>(d.panel) * kDRows * p.G,
                          szbytes, &bar.sz_full[szb], pol);
                sz_iss |= 1u << szb;
                sz_par = (sz_par & ~(1u << szb)) | (ph_sz << szb);
                if (++szb == kDSZBufs) {
                    szb = 0;
                    ph_sz ^= 1;
                }
                // code stage m holds steps kc0 + 4m .. kc0 + 4m + 3 (a last
                // partial stage reads past the split, or zeros past K: unused)
                for (int kc = d.kc0; kc < d.kc1; kc += kDGroups) {
                    if (!d_lane_wait(&bar.w_empty[sw], ph_w ^ 1, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar.w_full[sw], kDWBytes);
                    tma_load_2d(smem + C::kOffW + sw * kDWBytes, &p.tmap_w, kc * (kDChunk / 2),
                                d.panel * kDRows, &bar.w_full[sw], pol);
                    w_iss |= 1u << sw;
                    w_par = (w_par & ~(1u << sw)) | (ph_w << sw);
                    if (++sw == C::kStagesW) {
                        sw = 0;
                        ph_w ^= 1;
                    }
                }
            }
            // every copy issued here lands before the CTA may exit
            for (int i = 0; i < C::kStagesW; i++)
                if (w_iss >> i & 1u)
                    d_drain_wait(&bar.w_full[i], w_par >> i & 1u);
            for (int i = 0; i < kDSZBufs; i++)
                if (sz_iss >> i & 1u)
                    d_drain_wait(&bar.sz_full[i], sz_par >> i & 1u);
        }
        __syncwarp();
    } else if (warp == kDWarpProdB) {
        // ------------------------------------- TMA producer: token tiles
        if (lane == 0) {
            int sb = 0;
            uint32_t ph_b = 0, b_iss = 0, b_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
                const DUnit d = decode_unit(p, u);
                for (int kc = d.kc0; kc < d.kc1; kc++) {
                    if (!d_lane_wait(&bar.b_empty[sb], ph_b ^ 1, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar.b_full[sb], static_cast<uint32_t>(p.box_rows) * 128);
                    tma_load_2d_nohint(smem + C::kOffB + sb * C::kBBytes, &p.tmap_b, kc * kDChunk,
                                       d.t0, &bar.b_full[sb]);
                    b_iss |= 1u << sb;
                    b_par = (b_par & ~(1u << sb)) | (ph_b << sb);
                    if (++sb == C::kStagesB) {
                        sb = 0;
                        ph_b ^= 1;
                    }
                }
            }
            for (int i = 0; i < C::kStagesB; i++)
                if (b_iss >> i & 1u)
                    d_drain_wait(&bar.b_full[i], b_par >> i & 1u);
        }
        __syncwarp();
    } else if (warp == kDWarpMma) {
        // ------------------------------------------------------ MMA issuer
        // step kc of a unit comes from A stage (kc - kc0) % 4; apar holds the
        // parity of each A stage's next use
        int sb = 0;
        uint32_t ph_b = 0, n_unit = 0, apar = 0;
        const uint32_t a_s = smem_u32(smem + C::kOffA), b_s = smem_u32(smem + C::kOffB);
        bool ok = true;
        for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, n_unit++) {
            const DUnit d = decode_unit(p, u);
            const int set = n_unit & 1;
            if (!d_warp_wait(&bar.acc_empty[set], ((n_unit >> 1) & 1) ^ 1, abort_flag, status))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(set) * 256;
            const uint32_t idesc = idesc_f16_f32(kDRows, d.ntp);
            for (int kc = d.kc0; kc < d.kc1; kc++) {
                const int sa = (kc - d.kc0) % kDGroups;
                if (!d_warp_wait(&bar.a_full[sa], (apar >> sa) & 1u, abort_flag, status) ||
                    !d_warp_wait(&bar.b_full[sb], ph_b, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // K steps of 16: +32 B along the swizzled rows (+2 in the
                // descriptors' address field) of both operands
                const uint64_t ad = sdesc_sw128(a_s + sa * kDABytes);
                const uint64_t bd = sdesc_sw128(b_s + sb * C::kBBytes);
#pragma unroll
                for (int k = 0; k < kDChunk / 16; k++)
                    mma_ss_elect(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
                                 (kc != d.kc0 || k != 0) ? 1u : 0u);
                tc_commit_elect(&bar.a_empty[sa]);
                tc_commit_elect(&bar.b_empty[sb]);
                apar ^= 1u << sa;
                if (++sb == C::kStagesB) {
                    sb = 0;
                    ph_b ^= 1;
                }
            }
            if (!ok)
                break;
            tc_commit_elect(&bar.acc_full[set]);
        }
        // every MMA issued here completes before tensor memory is freed
        tc_commit_elect(&bar.drain[0]);
        d_drain_wait(&bar.drain[0], 0);
    } else if (warp < kDFirstEpi + kDNumEpi) {
        // -------------------------------------------------------- epilogue
        const int q4 = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        uint32_t n_unit = 0;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, n_unit++) {
            const DUnit d = decode_unit(p, u);
            const int set = n_unit & 1;
            if (!d_warp_wait(&bar.acc_full[set], (n_unit >> 1) & 1, abort_flag, status))
                break;
            tc_fence_after();
            const int n = d.panel * kDRows + 32 * q4 + lane;
            const uint32_t acc = tmem + lane_base + static_cast<uint32_t>(set) * 256;
            const int nblk = d.ntp / 16;
            for (int cb = 0; cb < nblk; cb++) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(acc + cb * 16, r);
                if (cb == nblk - 1) {     // the set goes back to the issuer
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_elect(&bar.acc_empty[set]);
                }
                const int tb = d.t0 + cb * 16;
                if (p.splits > 1) {
                    float *P = reinterpret_cast<float *>(p.out) +
                               static_cast<int64_t>(d.split) * p.M * p.N;
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        if (tb + i < p.M)
                            P[static_cast<int64_t>(tb + i) * p.N + n] = __uint_as_float(r[i]);
                } else {
                    uint16_t *Y = reinterpret_cast<uint16_t *>(p.out);
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        if (tb + i < p.M)
                            Y[static_cast<int64_t>(tb + i) * p.N + n] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i])));
                }
            }
        }
    } else {
        // --------------------------------------------------- dequantisation
        // group grp (two warps) expands step grp of every code stage into A
        // stage grp; thread gt of the group takes rows gt and gt + 64
        const int dqw = warp - kDFirstDq;
        const int grp = dqw / kDGroupWarps;
        const int gt = (dqw % kDGroupWarps) * 32 + lane;
        const int r0 = gt, r1 = gt + 64;
        const uint32_t w_base = smem_u32(smem + C::kOffW);
        const uint32_t a_stage = smem_u32(smem + C::kOffA) + grp * kDABytes;
        const uint32_t a_row0 = static_cast<uint32_t>((r0 >> 3) * 1024 + (r0 & 7) * 128);
        const uint32_t a_row1 = static_cast<uint32_t>((r1 >> 3) * 1024 + (r1 & 7) * 128);
        const uint32_t sw0 = static_cast<uint32_t>(r0 & 7), sw1 = static_cast<uint32_t>(r1 & 7);
        // the group's 32 bytes of a 128-byte code row: 16-byte pieces 2 grp
        // and 2 grp + 1, at positions piece ^ (row & 7) (128-byte swizzle)
        const uint32_t wq0a = r0 * 128 + (((2u * grp) ^ sw0) << 4);
        const uint32_t wq0b = r0 * 128 + (((2u * grp + 1) ^ sw0) << 4);
        const uint32_t wq1a = r1 * 128 + (((2u * grp) ^ sw1) << 4);
        const uint32_t wq1b = r1 * 128 + (((2u * grp + 1) ^ sw1) << 4);
        const uint32_t sz_base = smem_u32(smem + C::kOffSZ);
        uint32_t magic;   // fp16 1024.0 twice, kept in a register
        asm("mov.b32 %0, 0x64006400;" : "=r"(magic));
        int szb = 0, sw = 0;
        uint32_t ph_sz = 0, ph_w = 0, apar = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
            const DUnit d = decode_unit(p, u);
            if (!d_warp_wait(&bar.sz_full[szb], ph_sz, abort_flag, status))
                break;
            const uint32_t s_addr = sz_base + szb * kDSZBytes, z_addr = s_addr + kDZOff;
            for (int kc4 = d.kc0; kc4 < d.kc1; kc4 += kDGroups) {
                if (!d_warp_wait(&bar.w_full[sw], ph_w, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const int kc = kc4 + grp;
                const bool have = kc < d.kc1;     // warp-uniform
                uint4 q00, q01, q10, q11;
                float sf0 = 0.0f, zf0 = 0.0f, sf1 = 0.0f, zf1 = 0.0f;
                const uint32_t wst = w_base + sw * kDWBytes;
                if (have) {
                    q00 = lds128_d(wst + wq0a);
                    q01 = lds128_d(wst + wq0b);
                    q10 = lds128_d(wst + wq1a);
                    q11 = lds128_d(wst + wq1b);
                    const uint32_t g = static_cast<uint32_t>(kc * kDChunk) >> p.group_shift;
                    sf0 = lds_f16(s_addr + 2 * (r0 * p.G + g));
                    zf0 = lds_f16(z_addr + 2 * (r0 * p.G + g));
                    sf1 = lds_f16(s_addr + 2 * (r1 * p.G + g));
                    zf1 = lds_f16(z_addr + 2 * (r1 * p.G + g));
                }
                __syncwarp();
                mbar_arrive_elect(&bar.w_empty[sw]);
                if (++sw == C::kStagesW) {
                    sw = 0;
                    ph_w ^= 1;
                }
                if (!have)
                    continue;
                if (!d_warp_wait(&bar.a_empty[grp], ((apar & 1u) ^ 1u), abort_flag, status)) {
                    ok = false;
                    break;
                }
                apar ^= 1u;
                // a row's 16-byte piece j (block positions 8j .. 8j+7) sits at
                // piece position j ^ (row & 7) of its 128-byte line
                {
                    const __half2 s2 = __float2half2_rn(sf0);
                    const __half2 cz = __float2half2_rn(-zf0 * sf0);
                    const uint32_t w[8] = {q00.x, q00.y, q00.z, q00.w, q01.x, q01.y, q01.z, q01.w};
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        uint32_t o0, o1, o2, o3;
                        dequant8(w[j], s2, cz, magic, o0, o1, o2, o3);
                        sts128(a_stage + a_row0 + ((static_cast<uint32_t>(j) ^ sw0) << 4), o0, o1,
                               o2, o3);
                    }
                }
                {
                    const __half2 s2 = __float2half2_rn(sf1);
                    const __half2 cz = __float2half2_rn(-zf1 * sf1);
                    const uint32_t w[8] = {q10.x, q10.y, q10.z, q10.w, q11.x, q11.y, q11.z, q11.w};
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        uint32_t o0, o1, o2, o3;
                        dequant8(w[j], s2, cz, magic, o0, o1, o2, o3);
                        sts128(a_stage + a_row1 + ((static_cast<uint32_t>(j) ^ sw1) << 4), o0, o1,
                               o2, o3);
                    }
                }
                fence_proxy_async_smem();     // visible to the tensor cores' reads
                __syncwarp();
                mbar_arrive_elect(&bar.a_full[grp]);
            }
            if (!ok)
                break;
            __syncwarp();
            mbar_arrive_elect(&bar.sz_empty[szb]);
            if (++szb == kDSZBufs) {
                szb = 0;
                ph_sz ^= 1;
            }
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kDTmemCols);
    }
}

// y = bf16(sum over splits, in split order, of the fp32 partial sums)
__global__ void __launch_bounds__(256) splitk_sum_kernel(const float4 *__restrict__ part, int splits,
                                                         int64_t n4, uint2 *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
        float4 a = part[i];
        for (int s = 1; s < splits; s++) {
            const float4 b = part[static_cast<int64_t>(s) * n4 + i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        y[i] = pk;
    }
}

using EncodeFn = decltype(&cuTensorMapEncodeTiled);

EncodeFn encode_fn()
{
    static EncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    }
    return fn;
}

bool encode(EncodeFn fn, CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
            uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
            uint32_t box_outer, CUtensorMapSwizzle swizzle)
{
    const cuuint64_t gdim[2] = {inner, outer};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool dense_gemm_supported(int M, int N, int K, int group)
{
    return M >= 1 && N >= 128 && N % 128 == 0 && K % 64 == 0 && K >= kDWChunk &&
           (group == 64 || group == 128) && K % group == 0 && K / group <= kDMaxG;
}

// From the shape alone (so results do not depend on the GPU): enough splits
// of the contraction dim for about 128 units, at most 8, at least 4 steps each.
int dense_gemm_splits(int M, int N, int K)
{
    const int units = (N / kDRows) * ((M + kDMaxTok - 1) / kDMaxTok);
    const int kchunks = K / kDChunk;
    int s = std::max(1, std::min(kDMaxSplits, (128 + units - 1) / units));
    s = std::min(s, std::max(1, kchunks / 4));
    const int cps = (kchunks + s - 1) / s;
    return (kchunks + cps - 1) / cps;
}

size_t dense_gemm_partial_bytes(int M, int N, int K)
{
    const int s = dense_gemm_splits(M, N, K);
    return s > 1 ? static_cast<size_t>(s) * M * N * 4 : 0;
}

cudaError_t launch_dense_gemm(const DenseGemmProblem &q, cudaStream_t stream, const char **why)
{
    *why = nullptr;
    if (!dense_gemm_supported(q.M, q.N, q.K, q.group)) {
        *why = "shape outside the dense GEMM's limits";
        return cudaErrorInvalidValue;
    }
    DenseArgs a;
    a.sc = q.s;
    a.zp = q.z;
    a.dev_status = q.dev_status;
    a.M = q.M;
    a.N = q.N;
    a.K = q.K;
    a.G = q.K / q.group;
    a.group_shift = q.group == 128 ? 7 : 6;
    const int mpad = (q.M + 15) & ~15;
    a.box_rows = std::min(kDMaxTok, mpad);
    a.n_panels = q.N / kDRows;
    a.n_tiles = (q.M + kDMaxTok - 1) / kDMaxTok;
    a.n_kchunks = q.K / kDChunk;
    a.splits = dense_gemm_splits(q.M, q.N, q.K);
    a.chunks_per_split = (a.n_kchunks + a.splits - 1) / a.splits;
    a.n_units = a.n_panels * a.n_tiles * a.splits;
    a.out = a.splits > 1 ? static_cast<void *>(q.partials) : static_cast<void *>(q.y);
    if (a.splits > 1 && !q.partials) {
        *why = "split contraction needs the partial-sum buffer";
        return cudaErrorInvalidValue;
    }
    EncodeFn fn = encode_fn();
    if (!fn) {
        *why = "driver entry point cuTensorMapEncodeTiled not available";
        return cudaErrorNotSupported;
    }
    if (!encode(fn, &a.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, q.q, q.K / 2, q.N, q.K / 2,
                kDWChunk / 2, kDRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(fn, &a.tmap_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.xg, q.K, mpad,
                static_cast<uint64_t>(q.K) * 2, kDChunk, a.box_rows,
                CU_TENSOR_MAP_SWIZZLE_128B)) {
        *why = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static int sms[64] = {};
    static bool attr[64][2] = {};
    if (sms[dev & 63] == 0)
        cudaDeviceGetAttribute(&sms[dev & 63], cudaDevAttrMultiProcessorCount, dev);
    const bool small = a.box_rows <= DCfgSmall::kBRows;
    auto kern = small ? dense_gemm_kernel<DCfgSmall> : dense_gemm_kernel<DCfgLarge>;
    const size_t smem = small ? DCfgSmall::kSmemLaunch : DCfgLarge::kSmemLaunch;
    if (!attr[dev & 63][small]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem));
        if (err != cudaSuccess)
            return err;
        attr[dev & 63][small] = true;
    }
    const int grid = std::min(a.n_units, std::max(1, sms[dev & 63]));
    err = launch_pdl(kern, dim3(grid), dim3(kDThreads), smem, stream, a);
    if (err != cudaSuccess || a.splits == 1)
        return err;
    const int64_t n4 = static_cast<int64_t>(q.M) * q.N / 4;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256, 4096));
    return launch_pdl(splitk_sum_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      reinterpret_cast<const float4 *>(q.partials), a.splits, n4,
                      reinterpret_cast<uint2 *>(q.y));
}

}  // namespace w4
