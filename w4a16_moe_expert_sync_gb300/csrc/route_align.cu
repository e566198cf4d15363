// route_align.cu -- the router (softmax -> top-k -> renormalise) and the
// sync-free token-to-expert alignment.
//
// Router ("Inference: Making every denoising pass fast" -- Quantisation alone
// leaves a sparse execution problem): one warp per token.  The k largest
// logits are found by k rounds of a warp arg-max (ties to the lower expert
// index); softmax restricted to the selected logits is the full softmax
// renormalised over them, so the weights are exp(l_j - l_max) / sum_i
// exp(l_i - l_max), summed in slot order.
//
// Alignment ("dg-w4-kernels" -- Grouped MoE: sync-free and CUDA-graph safe;
// the grouped kernel "sorts assignments by expert, pads into regular
// blocks"): one CTA computes it with its warps; warp w owns a contiguous
// range of flat assignment indices (the expert ids staged in shared memory).
// Pass 1 builds one histogram per warp: the lanes that share an expert are
// found with one ballot per bit of the expert index and counted by their
// group's leader.  Pass 2 turns counts into padded expert offsets with a
// block scan and into per-warp start positions.  Pass 3 re-walks the range
// and places each assignment at its warp's running position plus its rank
// among earlier lanes with the same expert, which keeps the order stable.  No
// global atomics, no host round trip.  The fused launch runs this in every
// CTA, each writing a share of the outputs.
//
// Activation gather: the grouped gate_up GEMM reads its activations in slot
// order, xg[slot] = x[token of slot] converted to fp16 in the GEMMs'
// contraction order (korder.cuh), zero rows for padding slots.  The layer
// fuses alignment and gather into one launch.
#include <algorithm>
#include <cfloat>

#include "korder.cuh"
#include "checks.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4 {

// ------------------------------------------------------------------ router
// The router for one token, computed by one warp: the k largest logits by k
// rounds of a warp arg-max (ties to the lower expert index), then softmax
// over them.  Lane j < k returns the j-th choice in id/w; other lanes return
// id -1, w 0.  EPL = logits per lane (E <= 32 EPL).
template <int EPL>
__device__ __forceinline__ void route_token(const float *__restrict__ row, int E, int k, int lane,
                                            int *id, float *w)
{
    float v[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(row + e) : 0.0f;
        if (e >= E)
            taken |= 1u << i;
    }
    float my_val = 0.0f, top = 0.0f;
    int my_idx = -1;
    for (int j = 0; j < k; j++) {
        float bv = -FLT_MAX;
        int be = 0x7fffffff;
        bool have = false;
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            const int e = lane + 32 * i;
            if (!(taken >> i & 1u) && (!have || v[i] > bv)) {   // e increases with i
                bv = v[i];
                be = e;
                have = true;
            }
        }
        // warp arg-max: larger value wins, equal values go to the lower index
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const bool oh = __shfl_xor_sync(0xffffffffu, have ? 1 : 0, o) != 0;
            if (oh && (!have || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
                have = true;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (j == 0)
            top = bv;
        if (lane == j) {
            my_val = bv;
            my_idx = be;
        }
    }
    // The weights in float64, rounded to fp32 once: exp(l_j - l_top) over
    // the sum of the k selected, summed in slot order.  That is the
    // renormalised softmax of the k (the full softmax's normaliser cancels),
    // so the fp32 result is the float64 softmax's, bar a float64 rounding
    // difference that lands on an fp32 rounding boundary.
    const double ex = lane < k ? exp(static_cast<double>(my_val) - static_cast<double>(top)) : 0.0;
    double sum = 0.0;
    for (int j = 0; j < k; j++)
        sum += __shfl_sync(0xffffffffu, ex, j);
    *id = lane < k ? my_idx : -1;
    *w = lane < k ? static_cast<float>(ex / sum) : 0.0f;
}

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int M,
                                                    int E, int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ weights)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (t >= M)
        return;
    const int lane = threadIdx.x & 31;
    int id;
    float w;
    route_token<EPL>(logits + static_cast<int64_t>(t) * E, E, k, lane, &id, &w);
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = id;
        weights[static_cast<int64_t>(t) * k + lane] = w;
    }
}

cudaError_t launch_route(const float *logits, int M, int E, int k, int32_t *ids, float *w,
                         cudaStream_t stream)
{
    if (M == 0)
        return cudaSuccess;
    const int wpb = 8;
    const dim3 grid((M + wpb - 1) / wpb), block(32 * wpb);
    const int epl = (E + 31) / 32;
    cudaError_t err;
    if (epl <= 1)
        err = launch_pdl(route_kernel<1>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else if (epl <= 2)
        err = launch_pdl(route_kernel<2>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else if (epl <= 4)
        err = launch_pdl(route_kernel<4>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else if (epl <= 8)
        err = launch_pdl(route_kernel<8>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else if (epl <= 16)
        err = launch_pdl(route_kernel<16>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else if (epl <= 32)
        err = launch_pdl(route_kernel<32>, grid, block, 0, stream, logits, M, E, k, ids, w);
    else
        return cudaErrorInvalidValue;
    return err;
}

// --------------------------------------------------------------- alignment
constexpr int kAlignWarps = 32;     // the standalone alignment: one CTA of 1024 threads

__host__ __device__ size_t align_smem_bytes(int E, int nw)
{
    // per-warp histograms, expert totals, offsets, warp partial sums
    return sizeof(int) * (static_cast<size_t>(nw) * E + E + (E + 1) + 32);
}

// Assignments whose expert ids the alignment stages in shared memory (one
// coalesced load instead of one dependent load per pass and round).
constexpr int kAlignStagedIds = 16384;

// The lanes of the warp whose key equals this lane's, among the lanes with
// `valid` set (meaningful for valid lanes), from one ballot per key bit: a
// lane agrees with this one on bit b when the ballot of bit b has that lane
// set exactly when this lane's own bit b is set.  Costs nbits + 1 ballots
// whatever the number of distinct keys in the warp.
__device__ __forceinline__ unsigned match_key(int key, int nbits, bool valid)
{
    const unsigned full = 0xffffffffu;
    unsigned m = __ballot_sync(full, valid);
    for (int b = 0; b < nbits; b++) {
        const bool bit = (key >> b) & 1;
        const unsigned bal = __ballot_sync(full, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

// The alignment computed by one CTA of nw = blockDim.x / 32 warps, with
// blockDim.x >= E.  Every CTA of the grid computes the whole alignment in its
// own shared memory; the global outputs are split among the CTAs: a CTA
// writes sorted_ids for the assignments [own0, own1), the grid's threads
// split the padding slots and block owners one expert each, and CTA 0
// writes expert_offsets and num_padded and reports invalid ids.  With pos_sm
// the CTA also records the slot of each of its own assignments (or -1) at
// pos_sm[a - own0].  Returns through shared memory the padded offsets
// (offs_out[E+1]) and the per-expert counts (total_out[E]).
__device__ __forceinline__ void align_block(const int32_t *__restrict__ ids, int A, int E, int bm,
                                            int cap, int own0, int own1,
                                            int32_t *__restrict__ sorted_ids,
                                            int32_t *__restrict__ block_expert,
                                            int32_t *__restrict__ offsets,
                                            int32_t *__restrict__ num_padded,
                                            int32_t *__restrict__ dev_status, int *pos_sm,
                                            int *ids_sm, int **offs_out, int **total_out)
{
    extern __shared__ int sm[];
    const int nw = blockDim.x >> 5;
    int *hist = sm;                          // [nw][E]
    int *total = hist + nw * E;              // [E]
    int *offs = total + E;                   // [E+1]
    int *wsum = offs + E + 1;                // [32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int nbits = 32 - __clz(max(E - 1, 1));   // bits of an expert index

    // the ids, staged in shared memory when the caller gave room (ids_sm);
    // with ids == nullptr the caller has already put them there
    if (ids_sm && ids)
        for (int i = tid; i < A; i += blockDim.x)
            ids_sm[i] = __ldg(ids + i);
    auto id_at = [&](int a) { return ids_sm ? ids_sm[a] : __ldg(ids + a); };
    for (int i = tid; i < nw * E; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();

    const int chunk = (A + nw - 1) / nw;
    const int a0 = min(A, warp * chunk), a1 = min(A, a0 + chunk);
    // pass 1: per-warp histogram
    bool bad = false;
    for (int base = a0; base < a1; base += 32) {
        const int a = base + lane;
        const int e = a < a1 ? id_at(a) : -1;
        const bool valid = a < a1 && e >= 0 && e < E;
        bad |= (a < a1) && !valid;
        const unsigned grp = match_key(e, nbits, valid);
        if (valid && lane == __ffs(grp) - 1)
            hist[warp * E + e] += __popc(grp);
        __syncwarp();
    }
    if (blockIdx.x == 0 && __any_sync(full, bad) && lane == 0 && dev_status)
        atomicOr(dev_status, kDevBadExpertId);
    __syncthreads();

    // pass 2: totals, padded sizes, exclusive scan over experts
    int padded = 0, cnt = 0;
    if (tid < E) {
        for (int w = 0; w < nw; w++)
            cnt += hist[w * E + tid];
        padded = (cnt + bm - 1) / bm * bm;
        total[tid] = cnt;
    }
    int inc = padded;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, inc, o);
        if (lane >= o)
            inc += v;
    }
    if (lane == 31)
        wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int own = lane < nw ? wsum[lane] : 0;
        int s2 = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, s2, o);
            if (lane >= o)
                s2 += v;
        }
        if (lane < nw)
            wsum[lane] = s2 - own;             // exclusive prefix of warp sums
    }
    __syncthreads();
    if (tid < E) {
        const int excl = wsum[warp] + inc - padded;
        offs[tid] = excl;
        if (tid == E - 1)
            offs[E] = excl + padded;
        int run = excl;                        // per-warp start positions
        for (int w = 0; w < nw; w++) {
            const int c = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += c;
        }
    }
    __syncthreads();

    // pass 3: stable placement
    for (int base = a0; base < a1; base += 32) {
        const int a = base + lane;
        const int e = a < a1 ? id_at(a) : -1;
        const bool valid = a < a1 && e >= 0 && e < E;
        const unsigned grp = match_key(e, nbits, valid);
        int pos = 0;
        if (valid)
            pos = hist[warp * E + e] + __popc(grp & lt_mask);
        __syncwarp();
        if (valid && lane == __ffs(grp) - 1)
            hist[warp * E + e] += __popc(grp);
        __syncwarp();
        if (a < a1 && a >= own0 && a < own1) {   // lanes past a1 are another warp's
            if (sorted_ids && valid && W4_IN_BOUNDS(pos < cap, dev_status))
                sorted_ids[pos] = a;
            if (pos_sm)
                pos_sm[a - own0] = valid ? pos : -1;
        }
    }

    // pass 4: padding slots, block owners, offsets (split among the grid's
    // threads, one expert per thread)
    if (sorted_ids) {
        const int gtid = blockIdx.x * blockDim.x + tid, gstride = gridDim.x * blockDim.x;
        for (int e = gtid; e < E; e += gstride) {
            for (int sl = offs[e] + total[e]; sl < offs[e + 1]; sl++)
                if (W4_IN_BOUNDS(sl < cap, dev_status))
                    sorted_ids[sl] = A;
            for (int b = offs[e] / bm; b < offs[e + 1] / bm; b++)
                if (W4_IN_BOUNDS(b < cap / bm, dev_status))
                    block_expert[b] = e;
        }
        const int npad = offs[E];
        for (int sl = npad + gtid; sl < cap; sl += gstride)
            sorted_ids[sl] = A;
        for (int b = npad / bm + gtid; b < cap / bm; b += gstride)
            block_expert[b] = -1;
        if (blockIdx.x == 0) {
            for (int i = tid; i <= E; i += blockDim.x)
                offsets[i] = offs[i];
            if (tid == 0)
                num_padded[0] = npad;
        }
    }
    *offs_out = offs;
    *total_out = total;
}

__global__ void __launch_bounds__(kAlignWarps * 32, 1)
    moe_align_kernel(const int32_t *__restrict__ ids, int A, int E, int bm, int cap,
                     int32_t *__restrict__ sorted_ids, int32_t *__restrict__ block_expert,
                     int32_t *__restrict__ offsets, int32_t *__restrict__ num_padded,
                     int32_t *__restrict__ dev_status)
{
    extern __shared__ int sm[];
    int *ids_sm = A <= kAlignStagedIds ? sm + align_smem_bytes(E, kAlignWarps) / sizeof(int)
                                       : nullptr;
    int *offs, *total;
    align_block(ids, A, E, bm, cap, 0, A, sorted_ids, block_expert, offsets, num_padded,
                dev_status, nullptr, ids_sm, &offs, &total);
}

// bf16 bit patterns of magnitude >= 65536 (and inf, NaN) do not fit fp16's
// finite range: any of the eight in a 16-byte chunk?
__device__ __forceinline__ bool bf16x8_out_of_f16_range(uint4 v)
{
    auto big = [](uint32_t w) {
        return (w & 0x7FFFu) >= 0x4780u || ((w >> 16) & 0x7FFFu) >= 0x4780u;
    };
    return big(v.x) || big(v.y) || big(v.z) || big(v.w);
}

// The gathered rows (xg) are d fp16 values in block order followed by one
// 64-column block of group sums: column d + g holds the sum of the fp16
// values of group g (128 consecutive elements), columns from d/128 up to the
// next multiple of 16 hold zero.  The grouped GEMM multiplies them by the
// low parts of its dequantisation constants (grouped_gemm.cu).
constexpr int kXGroup = 128;
__host__ __device__ inline int64_t xg_stride(int d) { return static_cast<int64_t>(d) + 64; }

// Sum of the eight fp16 values of a converted chunk, reduced over the 16
// lanes that hold the 16 chunks of one group (lanes 16i .. 16i + 15 with
// consecutive chunk indices; all 16 call together), in a fixed order.
__device__ __forceinline__ float group_sum16(uint4 o)
{
    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        s += __low2float(h) + __high2float(h);
    }
    const unsigned mask = 0xFFFFu << (threadIdx.x & 16);
    s += __shfl_xor_sync(mask, s, 1);
    s += __shfl_xor_sync(mask, s, 2);
    s += __shfl_xor_sync(mask, s, 4);
    s += __shfl_xor_sync(mask, s, 8);
    return s;
}

// The sum-block column written by the thread of chunk c8 of a row: its
// group's sum (c8 % 16 == 0, column d + c8 / 16) or a zero column (c8 in
// [d/128, 16 ceil(d/2048))); -1 for neither.  *value gets the fp16 bits.
__device__ __forceinline__ int sum_column(int c8, int d, float gsum, uint16_t *value,
                                          bool *range)
{
    const int G = d / kXGroup;
    if ((c8 & 15) == 0) {
        *range |= !(fabsf(gsum) <= 65504.0f);
        *value = static_cast<uint16_t>(f16x2_sat(gsum, 0.0f));
        return d + c8 / 16;
    }
    if (c8 >= G && c8 < 16 * ((G + 15) / 16)) {
        *value = 0;
        return d + c8;
    }
    return -1;
}

// Standalone gather: xg[slot] = x[token of slot] (fp16, block order), zero
// for padding slots, for every slot below num_padded; activations outside
// fp16's finite range set W4_DEV_FP16_RANGE.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t *__restrict__ x, int d, int k,
                                                     int A, const int32_t *__restrict__ sorted_ids,
                                                     const int32_t *__restrict__ num_padded,
                                                     uint16_t *__restrict__ xg,
                                                     int32_t *__restrict__ dev_status)
{
    const int c8n = d / 8;
    const int64_t ld = xg_stride(d);
    const int64_t total = static_cast<int64_t>(__ldg(num_padded)) * c8n;
    bool range = false;
    // c8n is a multiple of 16: the 16 lanes of a group take the chunks of one
    // group of one row together
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t slot = i / c8n;
        const int c8 = static_cast<int>(i - slot * c8n);
        const int a = __ldg(sorted_ids + slot);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (static_cast<unsigned>(a) < static_cast<unsigned>(A)) {
            const uint4 raw = __ldg(
                reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(a / k) * d + 8 * c8));
            range |= bf16x8_out_of_f16_range(raw);
            o = bf16x8_to_f16_korder(raw);
        }
        uint16_t *row = xg + slot * ld;
        *reinterpret_cast<uint4 *>(row + 8 * c8) = o;
        const float gsum = group_sum16(o);
        uint16_t v;
        const int col = sum_column(c8, d, gsum, &v, &range);
        if (col >= 0)
            row[col] = v;
    }
    if (__any_sync(0xffffffffu, range) && (threadIdx.x & 31) == 0 && dev_status)
        atomicOr(dev_status, kDevFp16Range);
}

// The alignment of M tokens to a single expert with one slot each (the dense
// linear): slot i holds token i, slots [M, padded) are padding (sentinel M,
// zero rows); offsets = {0, padded}.  One thread per 16-byte chunk of xg.
__global__ void __launch_bounds__(256)
    identity_align_gather_kernel(const uint16_t *__restrict__ x, int M, int d, int padded,
                                 int32_t *__restrict__ sorted_ids, int32_t *__restrict__ offsets,
                                 uint16_t *__restrict__ xg)
{
    pdl_wait();
    pdl_trigger();
    const int c8n = d / 8;
    const int64_t total = static_cast<int64_t>(padded) * c8n;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = gtid; i < total; i += stride) {
        const int slot = static_cast<int>(i / c8n);
        const int c8 = static_cast<int>(i - static_cast<int64_t>(slot) * c8n);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (slot < M)
            o = bf16x8_to_f16_korder(
                __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(slot) * d) + c8));
        *reinterpret_cast<uint4 *>(xg + static_cast<int64_t>(slot) * d + 8 * c8) = o;
    }
    for (int64_t i = gtid; i < padded; i += stride)
        sorted_ids[i] = i < M ? static_cast<int32_t>(i) : M;
    if (gtid == 0) {
        offsets[0] = 0;
        offsets[1] = padded;
    }
}

cudaError_t launch_identity_align_gather(const uint16_t *x, int M, int d, int padded,
                                         int32_t *sorted_ids, int32_t *offsets, uint16_t *xg,
                                         cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(padded) * (d / 8);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 2048));
    return launch_pdl(identity_align_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256),
                      0, stream, x, M, d, padded, sorted_ids, offsets, xg);
}

// Fused alignment + gather (with ROUTE, router + alignment + gather from the
// logits: every CTA routes every token into shared memory first, with the
// same arithmetic as route_kernel, and writes ids and weights of its own
// tokens).  CTA b owns tokens [b*tpc, (b+1)*tpc), i.e. assignments
// [own0, own1).  It needs the alignment only for those: the padded offsets
// (from every expert's count) and, for each owned assignment, its rank among
// the assignments of its expert (the count of that expert's assignments
// before own0, plus its rank among the owned ones).  So every CTA counts all
// ids with shared-memory atomics, keeping apart those before own0, scans the
// padded counts, places its own assignments (one warp, in order) and copies
// its tokens' rows to their k slots.  The grid's threads write the padding
// slots and block owners one expert each.  The rows of padding slots in xg
// are not written: the GEMMs' outputs for those slots are discarded or
// zeroed.  The first kAheadTok x kAheadCols 16-byte chunks of a thread's rows
// are loaded before the counting so that their latency overlaps it.
constexpr int kAheadTok = 2, kAheadCols = 2;

__host__ __device__ inline int align_gather_threads(int E) { return E <= 512 ? 512 : (E + 31) / 32 * 32; }

constexpr int kRouteEpl = 4;    // the fused router: E <= 128

template <bool ROUTE>
__global__ void __launch_bounds__(1024, 1)
    moe_align_gather_kernel(const int32_t *__restrict__ ids, int M, int k, int E, int bm, int cap,
                            int32_t *__restrict__ sorted_ids, int32_t *__restrict__ block_expert,
                            int32_t *__restrict__ offsets, int32_t *__restrict__ num_padded,
                            int32_t *__restrict__ dev_status, const uint16_t *__restrict__ x,
                            int d, uint16_t *__restrict__ xg, int tpc,
                            const float *__restrict__ logits, int32_t *__restrict__ ids_out,
                            float *__restrict__ w_out)
{
    extern __shared__ int sm[];
    pdl_wait();
    pdl_trigger();
    const int A = M * k;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    int *cnt = sm;                  // [E] assignments per expert
    int *pre = cnt + E;             // [E] ... of them before own0
    int *offs = pre + E;            // [E+1] padded offsets
    int *pos = offs + E + 1;        // [tpc * k] slot of each owned assignment, -1 if skipped
    int *ids_sm = pos + tpc * k;    // [A] (ROUTE only)
    const int c8n = d / 8;
    const int t0 = min(M, static_cast<int>(blockIdx.x) * tpc), t1 = min(M, t0 + tpc);
    const int ntok = t1 - t0;
    const int own0 = t0 * k, own1 = t1 * k;
    // chunk c8 of this CTA's token tl is xr[tl * c8n + c8]
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t0) * d);
    uint4 ahead[kAheadTok][kAheadCols];   // raw bf16: converted after the alignment
#pragma unroll
    for (int tl = 0; tl < kAheadTok; tl++)
#pragma unroll
        for (int r = 0; r < kAheadCols; r++) {
            const int c8 = tid + r * nthr;
            ahead[tl][r] = tl < ntok && c8 < c8n ? __ldg(xr + tl * c8n + c8) : make_uint4(0, 0, 0, 0);
        }
    // this thread's first kIdsAhead ids, loaded before the first barrier so
    // that their latency overlaps it
    constexpr int kIdsAhead = 4;
    int ids_ahead[kIdsAhead];
    if constexpr (!ROUTE) {
#pragma unroll
        for (int i = 0; i < kIdsAhead; i++) {
            const int a = tid + i * nthr;
            ids_ahead[i] = a < A ? __ldg(ids + a) : -1;
        }
    }
    for (int i = tid; i < E; i += nthr) {
        cnt[i] = 0;
        pre[i] = 0;
    }
    if constexpr (ROUTE) {
        // every token's top-k into shared memory, this CTA's tokens also to
        // ids_out / w_out
        const int nw = nthr >> 5;
        for (int t = warp; t < M; t += nw) {
            int id;
            float w;
            route_token<kRouteEpl>(logits + static_cast<int64_t>(t) * E, E, k, lane, &id, &w);
            if (lane < k) {
                ids_sm[t * k + lane] = id;
                if (t >= t0 && t < t1) {
                    ids_out[static_cast<int64_t>(t) * k + lane] = id;
                    w_out[static_cast<int64_t>(t) * k + lane] = w;
                }
            }
        }
    }
    __syncthreads();
    auto id_at = [&](int a) { return ROUTE ? ids_sm[a] : __ldg(ids + a); };

    // counts: every valid id, and separately those before own0
    bool bad = false;
    auto count = [&](int a, int e) {
        if (e >= 0 && e < E) {
            atomicAdd(&cnt[e], 1);
            if (a < own0)
                atomicAdd(&pre[e], 1);
        } else {
            bad = true;
        }
    };
    int a_next = tid;
    if constexpr (!ROUTE) {
#pragma unroll
        for (int i = 0; i < kIdsAhead; i++, a_next += nthr)
            if (a_next < A)
                count(a_next, ids_ahead[i]);
    }
    for (int a = a_next; a < A; a += nthr)
        count(a, id_at(a));
    if (blockIdx.x == 0 && __any_sync(full, bad) && lane == 0 && dev_status)
        atomicOr(dev_status, kDevBadExpertId);
    __syncthreads();

    // padded offsets: exclusive scan of ceil(count / bm) * bm (warp 0; lane
    // l takes the run of experts [l * per, (l + 1) * per): a sum of its run,
    // one warp scan of the sums, then the run's offsets)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e_lo = min(E, lane * per), e_hi = min(E, e_lo + per);
        int run = 0;
        for (int e = e_lo; e < e_hi; e++)
            run += (cnt[e] + bm - 1) / bm * bm;
        int inc = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, inc, o);
            if (lane >= o)
                inc += v;
        }
        int base = inc - run;
        for (int e = e_lo; e < e_hi; e++) {
            offs[e] = base;
            base += (cnt[e] + bm - 1) / bm * bm;
        }
        if (lane == 31)
            offs[E] = inc;
    }
    __syncthreads();

    // stable placement of the owned assignments, in order (warp 0): rank =
    // the expert's assignments before own0 + those before it in [own0, a)
    if (warp == 0) {
        const int nbits = 32 - __clz(max(E - 1, 1));
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = own0; base < own1; base += 32) {
            const int a = base + lane;
            const int e = a < own1 ? id_at(a) : -1;
            const bool valid = a < own1 && e >= 0 && e < E;
            const unsigned grp = match_key(e, nbits, valid);
            const int slot = valid ? offs[e] + pre[e] + __popc(grp & lt_mask) : -1;
            __syncwarp();
            if (valid && lane == __ffs(grp) - 1)
                pre[e] += __popc(grp);
            __syncwarp();
            if (a < own1) {
                pos[a - own0] = slot;
                if (valid && W4_IN_BOUNDS(slot < cap, dev_status))
                    sorted_ids[slot] = a;
            }
        }
    }
    __syncthreads();

    // this CTA's rows to the slots of their assignments, in fp16 block order
    bool range = false;
    const int64_t ld = xg_stride(d);
    // (the 16 lanes of a group always call this together: c8n is a multiple
    // of 16 and each loop below gives a lane's group one chunk range)
    auto put = [&](int tl, int c8, uint4 raw) {
        range |= bf16x8_out_of_f16_range(raw);
        const uint4 o = bf16x8_to_f16_korder(raw);
        const float gsum = group_sum16(o);
        uint16_t v;
        const int col = sum_column(c8, d, gsum, &v, &range);
        for (int j = 0; j < k; j++) {
            const int slot = pos[tl * k + j];
            if (slot >= 0 && W4_IN_BOUNDS(slot < cap, dev_status)) {
                uint16_t *row = xg + static_cast<int64_t>(slot) * ld;
                *reinterpret_cast<uint4 *>(row + 8 * c8) = o;
                if (col >= 0)
                    row[col] = v;
            }
        }
    };
#pragma unroll
    for (int tl = 0; tl < kAheadTok; tl++)
#pragma unroll
        for (int r = 0; r < kAheadCols; r++) {
            const int c8 = tid + r * nthr;
            if (tl < ntok && c8 < c8n)
                put(tl, c8, ahead[tl][r]);
        }
    for (int tl = 0; tl < ntok; tl++)
        for (int c8 = tid + (tl < kAheadTok ? kAheadCols * nthr : 0); c8 < c8n; c8 += nthr)
            put(tl, c8, __ldg(xr + tl * c8n + c8));
    if (__any_sync(full, range) && lane == 0 && dev_status)
        atomicOr(dev_status, kDevFp16Range);

    // padding slots and block owners, one expert per warp of the grid (its
    // lanes over the expert's slots and blocks); the slots past the last
    // expert; offsets and num_padded from CTA 0
    const int gtid = blockIdx.x * nthr + tid, gstride = gridDim.x * nthr;
    const int nwarps = nthr >> 5;
    for (int e = blockIdx.x + gridDim.x * warp; e < E; e += gridDim.x * nwarps) {
        for (int sl = offs[e] + cnt[e] + lane; sl < offs[e + 1]; sl += 32)
            if (W4_IN_BOUNDS(sl < cap, dev_status))
                sorted_ids[sl] = A;
        for (int b = offs[e] / bm + lane; b < offs[e + 1] / bm; b += 32)
            if (W4_IN_BOUNDS(b < cap / bm, dev_status))
                block_expert[b] = e;
    }
    const int npad = offs[E];
    for (int sl = npad + gtid; sl < cap; sl += gstride)
        sorted_ids[sl] = A;
    for (int b = npad / bm + gtid; b < cap / bm; b += gstride)
        block_expert[b] = -1;
    if (blockIdx.x == 0) {
        for (int i = tid; i <= E; i += nthr)
            offsets[i] = offs[i];
        if (tid == 0)
            num_padded[0] = npad;
    }
}

static cudaError_t set_align_smem(const void *fn)
{
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

cudaError_t launch_align(const int32_t *ids, int M, int k, int E, int block_m, int64_t cap,
                         int32_t *sorted_ids, int32_t *block_expert, int32_t *offsets,
                         int32_t *num_padded, int32_t *dev_status, cudaStream_t stream)
{
    const int A = M * k;
    const size_t smem = align_smem_bytes(E, kAlignWarps) +
                        (A <= kAlignStagedIds ? sizeof(int) * static_cast<size_t>(A) : 0);
    cudaError_t err = set_align_smem(reinterpret_cast<const void *>(moe_align_kernel));
    if (err != cudaSuccess)
        return err;
    moe_align_kernel<<<1, kAlignWarps * 32, smem, stream>>>(
        ids, M * k, E, block_m, static_cast<int>(cap), sorted_ids, block_expert, offsets,
        num_padded, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t *x, int M, int d, int k, int64_t cap,
                          const int32_t *sorted_ids, const int32_t *num_padded, uint16_t *xg,
                          int32_t *dev_status, cudaStream_t stream)
{
    const int64_t total = cap * (d / 8);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 4096));
    gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, d, k, M * k, sorted_ids,
                                                                      num_padded, xg, dev_status);
    return cudaGetLastError();
}

// one CTA per SM whatever the batch (the padding rows are spread over all of
// them), the tokens of a CTA contiguous
static void align_gather_grid(int M, int num_sms, int *grid, int *tpc)
{
    *grid = std::max(1, num_sms);
    *tpc = std::max(1, (M + *grid - 1) / *grid);
}

size_t align_gather_smem_bytes(int M, int k, int E, int num_sms)
{
    int grid, tpc;
    align_gather_grid(M, num_sms, &grid, &tpc);
    // counts, counts before own0, offsets, owned slots (+ every id with the router)
    return sizeof(int) * (3 * static_cast<size_t>(E) + 1 + static_cast<size_t>(tpc) * k);
}

static size_t route_align_gather_smem_bytes(int M, int k, int E, int num_sms)
{
    return align_gather_smem_bytes(M, k, E, num_sms) + sizeof(int) * static_cast<size_t>(M) * k;
}

cudaError_t launch_align_gather(const int32_t *ids, int M, int k, int E, int block_m, int64_t cap,
                                int32_t *sorted_ids, int32_t *block_expert, int32_t *offsets,
                                int32_t *num_padded, int32_t *dev_status, const uint16_t *x,
                                int d, uint16_t *xg, int num_sms, cudaStream_t stream)
{
    const size_t smem = align_gather_smem_bytes(M, k, E, num_sms);
    cudaError_t err = set_align_smem(reinterpret_cast<const void *>(moe_align_gather_kernel<false>));
    if (err != cudaSuccess)
        return err;
    int grid, tpc;
    align_gather_grid(M, num_sms, &grid, &tpc);
    return launch_pdl(moe_align_gather_kernel<false>, dim3(grid), dim3(align_gather_threads(E)),
                      smem, stream, ids, M, k, E, block_m, static_cast<int>(cap), sorted_ids,
                      block_expert, offsets, num_padded, dev_status, x, d, xg, tpc,
                      static_cast<const float *>(nullptr), static_cast<int32_t *>(nullptr),
                      static_cast<float *>(nullptr));
}

bool route_align_gather_fits(int M, int k, int E, int num_sms)
{
    // Every CTA routes every token, a warp per token, each a chain of k
    // dependent warp reductions.  A separate router launch overlaps the
    // alignment launch's start (programmatic dependent launch) and costs ~3 us
    // more, which routing in the CTA exceeds beyond one token per warp
    // (measured: 22.5 us against 17.4 us at 32 tokens, 26.8 against 15.3 at 64).
    return E <= 32 * kRouteEpl && M <= align_gather_threads(E) / 32 &&
           static_cast<int64_t>(M) * k <= kAlignStagedIds &&
           route_align_gather_smem_bytes(M, k, E, num_sms) <= 200 * 1024;
}

cudaError_t launch_route_align_gather(const float *logits, int M, int k, int E, int block_m,
                                      int64_t cap, int32_t *ids, float *w, int32_t *sorted_ids,
                                      int32_t *block_expert, int32_t *offsets,
                                      int32_t *num_padded, int32_t *dev_status,
                                      const uint16_t *x, int d, uint16_t *xg, int num_sms,
                                      cudaStream_t stream)
{
    if (!route_align_gather_fits(M, k, E, num_sms))
        return cudaErrorInvalidValue;
    const size_t smem = route_align_gather_smem_bytes(M, k, E, num_sms);
    cudaError_t err = set_align_smem(reinterpret_cast<const void *>(moe_align_gather_kernel<true>));
    if (err != cudaSuccess)
        return err;
    int grid, tpc;
    align_gather_grid(M, num_sms, &grid, &tpc);
    return launch_pdl(moe_align_gather_kernel<true>, dim3(grid), dim3(align_gather_threads(E)),
                      smem, stream, static_cast<const int32_t *>(nullptr), M, k, E, block_m,
                      static_cast<int>(cap), sorted_ids, block_expert, offsets, num_padded,
                      dev_status, x, d, xg, tpc, logits, ids, w);
}

}  // namespace w4
