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
// blocks"): a single CTA of 32 warps.  Warp w owns a contiguous range of flat
// assignment indices.  Pass 1 builds one histogram per warp with
// __match_any_sync (lanes that share an expert are counted by their group's
// leader).  Pass 2 turns counts into padded expert offsets with a block scan
// and into per-warp start positions.  Pass 3 re-walks the range and places
// each assignment at its warp's running position plus its rank among earlier
// lanes with the same expert, which keeps the order stable.  No global
// atomics, no host round trip.
//
// Activation gather: the grouped gate_up GEMM reads its activations in slot
// order, xg[slot] = x[token of slot] converted to fp16 in the GEMMs'
// contraction order (korder.cuh), zero rows for padding slots.  The layer
// fuses alignment and gather into one launch.
#include <algorithm>
#include <cfloat>

#include "korder.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4 {

// ------------------------------------------------------------------ router
template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int M,
                                                    int E, int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ weights)
{
    const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (t >= M)
        return;
    const int lane = threadIdx.x & 31;
    const float *row = logits + static_cast<int64_t>(t) * E;
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
    int my_idx = 0;
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
    const float ex = lane < k ? expf(my_val - top) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < k; j++)
        sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = my_idx;
        weights[static_cast<int64_t>(t) * k + lane] = ex / sum;
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
    if (epl <= 1)
        route_kernel<1><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else if (epl <= 2)
        route_kernel<2><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else if (epl <= 4)
        route_kernel<4><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else if (epl <= 8)
        route_kernel<8><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else if (epl <= 16)
        route_kernel<16><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else if (epl <= 32)
        route_kernel<32><<<grid, block, 0, stream>>>(logits, M, E, k, ids, w);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// --------------------------------------------------------------- alignment
constexpr int kAlignWarps = 32;

__host__ __device__ size_t align_smem_bytes(int E)
{
    // per-warp histograms, expert totals, offsets, warp partial sums
    return sizeof(int) * (static_cast<size_t>(kAlignWarps) * E + E + (E + 1) + kAlignWarps);
}

// The alignment computed by one CTA of 1024 threads.  With write_global the
// CTA writes sorted_ids / block_expert / expert_offsets / num_padded and
// reports invalid ids; with pos_sm it records the slot of every flat
// assignment (or -1) in shared memory.  Returns through shared memory: the
// padded offsets (offs_out[E+1]) and per-expert counts (total_out[E]).
__device__ __forceinline__ void align_block(const int32_t *__restrict__ ids, int A, int E, int bm,
                                            int cap, bool write_global,
                                            int32_t *__restrict__ sorted_ids,
                                            int32_t *__restrict__ block_expert,
                                            int32_t *__restrict__ offsets,
                                            int32_t *__restrict__ num_padded,
                                            int32_t *__restrict__ dev_status, int *pos_sm,
                                            int **offs_out, int **total_out)
{
    extern __shared__ int sm[];
    int *hist = sm;                          // [32][E]
    int *total = hist + kAlignWarps * E;     // [E]
    int *offs = total + E;                   // [E+1]
    int *wsum = offs + E + 1;                // [32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int i = tid; i < kAlignWarps * E; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();

    const int chunk = (A + kAlignWarps - 1) / kAlignWarps;
    const int a0 = min(A, warp * chunk), a1 = min(A, a0 + chunk);
    // pass 1: per-warp histogram
    bool bad = false;
    {
        for (int base = a0; base < a1; base += 32) {
            const int a = base + lane;
            const int e = a < a1 ? __ldg(ids + a) : -1;
            const bool valid = a < a1 && e >= 0 && e < E;
            bad |= (a < a1) && !valid;
            const int key = valid ? e : E + lane;      // invalid lanes match nobody
            const unsigned grp = __match_any_sync(full, key);
            if (valid && lane == __ffs(grp) - 1)
                hist[warp * E + e] += __popc(grp);
            __syncwarp();
        }
    }
    if (write_global && __any_sync(full, bad) && lane == 0 && dev_status)
        atomicOr(dev_status, kDevBadExpertId);
    __syncthreads();

    // pass 2: totals, padded sizes, exclusive scan over experts
    int padded = 0, cnt = 0;
    if (tid < E) {
        for (int w = 0; w < kAlignWarps; w++)
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
        int s2 = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, s2, o);
            if (lane >= o)
                s2 += v;
        }
        wsum[lane] = s2 - wsum[lane];          // exclusive prefix of warp sums
    }
    __syncthreads();
    if (tid < E) {
        const int excl = wsum[warp] + inc - padded;
        offs[tid] = excl;
        if (tid == E - 1)
            offs[E] = excl + padded;
        int run = excl;                        // per-warp start positions
        for (int w = 0; w < kAlignWarps; w++) {
            const int c = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += c;
        }
    }
    __syncthreads();

    // pass 3: stable placement
    {
        for (int base = a0; base < a1; base += 32) {
            const int a = base + lane;
            const int e = a < a1 ? __ldg(ids + a) : -1;
            const bool valid = a < a1 && e >= 0 && e < E;
            const int key = valid ? e : E + lane;
            const unsigned grp = __match_any_sync(full, key);
            int pos = 0;
            if (valid)
                pos = hist[warp * E + e] + __popc(grp & lt_mask);
            __syncwarp();
            if (valid && lane == __ffs(grp) - 1)
                hist[warp * E + e] += __popc(grp);
            __syncwarp();
            if (a < a1) {
                if (write_global && valid)
                    sorted_ids[pos] = a;
                if (pos_sm)
                    pos_sm[a] = valid ? pos : -1;
            }
        }
    }

    // pass 4: padding, block owners, offsets
    if (write_global) {
        if (tid < E) {
            for (int sl = offs[tid] + total[tid]; sl < offs[tid + 1]; sl++)
                sorted_ids[sl] = A;
            for (int b = offs[tid] / bm; b < offs[tid + 1] / bm; b++)
                block_expert[b] = tid;
        }
        const int npad = offs[E];
        for (int sl = npad + tid; sl < cap; sl += blockDim.x)
            sorted_ids[sl] = A;
        for (int b = npad / bm + tid; b < cap / bm; b += blockDim.x)
            block_expert[b] = -1;
        for (int i = tid; i <= E; i += blockDim.x)
            offsets[i] = offs[i];
        if (tid == 0)
            num_padded[0] = npad;
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
    int *offs, *total;
    align_block(ids, A, E, bm, cap, true, sorted_ids, block_expert, offsets, num_padded,
                dev_status, nullptr, &offs, &total);
}

// Standalone gather: xg[slot] = x[token of slot] (fp16, block order), zero
// for padding slots, for every slot below num_padded.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t *__restrict__ x, int d, int k,
                                                     int A, const int32_t *__restrict__ sorted_ids,
                                                     const int32_t *__restrict__ num_padded,
                                                     uint16_t *__restrict__ xg)
{
    const int c8n = d / 8;
    const int64_t total = static_cast<int64_t>(__ldg(num_padded)) * c8n;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t slot = i / c8n;
        const int c8 = static_cast<int>(i - slot * c8n);
        const int a = __ldg(sorted_ids + slot);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (static_cast<unsigned>(a) < static_cast<unsigned>(A))
            o = bf16x8_to_f16_korder(__ldg(
                reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(a / k) * d + 8 * c8)));
        *reinterpret_cast<uint4 *>(xg + slot * d + 8 * c8) = o;
    }
}

// Fused alignment + gather.  Every CTA computes the (cheap) alignment in its
// own shared memory, so no CTA waits for another; CTA 0 also writes the
// alignment outputs.  CTA b then copies the rows of tokens
// [b*tpc, (b+1)*tpc) to the slots of their k assignments (each x row is read
// once) and zeroes the padding slots of experts e = b, b + G, ...
__global__ void __launch_bounds__(kAlignWarps * 32, 1)
    moe_align_gather_kernel(const int32_t *__restrict__ ids, int M, int k, int E, int bm, int cap,
                            int32_t *__restrict__ sorted_ids, int32_t *__restrict__ block_expert,
                            int32_t *__restrict__ offsets, int32_t *__restrict__ num_padded,
                            int32_t *__restrict__ dev_status, const uint16_t *__restrict__ x,
                            int d, uint16_t *__restrict__ xg, int tpc)
{
    extern __shared__ int sm[];
    pdl_wait();
    pdl_trigger();
    const int A = M * k;
    int *pos = sm + align_smem_bytes(E) / sizeof(int);   // [A]
    int *offs, *total;
    align_block(ids, A, E, bm, cap, blockIdx.x == 0, sorted_ids, block_expert, offsets, num_padded,
                dev_status, pos, &offs, &total);
    __syncthreads();
    const int c8n = d / 8;
    const int t0 = blockIdx.x * tpc, t1 = min(M, t0 + tpc);
    const int64_t n = static_cast<int64_t>(max(0, t1 - t0)) * c8n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const int t = t0 + static_cast<int>(i / c8n);
        const int c8 = static_cast<int>(i % c8n);
        const uint4 o = bf16x8_to_f16_korder(
            __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t) * d + 8 * c8)));
        for (int j = 0; j < k; j++) {
            const int slot = pos[t * k + j];
            if (slot >= 0)
                *reinterpret_cast<uint4 *>(xg + static_cast<int64_t>(slot) * d + 8 * c8) = o;
        }
    }
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const int s0 = offs[e] + total[e], s1 = offs[e + 1];
        const int64_t m = static_cast<int64_t>(s1 - s0) * c8n;
        for (int64_t i = threadIdx.x; i < m; i += blockDim.x) {
            const int64_t slot = s0 + i / c8n;
            *reinterpret_cast<uint4 *>(xg + slot * d + 8 * (i % c8n)) = make_uint4(0, 0, 0, 0);
        }
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
    const size_t smem = align_smem_bytes(E);
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
                          cudaStream_t stream)
{
    const int64_t total = cap * (d / 8);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 4096));
    gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, d, k, M * k, sorted_ids,
                                                                      num_padded, xg);
    return cudaGetLastError();
}

size_t align_gather_smem_bytes(int M, int k, int E)
{
    return align_smem_bytes(E) + sizeof(int) * static_cast<size_t>(M) * k;
}

cudaError_t launch_align_gather(const int32_t *ids, int M, int k, int E, int block_m, int64_t cap,
                                int32_t *sorted_ids, int32_t *block_expert, int32_t *offsets,
                                int32_t *num_padded, int32_t *dev_status, const uint16_t *x,
                                int d, uint16_t *xg, int num_sms, cudaStream_t stream)
{
    const size_t smem = align_gather_smem_bytes(M, k, E);
    cudaError_t err = set_align_smem(reinterpret_cast<const void *>(moe_align_gather_kernel));
    if (err != cudaSuccess)
        return err;
    // about two tokens per CTA at the pages' canvas, at most one CTA per SM
    const int grid = std::max(1, std::min(num_sms, (M + 1) / 2));
    const int tpc = (M + grid - 1) / grid;
    return launch_pdl(moe_align_gather_kernel, dim3(grid), dim3(kAlignWarps * 32), smem, stream,
                      ids, M, k, E, block_m, static_cast<int>(cap), sorted_ids, block_expert,
                      offsets, num_padded, dev_status, x, d, xg, tpc);
}

}  // namespace w4
