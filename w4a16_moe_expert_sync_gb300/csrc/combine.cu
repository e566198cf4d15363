// combine.cu -- fixed-order, atomics-free weighted combine
// ("Inference: Making every denoising pass fast" -- Quantisation alone leaves
// a sparse execution problem: a token's eight expert outputs are reduced in a
// fixed order instead of index_add_, because reordered floating-point sums
// change low bits and a one-ulp change can fork a denoising trajectory).
//
// Each thread owns four consecutive output columns of one token and runs the
// fp32 chain acc = fma(w_j, y_j, acc) for j = 0..k-1, always in that order,
// then rounds once to bf16.  Every output element has exactly one writer, so
// the result is bit-identical from run to run.
#include <cuda_bf16.h>

#include "combine_fold.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4 {

__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y,
                                                      const int32_t *__restrict__ ids,
                                                      const float *__restrict__ w, int M, int k,
                                                      int d, int E, uint16_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int d4 = d / 4;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(M) * d4)
        return;
    const int t = static_cast<int>(i / d4);
    const int c = static_cast<int>(i % d4) * 4;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    // eight assignments at a time: every load issued before the first FMA
    // (each assignment's y row exists; an invalid expert id only drops its
    // term), then the chain in assignment order
    for (int j0 = 0; j0 < k; j0 += 8) {
        float4 v[8];
        float wj[8];
        bool ok[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int j = j0 + u;
            ok[u] = false;
            if (j < k) {
                const int64_t a = static_cast<int64_t>(t) * k + j;
                const int e = __ldg(ids + a);
                ok[u] = e >= 0 && e < E;
                wj[u] = __ldg(w + a);
                v[u] = __ldcs(reinterpret_cast<const float4 *>(y + a * d + c));
            }
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            if (ok[u]) {
                a0 = fmaf(wj[u], v[u].x, a0);
                a1 = fmaf(wj[u], v[u].y, a1);
                a2 = fmaf(wj[u], v[u].z, a2);
                a3 = fmaf(wj[u], v[u].w, a3);
            }
        }
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a2, a3);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t *>(&lo);
    pk.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(out + static_cast<int64_t>(t) * d + c) = pk;
}

cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int M, int k,
                           int d, int E, uint16_t *out, cudaStream_t stream)
{
    const int64_t n = static_cast<int64_t>(M) * (d / 4);
    if (n == 0)
        return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                      y, ids, w, M, k, d, E, out);
}

// The counters of the combine folded into the down GEMM (combine_fold.cuh),
// one warp per token, for callers that run the down GEMM with the combine
// on their own (the layer sets them in its gate_up launch instead).
__global__ void __launch_bounds__(256) combine_prepare_kernel(const int32_t *__restrict__ ids,
                                                              int M, int k, int E, int d,
                                                              int32_t *__restrict__ cnt,
                                                              uint16_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t < M)
        fold_prepare_token(t, threadIdx.x & 31, ids, k, E, d, cnt, out);
}

cudaError_t launch_combine_prepare(const int32_t *ids, int M, int k, int E, int d, int32_t *cnt,
                                   uint16_t *out, cudaStream_t stream)
{
    if (M == 0)
        return cudaSuccess;
    return launch_pdl(combine_prepare_kernel, dim3(static_cast<unsigned>((M + 7) / 8)), dim3(256),
                      0, stream, ids, M, k, E, d, cnt, out);
}

}  // namespace w4
