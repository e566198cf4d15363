// rmsnorm.cu -- y = x / sqrt(mean(x^2) + eps) * weight over the last axis in
// one kernel ("dg-w4-kernels" -- RMSNorm; "Inference: Making every denoising
// pass fast" -- RMSNorm: each activation rescaled by its root-mean-square
// magnitude).  x, weight and y are bf16; the arithmetic is fp32 and y is
// rounded to bf16 once.
//
// One warp per row holds the row in registers (VPL 16-byte vectors per lane,
// d <= 32 * 8 * VPL), so x is read from HBM once and y written once.  Rows
// wider than that take a CTA per row that reads x twice (the second time
// from L2).
#include <cuda_bf16.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace w4 {

namespace {

constexpr int kNormWarps = 8;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float sumsq8(uint4 v)
{
    float s = 0.0f;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        s = fmaf(bf_lo(w[i]), bf_lo(w[i]), s);
        s = fmaf(bf_hi(w[i]), bf_hi(w[i]), s);
    }
    return s;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// y = (x * inv) * w for 8 elements
__device__ __forceinline__ uint4 scale8(uint4 v, uint4 w, float inv)
{
    uint4 o;
    o.x = pack_bf16x2(bf_lo(v.x) * inv * bf_lo(w.x), bf_hi(v.x) * inv * bf_hi(w.x));
    o.y = pack_bf16x2(bf_lo(v.y) * inv * bf_lo(w.y), bf_hi(v.y) * inv * bf_hi(w.y));
    o.z = pack_bf16x2(bf_lo(v.z) * inv * bf_lo(w.z), bf_hi(v.z) * inv * bf_hi(w.z));
    o.w = pack_bf16x2(bf_lo(v.w) * inv * bf_lo(w.w), bf_hi(v.w) * inv * bf_hi(w.w));
    return o;
}

template <int VPL>
__global__ void __launch_bounds__(32 * kNormWarps)
    rmsnorm_warp_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ w, int M, int d8,
                        float inv_d, float eps, uint4 *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    if (t >= M)
        return;
    const uint4 *xr = x + static_cast<int64_t>(t) * d8;
    uint4 v[VPL], wv[VPL];
    float ss = 0.0f;
    // x and weight loads all in flight together: one memory round trip
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int c = lane + 32 * i;
        v[i] = c < d8 ? __ldcs(xr + c) : make_uint4(0, 0, 0, 0);
        wv[i] = c < d8 ? __ldg(w + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < VPL; i++)
        ss += sumsq8(v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(fmaf(ss, inv_d, eps));
    uint4 *yr = y + static_cast<int64_t>(t) * d8;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int c = lane + 32 * i;
        if (c < d8)
            __stcs(yr + c, scale8(v[i], wv[i], inv));
    }
}

constexpr int kNormRowThreads = 512;

__global__ void __launch_bounds__(kNormRowThreads)
    rmsnorm_row_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ w, int M, int d8,
                       float inv_d, float eps, uint4 *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *xr = x + static_cast<int64_t>(t) * d8;
    float ss = 0.0f;
    for (int c = tid; c < d8; c += kNormRowThreads)
        ss += sumsq8(__ldg(xr + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float part[kNormRowThreads / 32];
    if (lane == 0)
        part[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int i = 0; i < kNormRowThreads / 32; i++)   // the same order in every thread
        tot += part[i];
    const float inv = rsqrtf(fmaf(tot, inv_d, eps));
    uint4 *yr = y + static_cast<int64_t>(t) * d8;
    for (int c = tid; c < d8; c += kNormRowThreads)
        __stcs(yr + c, scale8(__ldg(xr + c), __ldg(w + c), inv));
}

template <int VPL>
cudaError_t launch_warp(const uint16_t *x, const uint16_t *w, int M, int d, float eps, uint16_t *y,
                        cudaStream_t stream)
{
    return launch_pdl(rmsnorm_warp_kernel<VPL>, dim3((M + kNormWarps - 1) / kNormWarps),
                      dim3(32 * kNormWarps), 0, stream, reinterpret_cast<const uint4 *>(x),
                      reinterpret_cast<const uint4 *>(w), M, d / 8, 1.0f / static_cast<float>(d),
                      eps, reinterpret_cast<uint4 *>(y));
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t *x, const uint16_t *w, int M, int d, float eps,
                           uint16_t *y, cudaStream_t stream)
{
    if (M == 0)
        return cudaSuccess;
    const int vpl = (d / 8 + 31) / 32;
    if (vpl <= 1)
        return launch_warp<1>(x, w, M, d, eps, y, stream);
    if (vpl <= 2)
        return launch_warp<2>(x, w, M, d, eps, y, stream);
    if (vpl <= 4)
        return launch_warp<4>(x, w, M, d, eps, y, stream);
    if (vpl <= 8)
        return launch_warp<8>(x, w, M, d, eps, y, stream);
    if (vpl <= 12)
        return launch_warp<12>(x, w, M, d, eps, y, stream);
    if (vpl <= 16)
        return launch_warp<16>(x, w, M, d, eps, y, stream);
    return launch_pdl(rmsnorm_row_kernel, dim3(M), dim3(kNormRowThreads), 0, stream,
                      reinterpret_cast<const uint4 *>(x), reinterpret_cast<const uint4 *>(w), M,
                      d / 8, 1.0f / static_cast<float>(d), eps, reinterpret_cast<uint4 *>(y));
}

}  // namespace w4
