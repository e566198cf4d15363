// quantize.cu -- quantize_w4: asymmetric uint4 with an fp16 scale and zero
// point per group, two codes per byte ("diffusiongemma-26B-A4B-w4a16" --
// Checkpoint format; -- Benchmarks: round-to-nearest min/max, no calibration).
//
// One warp per (row, group).  Each lane holds group/32 consecutive elements;
// the group's min and max come from a warp reduction.  Every rounding step is
// an explicit IEEE fp32 operation (no contraction into FMA) so that the codes,
// scales and zeros are bit-identical on any conforming implementation:
//   s = (max - min) / 15 -> fp16 (zero -> 1.0); z = -min / s16 -> fp16;
//   q = clamp(rint(w / s16 + z16), 0, 15), rint rounding half to even.
#include <cuda_fp16.h>

#include "launch.h"

namespace w4 {

template <int EPL>
__global__ void __launch_bounds__(256) quantize_w4_kernel(const float *__restrict__ W,
                                                          int64_t n_groups, int group,
                                                          uint8_t *__restrict__ q,
                                                          uint16_t *__restrict__ s,
                                                          uint16_t *__restrict__ z)
{
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    if (gw >= n_groups)
        return;
    const int lane = threadIdx.x & 31;
    // groups are contiguous: row r, group g starts at r*K + g*group = gw*group
    const float *src = W + gw * group + lane * EPL;
    float v[EPL];
#pragma unroll
    for (int i = 0; i < EPL; i += 2) {
        const float2 t = __ldg(reinterpret_cast<const float2 *>(src + i));
        v[i] = t.x;
        v[i + 1] = t.y;
    }
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int i = 1; i < EPL; i++) {
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    __half sh = __float2half_rn(sc);
    if ((__half_as_ushort(sh) & 0x7fffu) == 0)
        sh = __ushort_as_half(static_cast<unsigned short>(0x3c00u));
    const float sf = __half2float(sh);
    const float zf = __fadd_rn(__fdiv_rn(-lo, sf), 0.0f);
    const __half zh = __float2half_rn(zf);
    const float zz = __half2float(zh);

    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const float t = __fadd_rn(__fdiv_rn(v[i], sf), zz);
        const float r = rintf(t);
        const int qi = r < 0.0f ? 0 : (r > 15.0f ? 15 : static_cast<int>(r));
        packed |= static_cast<uint32_t>(qi) << (4 * i);
    }
    uint8_t *dst = q + gw * (group / 2) + lane * (EPL / 2);
    if constexpr (EPL == 2)
        *dst = static_cast<uint8_t>(packed);
    else if constexpr (EPL == 4)
        *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
    else
        *reinterpret_cast<uint32_t *>(dst) = packed;
    if (lane == 0) {
        s[gw] = __half_as_ushort(sh);
        z[gw] = __half_as_ushort(zh);
    }
}

cudaError_t launch_quantize(const float *W, int64_t rows, int K, int group, uint8_t *q,
                            uint16_t *s, uint16_t *z, cudaStream_t stream)
{
    const int64_t n_groups = rows * (K / group);
    if (n_groups == 0)
        return cudaSuccess;
    const int warps_per_block = 8;
    const int64_t blocks = (n_groups + warps_per_block - 1) / warps_per_block;
    if (blocks > 0x7fffffff)
        return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks)), block(32 * warps_per_block);
    switch (group) {
    case 64:
        quantize_w4_kernel<2><<<grid, block, 0, stream>>>(W, n_groups, group, q, s, z);
        break;
    case 128:
        quantize_w4_kernel<4><<<grid, block, 0, stream>>>(W, n_groups, group, q, s, z);
        break;
    case 256:
        quantize_w4_kernel<8><<<grid, block, 0, stream>>>(W, n_groups, group, q, s, z);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace w4
