// korder.cuh -- the contraction order used inside every block of 8 elements
// by the grouped GEMMs, and the helpers that produce activations in it.
//
// Eight uint4 codes sit in one 32-bit word (code i in bits 4i..4i+3).  Masking
// the word >> 4i with 0x000F000F gives the 16-bit pairs (q0,q4) (q1,q5)
// (q2,q6) (q3,q7) with one shift and one LOP3 each, so position p of
// a block holds original index k(p) = (p >> 1) + 4 * (p & 1), and original
// index k sits at position pos(k) = 2 * (k & 3) + (k >> 2).  Permuting both
// operands of a dot product the same way leaves it unchanged.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace w4 {

__host__ __device__ constexpr int korder_pos(int k) { return ((k & 3) << 1) | (k >> 2); }

// fp32 pair -> fp16x2 (lo in the low half), round to nearest, saturating at
// +-65504 instead of overflowing to infinity.
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 bf16 values x0..x7 (16 bytes) -> 8 fp16 values in block order
// x0 x4 x1 x5 x2 x6 x3 x7.  bf16 -> fp16 is exact for magnitudes in
// [2^-14, 65504] and rounds to the nearest fp16 subnormal below that;
// larger magnitudes saturate to +-65504.
__device__ __forceinline__ uint4 bf16x8_to_f16_korder(uint4 v)
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

}  // namespace w4
