// Activations as sums of MXFP8 terms: the B operand of the block-scaled
// tensor-core GEMMs.
//
// A 32-element block v of one activation row (32 consecutive K elements:
// hidden units for W13, intermediate features for W2) is written as
//     v = sum_t 2^(e1 - 4t) * q_t + r,   t = 0 .. NT-1,
// q_t E4M3 values (OCP FP8: 1 sign, 4 exponent bits with bias 7, 3 mantissa
// bits, largest finite 448), 2^(e1 - 4t) an E8M0 scale per block and term.
// e1 is the smallest exponent with max|v| <= 448 * 2^e1, so the first term
// never saturates. Each q_t is the E4M3 round-to-nearest-even of the residual
// left by the terms before it, divided by its scale; the residual after term
// t is at most half an E4M3 ulp (16 * 2^(e1 - 4t) at the top binade), which
// the next scale, 2^-4 smaller, holds without saturation.
// A bf16 value (8 significant bits) is represented exactly by two terms
// unless the block's magnitudes span more than E4M3's 2^17 range; an fp32
// value keeps about 8 bits with two terms and about 12 with three.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

namespace moe {

// 2^n for -149 <= n <= 127, built from its bits.
__device__ __forceinline__ float pow2f(int n)
{
    return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(1 << (n + 149));
}

// Smallest e (>= -127) with mx <= 448 * 2^e; -127 for a zero block.
__device__ __forceinline__ int mxfp8_block_exp(float mx)
{
    const int bits = __float_as_int(mx);
    const int ex = (bits >> 23) & 0xFF;
    if (!(mx > 0.f) || ex == 0) return -127;       // zero (or below the fp32 normal range)
    const int E = ex - 127;                         // mx = 1.m * 2^E
    const int e = (bits & 0x7FFFFF) <= 0x600000 ? E - 8 : E - 7;   // 1.m <= 1.75: 448 * 2^(E-8) suffices
    return e < -127 ? -127 : e;
}

// E4M3 (round to nearest even, saturating to +-448) of two values: byte 0 = lo, byte 1 = hi.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// The two E4M3 values of a 16-bit pair (byte 0 -> .x, byte 1 -> .y), exactly.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t pair)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(pair));
    const __half2 hh = *reinterpret_cast<const __half2 *>(&h2);
    return make_float2(__low2float(hh), __high2float(hh));
}

// Term t of a pair of values sharing the block exponent e1: returns the E4M3 byte pair and
// subtracts the represented part from the residuals r0, r1. `sbyte` receives the E8M0 scale byte.
__device__ __forceinline__ uint32_t mxfp8_term_pair(float &r0, float &r1, int e1, int t, uint32_t &sbyte)
{
    int et = e1 - 4 * t;
    if (et < -127) et = -127;
    sbyte = (uint32_t)(et + 127);
    const float inv = pow2f(-et > 127 ? 127 : -et), sc = pow2f(et);
    const uint32_t q = e4m3x2_rn(r0 * inv, r1 * inv);
    const float2 v = e4m3x2_value(q);
    r0 -= v.x * sc;
    r1 -= v.y * sc;
    return q;
}

// Term t of two values with their own block exponents e0 and e1 (one conversion for both; the
// conversion rounds each element on its own): returns the E4M3 byte pair (byte 0 for r0) and the two
// E8M0 scale bytes, and updates both residuals.
__device__ __forceinline__ uint32_t mxfp8_term_2x(float &r0, float &r1, int e0, int e1, int t, uint32_t &sb0,
                                                  uint32_t &sb1)
{
    int et0 = e0 - 4 * t, et1 = e1 - 4 * t;
    if (et0 < -127) et0 = -127;
    if (et1 < -127) et1 = -127;
    sb0 = (uint32_t)(et0 + 127);
    sb1 = (uint32_t)(et1 + 127);
    const float inv0 = pow2f(-et0 > 127 ? 127 : -et0), inv1 = pow2f(-et1 > 127 ? 127 : -et1);
    const uint32_t q = e4m3x2_rn(r0 * inv0, r1 * inv1);
    const float2 v = e4m3x2_value(q);
    r0 -= v.x * pow2f(et0);
    r1 -= v.y * pow2f(et1);
    return q;
}

}  // namespace moe
