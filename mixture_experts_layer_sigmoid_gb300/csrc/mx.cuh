// mx.cuh -- MXFP8 block encoding shared by the quantisers (quant_mx.cu) and the
// GEMM epilogues that quantise their own output (gemm_mx.cu).
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): MXFP8 with 1x32 granularity. A block of 32
// values with largest magnitude amax gets the scale 2^e, e the smallest
// integer with amax <= 448 2^e, clamped to [-127, 127] (-127 for an all-zero
// block), stored as the UE8M0 byte e + 127; each value is stored as the E4M3
// code of v 2^-e (exact scaling, round to nearest even).
// Scale atoms: an operand read as [rows][K] keeps one 512-byte atom per
// 128-row tile and 128-deep K block, byte atom_byte(m, j) holding the scale
// of tile row m and 32-deep sub-block j.
#pragma once
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// e of a block maximum (a non-negative bf16 or fp32 value): amax = 1.f 2^(E-127)
// with f the 23-bit fraction; amax <= 448 2^e with 448 = 1.75 2^8.
__device__ __forceinline__ int mx_exp(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    const int E = (int)(b >> 23);
    if (E == 0) return -127;                       // zero or below 2^-126
    const int e = (b & 0x7FFFFFu) <= 0x600000u ? E - 135 : E - 134;
    return e < -127 ? -127 : e;
}

// 2^-e as an fp32 (e in [-127, 127]; 2^-127 is a subnormal, still exact)
__device__ __forceinline__ float mx_inv(int e)
{
    const int be = 127 - e;                        // biased exponent of 2^-e
    return be >= 1 ? __uint_as_float((uint32_t)be << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ size_t atom_byte(int m, int j) { return (size_t)(16 * (m & 31) + 4 * (m >> 5) + j); }

// 32 values -> their block exponent and 32 codes (two 16-byte words)
__device__ __forceinline__ int encode32(const float* v, uint4& c0, uint4& c1)
{
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
    const int e = mx_exp(a);
    const float s = mx_inv(e);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = e4m3x4(v[4 * i] * s, v[4 * i + 1] * s, v[4 * i + 2] * s, v[4 * i + 3] * s);
    c0 = make_uint4(w[0], w[1], w[2], w[3]);
    c1 = make_uint4(w[4], w[5], w[6], w[7]);
    return e;
}

}  // namespace moe
