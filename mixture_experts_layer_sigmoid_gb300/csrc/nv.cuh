// nv.cuh -- NVFP4 block encoding shared by the quantisers (quant_nv.cu) and
// the grouped GEMM's epilogue (gemm_mx.cu).
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): NVFP4 for Blackwell. The pages fix no
// parameters; the format: E2M1 values (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
// 6), one unsigned E4M3 scale per 16 values along K, and one fp32 scale per
// tensor, S = 2688 / amax (2688 = 448 x 6; S = 1 for an all-zero tensor).
// Per block, each step an fp32 operation rounded to nearest even:
// a = max |v|, sb = E4M3(a S / 6) (the product first), s = value(sb),
// r = S / s, code = E2M1(v r) (ties to the even code, saturating at 6, the
// sign bit kept, zero included; all codes 0 when s = 0). A value reads as code x s / S: the tensor cores
// multiply the codes by their block scales, and the GEMM's epilogue divides
// by the two operands' tensor scales.
// Codes are packed two per byte, the lower-index value in the low nibble.
// Scale atoms: an operand read as [rows][K] keeps one 512-byte atom per
// 128-row tile and 64-value K chunk, byte atom_byte(m, j) holding the scale
// of tile row m and 16-value sub-block j of the chunk.
#pragma once
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ float nv_tensor_scale(float amax) { return amax > 0.f ? __fdiv_rn(2688.f, amax) : 1.f; }

// 1 / (S_a S_b): the factor that takes an accumulator of code x scale
// products back to values
__device__ __forceinline__ float nv_unscale(float amax_a, float amax_b)
{
    return 1.f / (nv_tensor_scale(amax_a) * nv_tensor_scale(amax_b));
}

// value of an unsigned E4M3 byte (E4M3 with the sign bit clear: 4 exponent
// bits with bias 7, 3 mantissa bits, subnormals below exponent 1)
__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    const int e = (int)((b >> 3) & 15u), m = (int)(b & 7u);
    return e == 0 ? (float)m * 0.001953125f : __uint_as_float((uint32_t)(e + 120) << 23) * (1.f + 0.125f * (float)m);
}

// E2M1 codes of two fp32 values in one byte, a in the low four bits: the
// conversion instruction (round to nearest even, saturating at 6, the sign
// kept)
__device__ __forceinline__ uint32_t e2m1x2(float a, float b)
{
    return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest) & 0xFFu;
}

// 16 values of one block -> their E4M3 scale byte and 16 codes (8 bytes)
__device__ __forceinline__ uint32_t nv_encode16(const float* v, float S, uint2& codes)
{
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
    const float sf = __fdiv_rn(__fmul_rn(a, S), 6.f);
    const uint32_t sb = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(sf, 0.f), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
    const float s = e4m3_value(sb);
    uint32_t w[2] = {0u, 0u};
    if (s > 0.f) {
        const float r = __fdiv_rn(S, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i >> 2] |= e2m1x2(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r)) << (8 * (i & 3));
    }
    codes = make_uint2(w[0], w[1]);
    return sb;
}

}  // namespace moe
