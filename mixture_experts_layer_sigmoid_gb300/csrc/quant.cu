// quant.cu -- blockwise FP8 (E4M3) quantisers of the MOE_FP8_BLOCK layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5:
// blockwise FP8 with 1x128 activation/gradient tiles and 128x128 weight
// blocks; §5 (Kernel and shape optimization): quantisation fused with the
// padding of the dynamic expert segments. Each block's scale is
// s = amax / 448 (fp32, IEEE division; s = 1 for an all-zero block) and a
// value v is stored as E4M3(v / s), rounded to nearest even and saturated.
//
// Kernels:
//   permute_quant_kernel  x -> permuted rows Xp (bf16) and their 1x128 codes
//   quant_rows_kernel     [rows][C] bf16 -> codes [rows][C], 1x128 scales
//   quant_t_kernel        [rows][C] bf16 -> transposed codes [C][rows], scales
//                         per column over 128 rows, or per 128x128 tile
//   quant_w_kernel        weights [E][R][C] -> 128x128-block codes in both
//                         orientations ([E][R][C] and [E][C][R])
#include "internal.h"

#include <cuda_fp8.h>

namespace moe {
namespace {

__device__ __forceinline__ float block_scale(float amax)
{
    return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
}

__device__ __forceinline__ uint8_t e4m3(float v, float s)
{
    return (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE, __NV_E4M3);
}

// 8 bf16 -> 8 fp32
__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8])
{
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint2 codes8(const float (&v)[8], float s)
{
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= (uint32_t)e4m3(v[i], s) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= (uint32_t)e4m3(v[4 + i], s) << (8 * i);
    return make_uint2(lo, hi);
}

// amax over the 16 lanes that share one 128-element block (8 values each)
__device__ __forceinline__ float amax16(const float (&v)[8])
{
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    return a;
}

// Blocks [0, T): token t -> its k rows of Xp (bf16) and Xq (codes, scales).
// Blocks [T, T+E): pad rows of expert e: zero rows, unit scales.
__global__ void __launch_bounds__(128)
permute_quant_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ row_of,
                     const int* __restrict__ poff, const int* __restrict__ counts, int T_, int H,
                     int k, __nv_bfloat16* __restrict__ Xp, uint8_t* __restrict__ Xq,
                     float* __restrict__ sX)
{
    const int b = blockIdx.x;
    const int nv = H / 8, nb = H / 128;
    if (b >= T_) {
        const int e = b - T_;
        for (int r = poff[e] + counts[e]; r < poff[e + 1]; ++r) {
            for (int v = threadIdx.x; v < nv; v += blockDim.x) {
                reinterpret_cast<uint4*>(Xp + (size_t)r * H)[v] = make_uint4(0, 0, 0, 0);
                reinterpret_cast<uint2*>(Xq + (size_t)r * H)[v] = make_uint2(0, 0);
            }
            for (int j = threadIdx.x; j < nb; j += blockDim.x) sX[(size_t)r * nb + j] = 1.f;
        }
        return;
    }
    int rows[kMaxK];
    for (int j = 0; j < k; ++j) rows[j] = row_of[(size_t)b * k + j];
    // whole warps iterate together (the 16-lane amax shuffles need them);
    // nv is a multiple of 16, so a 16-lane group is all in or all out
    for (int v0 = 0; v0 < nv; v0 += blockDim.x) {
        const int v = v0 + threadIdx.x;
        const bool act = v < nv;
        const uint4 u = act ? reinterpret_cast<const uint4*>(x + (size_t)b * H)[v] : make_uint4(0, 0, 0, 0);
        float f[8];
        unpack8(u, f);
        const float s = block_scale(amax16(f));
        if (!act) continue;
        const uint2 c = codes8(f, s);
        for (int j = 0; j < k; ++j) {
            reinterpret_cast<uint4*>(Xp + (size_t)rows[j] * H)[v] = u;
            reinterpret_cast<uint2*>(Xq + (size_t)rows[j] * H)[v] = c;
            if ((threadIdx.x & 15) == 0) sX[(size_t)rows[j] * nb + v / 16] = s;
        }
    }
}

// One block per row (rows < *rows_dev); C a multiple of 128.
__global__ void __launch_bounds__(128)
quant_rows_kernel(const __nv_bfloat16* __restrict__ in, const int* __restrict__ rows_dev,
                  int rows_fixed, int C, uint8_t* __restrict__ q, float* __restrict__ s)
{
    const int r = blockIdx.x;
    if (r >= (rows_dev ? *rows_dev : rows_fixed)) return;
    const int nv = C / 8, nb = C / 128;
    for (int v0 = 0; v0 < nv; v0 += blockDim.x) {
        const int v = v0 + threadIdx.x;
        const bool act = v < nv;
        float f[8];
        unpack8(act ? reinterpret_cast<const uint4*>(in + (size_t)r * C)[v] : make_uint4(0, 0, 0, 0), f);
        const float sc = block_scale(amax16(f));
        if (!act) continue;
        reinterpret_cast<uint2*>(q + (size_t)r * C)[v] = codes8(f, sc);
        if ((threadIdx.x & 15) == 0) s[(size_t)r * nb + v / 16] = sc;
    }
}

// Tile (128 rows x 128 columns) of in [rows][C] -> qT [C][rows_cap].
// tiles == 0: one scale per column of the tile, sT[c][rb] (row stride
// rows_cap/128); tiles == 1: one scale per tile, sT[cb][rb].
__global__ void __launch_bounds__(256)
quant_t_kernel(const __nv_bfloat16* __restrict__ in, const int* __restrict__ rows_dev,
               int rows_fixed, int C, int rows_cap, int tiles, uint8_t* __restrict__ qT,
               float* __restrict__ sT)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    __shared__ float red[256];
    const int cb = blockIdx.x, rb = blockIdx.y;
    const int r0 = rb * 128, c0 = cb * 128;
    if (r0 >= (rows_dev ? *rows_dev : rows_fixed)) return;
    // load 128 x 128 (16 vectors of 8 per row)
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
        const int rr = i / 16, vv = i % 16;
        *reinterpret_cast<uint4*>(&tile[rr][vv * 8]) =
            reinterpret_cast<const uint4*>(in + (size_t)(r0 + rr) * C + c0)[vv];
    }
    __syncthreads();
    // column amax: threads (c = tid % 128, half = tid / 128) over 64 rows each
    const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
    float a = 0.f;
    for (int rr = half * 64; rr < half * 64 + 64; ++rr) a = fmaxf(a, fabsf(__bfloat162float(tile[rr][c])));
    red[threadIdx.x] = a;
    __syncthreads();
    float sc;
    if (tiles) {
        if (threadIdx.x < 128) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + 128]);
        __syncthreads();
        for (int off = 64; off > 0; off >>= 1) {
            if (threadIdx.x < off) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + off]);
            __syncthreads();
        }
        sc = block_scale(red[0]);
        if (threadIdx.x == 0) sT[(size_t)cb * (rows_cap / 128) + rb] = sc;
    } else {
        sc = block_scale(fmaxf(red[c], red[c + 128]));
        if (half == 0) sT[(size_t)(c0 + c) * (rows_cap / 128) + rb] = sc;
    }
    // column c -> output row c0 + c, bytes [r0 + 64 half, +64)
    uint8_t* dst = qT + (size_t)(c0 + c) * rows_cap + r0 + half * 64;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t word = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b)
                word |= (uint32_t)e4m3(__bfloat162float(tile[half * 64 + g * 16 + q4 * 4 + b][c]), sc) << (8 * b);
            w[q4] = word;
        }
        reinterpret_cast<uint4*>(dst)[g] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 128x128 block (rb, cb) of expert e of W [E][R][C] -> codes in both
// orientations and the block's scale in both scale layouts.
__global__ void __launch_bounds__(256)
quant_w_kernel(const __nv_bfloat16* __restrict__ W, int R, int C, uint8_t* __restrict__ q,
               float* __restrict__ s, uint8_t* __restrict__ qT, float* __restrict__ sT)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    __shared__ float red[256];
    const int cb = blockIdx.x, rb = blockIdx.y, e = blockIdx.z;
    const size_t base = (size_t)e * R * C;
    const int r0 = rb * 128, c0 = cb * 128;
    float a = 0.f;
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
        const int rr = i / 16, vv = i % 16;
        const uint4 u = reinterpret_cast<const uint4*>(W + base + (size_t)(r0 + rr) * C + c0)[vv];
        *reinterpret_cast<uint4*>(&tile[rr][vv * 8]) = u;
        float f[8];
        unpack8(u, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
    }
    red[threadIdx.x] = a;
    __syncthreads();
    for (int off = 128; off > 0; off >>= 1) {
        if (threadIdx.x < off) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + off]);
        __syncthreads();
    }
    const float sc = block_scale(red[0]);
    if (threadIdx.x == 0) {
        s[((size_t)e * (R / 128) + rb) * (C / 128) + cb] = sc;
        sT[((size_t)e * (C / 128) + cb) * (R / 128) + rb] = sc;
    }
    // original orientation: thread -> (row, 64 columns)
    {
        const int rr = threadIdx.x >> 1, hf = threadIdx.x & 1;
        uint8_t* dst = q + base + (size_t)(r0 + rr) * C + c0 + hf * 64;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) word |= (uint32_t)e4m3(__bfloat162float(tile[rr][hf * 64 + g * 16 + q4 * 4 + b]), sc) << (8 * b);
                w[q4] = word;
            }
            reinterpret_cast<uint4*>(dst)[g] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    // transposed: thread -> (column, 64 rows)
    {
        const int cc = threadIdx.x >> 1, hf = threadIdx.x & 1;
        uint8_t* dst = qT + base + (size_t)(c0 + cc) * R + r0 + hf * 64;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) word |= (uint32_t)e4m3(__bfloat162float(tile[hf * 64 + g * 16 + q4 * 4 + b][cc]), sc) << (8 * b);
                w[q4] = word;
            }
            reinterpret_cast<uint4*>(dst)[g] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace

cudaError_t launch_permute_quant(const __nv_bfloat16* x, const int* row_of, const int* poff,
                                 const int* counts, int T_, int H, int E, int k, __nv_bfloat16* Xp,
                                 uint8_t* Xq, float* sX, cudaStream_t s)
{
    permute_quant_kernel<<<T_ + E, 128, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xp, Xq, sX);
    return cudaGetLastError();
}

cudaError_t launch_quant_rows(const __nv_bfloat16* in, const int* rows_dev, int rows_max, int C,
                              uint8_t* q, float* sc, cudaStream_t s)
{
    quant_rows_kernel<<<rows_max, 128, 0, s>>>(in, rows_dev, rows_max, C, q, sc);
    return cudaGetLastError();
}

cudaError_t launch_quant_t(const __nv_bfloat16* in, const int* rows_dev, int rows_cap, int C,
                           int tiles, uint8_t* qT, float* sT, cudaStream_t s)
{
    dim3 grid(C / 128, rows_cap / 128);
    quant_t_kernel<<<grid, 256, 0, s>>>(in, rows_dev, rows_cap, C, rows_cap, tiles, qT, sT);
    return cudaGetLastError();
}

cudaError_t launch_quant_w(const __nv_bfloat16* W, int E, int R, int C, uint8_t* q, float* sc,
                           uint8_t* qT, float* sT, cudaStream_t s)
{
    dim3 grid(C / 128, R / 128, E);
    quant_w_kernel<<<grid, 256, 0, s>>>(W, R, C, q, sc, qT, sT);
    return cudaGetLastError();
}

}  // namespace moe
