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
//   quant_w_kernel        weights [E][R][C] -> 128x128-block codes [E][R][C]
//                         (and optionally [E][C][R])
#include "internal.h"

#include <cuda_fp8.h>

namespace moe {
namespace {

__device__ __forceinline__ float block_scale(float amax)
{
    return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
}

// E4M3(v / s), rounded to nearest even and saturated, given r = 1/s rounded
// to nearest. y = v r is within two units in the last place of the rounded
// quotient, so both round to the same E4M3 value unless y lies within a few
// units of a rounding midpoint (the 20 mantissa bits E4M3 drops are within 4
// of half) or below the E4M3 normal range, where the rounding position moves;
// those rare values take the IEEE division itself.
__device__ __forceinline__ uint8_t e4m3(float v, float s, float r)
{
    float y = v * r;
    const uint32_t b = __float_as_uint(y) & 0x7fffffffu;
    if (b != 0u) {
        const int dist = (int)(b & 0xFFFFFu) - 0x80000;
        if ((b >> 23) < 121u || (dist >= -4 && dist <= 4)) y = __fdiv_rn(v, s);
    }
    return (uint8_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
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
    const float r = __frcp_rn(s);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= (uint32_t)e4m3(v[i], s, r) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= (uint32_t)e4m3(v[4 + i], s, r) << (8 * i);
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

// ---- 128x128 tiles: bf16 tile and its codes staged in shared memory.
// Codes are kept row-major with 144-byte rows; the 16-byte chunk k of row r
// sits at chunk k ^ ((r / 16) % 8), which makes the transposed read-out
// (4 columns x 16 rows per thread) free of bank conflicts.
constexpr int kQS = 144;
__device__ __forceinline__ int qs_off(int r, int byte)
{
    return r * kQS + ((((byte >> 4) ^ (r >> 4)) & 7) << 4) + (byte & 15);
}

// Load a 128x128 bf16 tile (row stride ld elements) into tile[][136]; returns
// this thread's amax over the 64 values it loaded.
__device__ __forceinline__ float load_tile(const __nv_bfloat16* __restrict__ src, size_t ld,
                                           __nv_bfloat16 (*tile)[136])
{
    uint4 u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = threadIdx.x + 256 * j, rr = i >> 4, vv = i & 15;
        u[j] = reinterpret_cast<const uint4*>(src + (size_t)rr * ld)[vv];
    }
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = threadIdx.x + 256 * j, rr = i >> 4, vv = i & 15;
        *reinterpret_cast<uint4*>(&tile[rr][vv * 8]) = u[j];
        float f[8];
        unpack8(u[j], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) a = fmaxf(a, fabsf(f[q]));
    }
    return a;
}

// max over the 256 threads of the block (red: 8 floats of shared memory)
__device__ __forceinline__ float block_max(float a, float* red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w]);
    return a;
}

// Row-wise encoding: thread -> row t/2, columns 64 (t%2) + [0, 64), each
// divided by its column's scale (sc_col, reciprocals rc_col) or the tile's
// (sc_col == null).
// Codes go to qs and, when dst is given, to dst (row stride ld bytes).
__device__ __forceinline__ void encode_rows(__nv_bfloat16 (*tile)[136], float sc, const float* sc_col,
                                            const float* rc_col, uint8_t* qs, uint8_t* dst, size_t ld)
{
    const int rr = threadIdx.x >> 1, hf = threadIdx.x & 1;
    const float rc = __frcp_rn(sc);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int c0 = hf * 64 + g * 16;
        float f[16];
        unpack8(*reinterpret_cast<const uint4*>(&tile[rr][c0]), *reinterpret_cast<float(*)[8]>(f));
        unpack8(*reinterpret_cast<const uint4*>(&tile[rr][c0 + 8]), *reinterpret_cast<float(*)[8]>(f + 8));
        uint32_t w[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t word = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = 4 * q4 + b;
                word |= (uint32_t)(sc_col ? e4m3(f[c], sc_col[c0 + c], rc_col[c0 + c]) : e4m3(f[c], sc, rc))
                        << (8 * b);
            }
            w[q4] = word;
        }
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(qs + qs_off(rr, c0)) = v;
        if (dst) *reinterpret_cast<uint4*>(dst + (size_t)rr * ld + c0) = v;
    }
}

// Transposed write-out of the staged codes: thread -> columns 4 (t/8) + [0, 4),
// rows 16 (t%8) + [0, 16); dst row c (= tile column c) has stride ldT bytes.
// Eight consecutive threads complete one 128-byte line of an output row.
__device__ __forceinline__ void write_transposed(const uint8_t* qs, uint8_t* dstT, size_t ldT)
{
    const int cg = threadIdx.x >> 3, ch = threadIdx.x & 7;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = *reinterpret_cast<const uint32_t*>(qs + qs_off(16 * ch + i, 4 * cg));
    uint32_t o[4][4];   // [column j][group of 4 rows]
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t lo01 = __byte_perm(w[4 * g], w[4 * g + 1], 0x5140);
        const uint32_t hi01 = __byte_perm(w[4 * g], w[4 * g + 1], 0x7362);
        const uint32_t lo23 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x5140);
        const uint32_t hi23 = __byte_perm(w[4 * g + 2], w[4 * g + 3], 0x7362);
        o[0][g] = __byte_perm(lo01, lo23, 0x5410);
        o[1][g] = __byte_perm(lo01, lo23, 0x7632);
        o[2][g] = __byte_perm(hi01, hi23, 0x5410);
        o[3][g] = __byte_perm(hi01, hi23, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(dstT + (size_t)(4 * cg + j) * ldT + 16 * ch) =
            make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
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
    __shared__ __align__(16) uint8_t qs[128 * kQS];
    __shared__ float red[256];
    __shared__ float scol[128], rcol[128];
    const int cb = blockIdx.x, rb = blockIdx.y;
    const int r0 = rb * 128, c0 = cb * 128;
    if (r0 >= (rows_dev ? *rows_dev : rows_fixed)) return;
    const float at = load_tile(in + (size_t)r0 * C + c0, C, tile);
    float sc = 0.f;
    if (tiles) {
        sc = block_scale(block_max(at, red));
        if (threadIdx.x == 0) sT[(size_t)cb * (rows_cap / 128) + rb] = sc;
    } else {
        __syncthreads();
        // column amax: threads (c = tid % 128, half = tid / 128) over 64 rows each
        const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
        float a = 0.f;
        for (int rr = half * 64; rr < half * 64 + 64; ++rr) a = fmaxf(a, fabsf(__bfloat162float(tile[rr][c])));
        red[threadIdx.x] = a;
        __syncthreads();
        if (half == 0) {
            const float s1 = block_scale(fmaxf(red[c], red[c + 128]));
            scol[c] = s1;
            rcol[c] = __frcp_rn(s1);
            sT[(size_t)(c0 + c) * (rows_cap / 128) + rb] = s1;
        }
    }
    __syncthreads();
    encode_rows(tile, tiles ? sc : 1.f, tiles ? nullptr : scol, rcol, qs, nullptr, 0);
    __syncthreads();
    write_transposed(qs, qT + (size_t)c0 * rows_cap + r0, rows_cap);
}

// 128x128 block (rb, cb) of expert e of W [E][R][C] -> codes and the block's
// scale, and (qT, sT given) the transposed codes and scale layout too.
__global__ void __launch_bounds__(256)
quant_w_kernel(const __nv_bfloat16* __restrict__ W, int R, int C, uint8_t* __restrict__ q,
               float* __restrict__ s, uint8_t* __restrict__ qT, float* __restrict__ sT)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    __shared__ __align__(16) uint8_t qs[128 * kQS];
    __shared__ float red[8];
    const int cb = blockIdx.x, rb = blockIdx.y, e = blockIdx.z;
    const size_t base = (size_t)e * R * C;
    const int r0 = rb * 128, c0 = cb * 128;
    const float sc = block_scale(block_max(load_tile(W + base + (size_t)r0 * C + c0, C, tile), red));
    if (threadIdx.x == 0) {
        s[((size_t)e * (R / 128) + rb) * (C / 128) + cb] = sc;
        if (sT) sT[((size_t)e * (C / 128) + cb) * (R / 128) + rb] = sc;
    }
    encode_rows(tile, sc, nullptr, nullptr, qs, q + base + (size_t)r0 * C + c0, C);
    if (!qT) return;                      // block-uniform
    __syncthreads();
    write_transposed(qs, qT + base + (size_t)c0 * R + r0, R);
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
    if (rows_max <= 0) return cudaSuccess;
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
