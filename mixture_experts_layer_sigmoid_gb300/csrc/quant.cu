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
//   permute_quant_kernel  x -> the 1x128 codes of the permuted rows (and,
//                         optionally, the bf16 permuted rows Xp)
//   quant_tiles_kernel    [rows][C] bf16 in 128x128 tiles -> any of: codes
//                         [rows][C] with 1x128 row scales or one scale per
//                         tile (weights), transposed codes [C][rows] with
//                         per-column (over 128 rows) or per-tile scales
#include "internal.h"

#include <cuda_fp8.h>

namespace moe {
namespace {

__device__ __forceinline__ float block_scale(float amax)
{
    return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
}

// The E4M3 codes of two values at once (scales s0, s1, rounded reciprocals
// r0, r1). The fp32 quotient RN(v / s) is formed with Markstein's correction
// of the product (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//   y0 = RN(v r),  y1 = RN(y0 + r RN(v - s y0))   (two fused multiply-adds),
// in packed f32x2 arithmetic. For a block maximum amax (bf16) with scale
// s = RN(amax / 448) >= 2^-112 and every bf16 v with |v| <= amax, E4M3(y1)
// equals E4M3(RN(v / s)): an exhaustive check over all such pairs
// (tests/e4m3_quotient_check.c) finds no difference;
// below that the remainder can underflow, and such tiny scales take the IEEE
// division. x.x of the packed pair is the low byte.
constexpr float kMinFastScale = 0x1p-112f;
__device__ __forceinline__ uint64_t f2_pack(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v)
{
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
__device__ __forceinline__ uint32_t e4m3x2(float v0, float v1, float s0, float s1, float r0, float r1)
{
    float2 y;
    if (s0 >= kMinFastScale && s1 >= kMinFastScale) {
        const uint64_t v = f2_pack(v0, v1), r = f2_pack(r0, r1), ns = f2_pack(-s0, -s1);
        uint64_t y0, e, y1;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y0) : "l"(v), "l"(r));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(ns), "l"(y0), "l"(v));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y1) : "l"(e), "l"(r), "l"(y0));
        y = f2_unpack(y1);
    } else {
        y = make_float2(__fdiv_rn(v0, s0), __fdiv_rn(v1, s1));
    }
    return (uint32_t)__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
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
    const uint32_t p0 = e4m3x2(v[0], v[1], s, s, r, r), p1 = e4m3x2(v[2], v[3], s, s, r, r);
    const uint32_t p2 = e4m3x2(v[4], v[5], s, s, r, r), p3 = e4m3x2(v[6], v[7], s, s, r, r);
    return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
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
                if (Xp) reinterpret_cast<uint4*>(Xp + (size_t)r * H)[v] = make_uint4(0, 0, 0, 0);
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
            if (Xp) reinterpret_cast<uint4*>(Xp + (size_t)rows[j] * H)[v] = u;
            reinterpret_cast<uint2*>(Xq + (size_t)rows[j] * H)[v] = c;
            if ((threadIdx.x & 15) == 0) sX[(size_t)rows[j] * nb + v / 16] = s;
        }
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
    // lanes 0-15 of a warp take 16 consecutive rows at one column half and
    // lanes 16-31 the same rows at the other, so that each 8-lane phase of a
    // 16-byte shared load meets 8 different bank groups (row stride 68 words)
    const int lane = threadIdx.x & 31;
    const int rr = (threadIdx.x >> 5) * 16 + (lane & 15), hf = lane >> 4;
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
            const int c = 4 * q4;
            if (sc_col) {   // 16-byte aligned per-column scales and reciprocals
                const float4 a = reinterpret_cast<const float4*>(sc_col + c0)[q4];
                const float4 r = reinterpret_cast<const float4*>(rc_col + c0)[q4];
                w[q4] = e4m3x2(f[c], f[c + 1], a.x, a.y, r.x, r.y) |
                        (e4m3x2(f[c + 2], f[c + 3], a.z, a.w, r.z, r.w) << 16);
            } else {
                w[q4] = e4m3x2(f[c], f[c + 1], sc, sc, rc, rc) | (e4m3x2(f[c + 2], f[c + 3], sc, sc, rc, rc) << 16);
            }
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

// One pass over a bf16 matrix in[rows][C] (rows and C multiples of 128) in
// 128x128 tiles; a persistent block stages each tile in shared memory and
// has the next tile's loads in flight while it encodes the current one. Outputs (template modes):
//   QM 1: row codes q[rows][C], one scale per row and 128 columns, s[rows][C/128]
//   QM 2: tile codes q[rows][C], one scale per tile, s[rows/128][C/128]
//   TM 1: transposed codes qT[C][rows_cap], one scale per column and 128 rows,
//         sT[C][rows_cap/128]
//   TM 2: transposed codes qT[C][rows_cap], one scale per tile, sT[C/128][rows_cap/128]
// Expert-stacked weights [E][R][C] with R a multiple of 128 are rows = E R.
// With a gather map, row r is token gather_slot[r] / gather_k of the input
// (the permuted rows of the layer input without their bf16 copy).
template <int QM, int TM>
__global__ void __launch_bounds__(256, (QM == 0 && TM == 1) ? 3 : 2)
quant_tiles_kernel(const __nv_bfloat16* __restrict__ in, const int* __restrict__ rows_dev,
                   int rows_fixed, int C, int rows_cap, uint8_t* __restrict__ q,
                   float* __restrict__ s, uint8_t* __restrict__ qT, float* __restrict__ sT,
                   const int* __restrict__ gslot, int gk)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    __shared__ __align__(16) uint8_t qs[TM ? 128 * kQS : 16];
    __shared__ float red[256];
    __shared__ __align__(16) float scol[128];
    __shared__ __align__(16) float rcol[128];
    __shared__ __align__(16) float colmax[TM == 1 ? 8 : 1][128];   // per warp, per tile column
    const int rows = rows_dev ? *rows_dev : rows_fixed;
    const int ncb = C / 128;
    const int ntiles = (rows / 128) * ncb;
    const int tid = threadIdx.x, sub = tid & 15;   // 16 threads per tile row, 8 columns each
    uint4 u[8];                                     // rows (tid / 16) + 16 j of the tile
    // With a gather map, row r of the tile is token gslot[r] / gk of `in`
    // (zeros for a pad row); the map entries of this thread's rows are read
    // one tile ahead of their data, so the data loads never wait on them.
    int sl[8];
    auto load_slots = [&](int t) {
        const int rb = t / ncb;
#pragma unroll
        for (int j = 0; j < 8; ++j) sl[j] = gslot[rb * 128 + (tid >> 4) + 16 * j];
    };
    auto fetch = [&](int t) {
        const int rb = t / ncb, cb = t - rb * ncb;
        if (gslot) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                u[j] = sl[j] >= 0 ? *reinterpret_cast<const uint4*>(in + (size_t)(sl[j] / gk) * C +
                                                                    (size_t)cb * 128 + sub * 8)
                                  : make_uint4(0, 0, 0, 0);
            if (t + (int)gridDim.x < ntiles) load_slots(t + gridDim.x);
        } else {
            const __nv_bfloat16* src = in + (size_t)rb * 128 * C + (size_t)cb * 128 + sub * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) u[j] = *reinterpret_cast<const uint4*>(src + (size_t)((tid >> 4) + 16 * j) * C);
        }
    };
    int t = blockIdx.x;
    if (gslot && t < ntiles) load_slots(t);
    if (t < ntiles) fetch(t);
    for (; t < ntiles; t += gridDim.x) {
        const int rb = t / ncb, cb = t - rb * ncb;
        const int r0 = rb * 128, c0 = cb * 128;
        // stage the tile, then put the next tile's loads in flight for the
        // whole of this tile's encoding
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(&tile[(tid >> 4) + 16 * j][sub * 8]) = u[j];
        if (TM == 1) {
            // per-column amax of this thread's 8 rows, then of the warp's 16
            // (lanes l and l ^ 16 hold the same columns), one partial per warp
            // (bf16 pairs: the largest magnitude of bf16 values is exact in bf16)
            __nv_bfloat162 cm[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cm[i] = __float2bfloat162_rn(0.f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) cm[i] = __hmax2(cm[i], __habs2(h[i]));
            }
            float cf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t bits = *reinterpret_cast<const uint32_t*>(&cm[i]);
                bits = __shfl_xor_sync(0xffffffffu, bits, 16);
                const __nv_bfloat162 other = *reinterpret_cast<const __nv_bfloat162*>(&bits);
                const float2 m = __bfloat1622float2(__hmax2(cm[i], other));
                cf[2 * i] = m.x;
                cf[2 * i + 1] = m.y;
            }
            if ((tid & 31) < 16) {
                float4* dst = reinterpret_cast<float4*>(&colmax[tid >> 5][sub * 8]);
                dst[0] = make_float4(cf[0], cf[1], cf[2], cf[3]);
                dst[1] = make_float4(cf[4], cf[5], cf[6], cf[7]);
            }
        }
        if (t + (int)gridDim.x < ntiles) fetch(t + gridDim.x);
        // row codes and amax from this thread's own staged values
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int rr = (tid >> 4) + 16 * j;
            float f[8];
            unpack8(*reinterpret_cast<const uint4*>(&tile[rr][sub * 8]), f);
            if (QM == 1) {
                const float ra = amax16(f);                 // the row's 128 values are on 16 lanes
                const float sr = block_scale(ra);
                *reinterpret_cast<uint2*>(q + (size_t)(r0 + rr) * C + c0 + sub * 8) = codes8(f, sr);
                if (sub == 0) s[(size_t)(r0 + rr) * ncb + cb] = sr;
                amax = fmaxf(amax, ra);                     // the tile's amax too (TM 2)
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            }
        }
        float st = 1.f;
        if (QM == 2 || TM == 2) st = block_scale(block_max(amax, red));   // also a barrier
        else __syncthreads();                                              // the tile is staged
        if (QM == 2) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int rr = (tid >> 4) + 16 * j;
                float f[8];
                unpack8(*reinterpret_cast<const uint4*>(&tile[rr][sub * 8]), f);
                *reinterpret_cast<uint2*>(q + (size_t)(r0 + rr) * C + c0 + sub * 8) = codes8(f, st);
            }
            if (tid == 0) s[(size_t)rb * ncb + cb] = st;
        }
        if (TM) {
            if (TM == 1) {
                // column amax from the eight warps' partials (written before
                // the barrier that follows the staging)
                if (tid < 128) {
                    float a = colmax[0][tid];
#pragma unroll
                    for (int w = 1; w < 8; ++w) a = fmaxf(a, colmax[w][tid]);
                    const float s1 = block_scale(a);
                    scol[tid] = s1;
                    rcol[tid] = __frcp_rn(s1);
                    sT[(size_t)(c0 + tid) * (rows_cap / 128) + rb] = s1;
                }
                __syncthreads();
            } else if (tid == 0) {
                sT[(size_t)cb * (rows_cap / 128) + rb] = st;
            }
            encode_rows(tile, st, TM == 1 ? scol : nullptr, rcol, qs, nullptr, 0);
            __syncthreads();
            write_transposed(qs, qT + (size_t)c0 * rows_cap + r0, rows_cap);
        }
        __syncthreads();   // shared buffers are free for the next tile
    }
}

template <int QM, int TM>
cudaError_t run_quant(const QuantJob& j, cudaStream_t st)
{
    // computed once (thread-safe initialisation of a function-local static)
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_tiles_kernel<QM, TM>, 256, 0) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = 1;
        }
        return n;
    }();
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const long long tiles = (long long)(j.rows_max / 128) * (j.C / 128);
    if (tiles <= 0) return cudaSuccess;
    const long long grid = tiles < (long long)sms * per_sm ? tiles : (long long)sms * per_sm;
    quant_tiles_kernel<QM, TM><<<(unsigned)grid, 256, 0, st>>>(j.in, j.rows_dev, j.rows_max, j.C,
                                                               j.rows_cap, j.q, j.s, j.qT, j.sT,
                                                               j.gather_slot, j.gather_k);
    count_launches();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute_quant(const __nv_bfloat16* x, const int* row_of, const int* poff,
                                 const int* counts, int T_, int H, int E, int k, __nv_bfloat16* Xp,
                                 uint8_t* Xq, float* sX, cudaStream_t s)
{
    permute_quant_kernel<<<T_ + E, 128, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xp, Xq, sX);
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_quant(const QuantJob& j, cudaStream_t s)
{
    if (j.C % 128 || j.rows_max % 128 || j.rows_cap % 128) return cudaErrorInvalidValue;
    const int qm = j.q ? (j.q_tiles ? 2 : 1) : 0;
    const int tm = j.qT ? (j.t_tiles ? 2 : 1) : 0;
    switch (qm * 3 + tm) {
    case 1: return run_quant<0, 1>(j, s);
    case 2: return run_quant<0, 2>(j, s);
    case 3: return run_quant<1, 0>(j, s);
    case 5: return run_quant<1, 2>(j, s);
    case 6: return run_quant<2, 0>(j, s);
    case 8: return run_quant<2, 2>(j, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
