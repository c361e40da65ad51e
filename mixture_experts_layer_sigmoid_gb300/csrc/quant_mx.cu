// quant_mx.cu -- MXFP8 quantisers of the MOE_MXFP8 layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): MXFP8, the default FP8 recipe on Blackwell,
// with 1x32 granularity. Each block of 32 values along a GEMM's contraction
// dimension K shares a power-of-two scale 2^e, kept as an UE8M0 byte e + 127,
// with e the smallest integer such that amax <= 448 2^e (nothing saturates),
// clamped to [-127, 127] (e = -127 for an all-zero block); a value v is
// stored as the E4M3 code of v 2^-e (exact scaling, then round to nearest
// even). The tensor cores apply the scales inside the MMA
// (tcgen05.mma.kind::mxf8f6f4.block_scale), one per row of A / column of B
// and 32-deep K block.
//
// Scale layout ("scale atoms", what gemm_mx.cu copies into tensor memory):
// an operand read as [rows][K] (rows = the MMA's M or N index) keeps, for
// each 128-row tile rt and 128-deep K block kb, one 512-byte atom at
// (rt * K/128 + kb) * 512 whose byte 16 (m % 32) + 4 (m / 32) + j holds the
// scale of tile row m and 32-deep sub-block j.
//
// Kernels:
//   mx_permute_kernel  x -> the row codes of the permuted rows (K = H) and
//                      their scale atoms; pad rows get zero codes.
//   mx_tiles_kernel    [rows][C] bf16 in 128x128 tiles -> row codes (K runs
//                      along the rows) and/or column codes (K runs down the
//                      columns), the latter stored either transposed
//                      [C][rows_cap] (the weight-gradient operands) or in
//                      place [rows][C] (expert weights read MN-major), each
//                      with its scale atoms.
#include "internal.h"
#include "mx.cuh"

#include <cuda_fp8.h>

namespace moe {
namespace {

__device__ __forceinline__ void unpack8f(const uint4& u, float* v)
{
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// Blocks [0, T): token t -> row codes of its k permuted rows. Blocks
// [T, T+E): pad rows of expert e (zero codes, scale byte 0). One warp per
// 128-column block of the row: lane l takes columns 4l .. 4l+3, and eight
// lanes share a 32-column MX block.
__global__ void __launch_bounds__(128)
mx_permute_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ row_of,
                  const int* __restrict__ poff, const int* __restrict__ counts, int T_, int H, int k,
                  uint8_t* __restrict__ Xq, uint8_t* __restrict__ sfX)
{
    const int b = blockIdx.x;
    const int KB = H / 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (b >= T_) {
        const int e = b - T_;
        for (int r = poff[e] + counts[e]; r < poff[e + 1]; ++r) {
            for (int v = threadIdx.x; v < H / 16; v += blockDim.x)
                reinterpret_cast<uint4*>(Xq + (size_t)r * H)[v] = make_uint4(0, 0, 0, 0);
            for (int kb = threadIdx.x; kb < KB; kb += blockDim.x) {
                uint8_t* a = sfX + ((size_t)(r >> 7) * KB + kb) * 512;
                *reinterpret_cast<uint32_t*>(a + atom_byte(r & 127, 0)) = 0u;
            }
        }
        return;
    }
    int rows[kMaxK];
    for (int j = 0; j < k; ++j) rows[j] = row_of[(size_t)b * k + j];
    for (int kb = warp; kb < KB; kb += blockDim.x / 32) {
        const uint2 u = reinterpret_cast<const uint2*>(x + (size_t)b * H + kb * 128)[lane];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
        float a = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const int e = mx_exp(a);
        const float s = mx_inv(e);
        const uint32_t c = e4m3x4(f0.x * s, f0.y * s, f1.x * s, f1.y * s);
        for (int j = 0; j < k; ++j) {
            const int r = rows[j];
            reinterpret_cast<uint32_t*>(Xq + (size_t)r * H + kb * 128)[lane] = c;
            if ((lane & 7) == 0)
                sfX[((size_t)(r >> 7) * KB + kb) * 512 + atom_byte(r & 127, lane >> 3)] = (uint8_t)(e + 127);
        }
    }
}

// One 128x128 tile per iteration of a persistent block (256 threads).
//   ROWQ: codes q[rows][C], blocks of 32 along each row (K = C); atoms
//         sf[(rb * C/128 + cb) * 512].
//   COLQ 1: transposed codes qc[C][rows_cap], blocks of 32 down each column
//           (K = rows); atoms sfc[(cb * rows_cap/128 + rb) * 512].
//   COLQ 2: in-place codes qc[rows][C], blocks of 32 down each column of each
//           group of `grp` rows (expert-stacked weights [E][grp][C], read
//           MN-major with K = grp); atoms of operand row e C + c:
//           sfc[((e C + c0) / 128 * grp/128 + kb) * 512].
// With a gather map, row r of the input is token gslot[r] / gk of `in`
// (zeros where gslot[r] < 0); with rows_valid > 0, rows from rows_valid on
// read as zeros (a dense group of rows padded to a multiple of 128). Rows
// beyond *rows_dev (or rows_fixed) are not visited.
template <bool ROWQ, int COLQ>
__global__ void __launch_bounds__(256)
mx_tiles_kernel(const __nv_bfloat16* __restrict__ in, const int* __restrict__ rows_dev, int rows_fixed,
                int C, int rows_cap, int grp, uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                uint8_t* __restrict__ qc, uint8_t* __restrict__ sfc, const int* __restrict__ gslot, int gk,
                int rows_valid)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    const int rows = rows_dev ? *rows_dev : rows_fixed;
    const int ncb = C / 128;
    const int ntiles = (rows / 128) * ncb;
    const int tid = threadIdx.x;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int rb = t / ncb, cb = t - rb * ncb;
        const int r0 = rb * 128, c0 = cb * 128;
        // stage: thread -> 16-byte chunk (tid & 15) of rows (tid >> 4) + 16 i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = (tid >> 4) + 16 * i, ch = tid & 15;
            uint4 u;
            if (gslot) {
                const int sl = gslot[r0 + rr];
                u = sl >= 0 ? *reinterpret_cast<const uint4*>(in + (size_t)(sl / gk) * C + c0 + ch * 8)
                            : make_uint4(0, 0, 0, 0);
            } else if (rows_valid > 0 && r0 + rr >= rows_valid) {
                u = make_uint4(0, 0, 0, 0);   // padding rows of a dense group
            } else {
                u = *reinterpret_cast<const uint4*>(in + (size_t)(r0 + rr) * C + c0 + ch * 8);
            }
            *reinterpret_cast<uint4*>(&tile[rr][ch * 8]) = u;
        }
        __syncthreads();
        if (ROWQ) {
            // unit = (row m, 32-column block j): two per thread
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int unit = tid + 256 * p, m = unit >> 2, j = unit & 3;
                float v[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) unpack8f(*reinterpret_cast<const uint4*>(&tile[m][32 * j + 8 * c]), v + 8 * c);
                uint4 w0, w1;
                const int e = encode32(v, w0, w1);
                uint4* dst = reinterpret_cast<uint4*>(q + (size_t)(r0 + m) * C + c0 + 32 * j);
                dst[0] = w0;
                dst[1] = w1;
                sf[((size_t)rb * ncb + cb) * 512 + atom_byte(m, j)] = (uint8_t)(e + 127);
            }
        }
        if (COLQ) {
            // unit = (column c, 32-row block j): thread -> column tid & 127, blocks
            // (tid >> 7) and (tid >> 7) + 2; a warp reads 32 consecutive columns
            uint32_t cw[2][8];   // COLQ 2: the codes of both units, four rows per word
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int c = tid & 127, j = (tid >> 7) + 2 * p;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[32 * j + i][c]);
                float a = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
                const int e = mx_exp(a);
                const uint8_t eb = (uint8_t)(e + 127);
                if (COLQ == 1) {
                    uint4 w0, w1;
                    encode32(v, w0, w1);
                    uint4* dst = reinterpret_cast<uint4*>(qc + (size_t)(c0 + c) * rows_cap + r0 + 32 * j);
                    dst[0] = w0;
                    dst[1] = w1;
                    sfc[((size_t)cb * (rows_cap / 128) + rb) * 512 + atom_byte(c, j)] = eb;
                } else {
                    const float sc = mx_inv(e);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        cw[p][i] = e4m3x4(v[4 * i] * sc, v[4 * i + 1] * sc, v[4 * i + 2] * sc, v[4 * i + 3] * sc);
                    const int e_grp = r0 / grp, kb = (r0 % grp) / 128;
                    sfc[(((size_t)e_grp * C + c0) / 128 * (grp / 128) + kb) * 512 + atom_byte(c, j)] = eb;
                }
            }
            if (COLQ == 2) {
                // in-place codes: through shared memory (the tile buffer, now
                // read), then out in 16-byte row chunks
                constexpr int kCS = 144;                  // code row stride, bytes
                uint8_t* ct = reinterpret_cast<uint8_t*>(&tile[0][0]);
                __syncthreads();
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int c = tid & 127, j = (tid >> 7) + 2 * p;
#pragma unroll
                    for (int i = 0; i < 32; ++i) ct[(32 * j + i) * kCS + c] = (uint8_t)(cw[p][i >> 2] >> (8 * (i & 3)));
                }
                __syncthreads();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int idx = tid + 256 * q4, row = idx >> 3, ch = idx & 7;
                    *reinterpret_cast<uint4*>(qc + (size_t)(r0 + row) * C + c0 + 16 * ch) =
                        *reinterpret_cast<const uint4*>(ct + row * kCS + 16 * ch);
                }
            }
        }
        __syncthreads();   // the tile buffer is free for the next tile
    }
}

template <bool ROWQ, int COLQ>
cudaError_t run_mx(const MxQuantJob& j, cudaStream_t st)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const long long tiles = (long long)(j.rows_max / 128) * (j.C / 128);
    if (tiles <= 0) return cudaSuccess;
    const long long cap = 4ll * sms;
    const long long grid = tiles < cap ? tiles : cap;
    mx_tiles_kernel<ROWQ, COLQ><<<(unsigned)grid, 256, 0, st>>>(j.in, j.rows_dev, j.rows_max, j.C, j.rows_cap,
                                                              j.grp, j.q, j.sf, j.qc, j.sfc, j.gather_slot,
                                                              j.gather_k, j.rows_valid);
    count_launches();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_permute(const __nv_bfloat16* x, const int* row_of, const int* poff, const int* counts,
                              int T_, int H, int E, int k, uint8_t* Xq, uint8_t* sfX, cudaStream_t s)
{
    if (H % 128) return cudaErrorInvalidValue;
    mx_permute_kernel<<<T_ + E, 128, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xq, sfX);
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_mx_quant(const MxQuantJob& j, cudaStream_t s)
{
    if (j.C % 128 || j.rows_max % 128 || j.rows_cap % 128 || (j.col_mode == 2 && (j.grp <= 0 || j.grp % 128)))
        return cudaErrorInvalidValue;
    const bool rq = j.q != nullptr;
    const int cq = j.qc ? j.col_mode : 0;
    if (rq && cq == 0) return run_mx<true, 0>(j, s);
    if (rq && cq == 1) return run_mx<true, 1>(j, s);
    if (rq && cq == 2) return run_mx<true, 2>(j, s);
    if (!rq && cq == 1) return run_mx<false, 1>(j, s);
    if (!rq && cq == 2) return run_mx<false, 2>(j, s);
    return cudaErrorInvalidValue;
}

}  // namespace moe
