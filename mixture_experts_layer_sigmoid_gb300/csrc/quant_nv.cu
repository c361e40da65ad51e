// quant_nv.cu -- NVFP4 quantisers of the MOE_NVFP4 layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes: NVFP4 for Blackwell; Kernel and shape
// optimization: grouped quantisation ahead of the grouped NVFP4 GEMMs).
// Encoding: nv.cuh. A tensor, for the per-tensor fp32 scale, is one expert's
// part of a grouped operand (its segment of the permuted rows, or its weight
// matrix), or the whole of a dense operand; fc1's gate and up halves share
// one tensor scale (the caller runs the maximum pass over both into one
// array).
//
// Kernels:
//   nv_amax_kernel   the largest magnitude of each tensor: one 128 x 128
//                    tile per iteration, one atomicMax per tile (magnitudes
//                    are non-negative, so their bit patterns order like the
//                    values).
//   nv_tiles_kernel  [rows][C] bf16 in 128 x 128 tiles -> row codes (K runs
//                    along the rows) and/or transposed codes (K runs down
//                    the columns), each with its scale atoms.
//   nv_token_amax_kernel, nv_permute_kernel
//                    the permuted rows of x without gathering them twice:
//                    each expert's maximum is the largest row maximum of the
//                    tokens it keeps (one pass over x), then each token's row
//                    is read once and written as the row codes of its k
//                    permuted rows, each in its expert's tensor scale.
#include "internal.h"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {
namespace {

// tensor (scale segment) of the 128-row tile starting at row r0
__device__ __forceinline__ int nv_segment(const NvQuantJob& j, int r0)
{
    if (j.seg_off) {   // routed rows: the expert whose padded segment holds r0
        int lo = 0, hi = j.nseg - 1;
        while (lo < hi) {   // last e with seg_off[e] <= r0
            const int mid = (lo + hi + 1) >> 1;
            if (j.seg_off[mid] <= r0) lo = mid; else hi = mid - 1;
        }
        return lo;
    }
    return j.seg_rows > 0 ? r0 / j.seg_rows : 0;
}

// one 16-byte chunk (8 values from column c) of row r: gathered rows, zero
// rows past rows_valid
__device__ __forceinline__ uint4 nv_chunk(const NvQuantJob& j, int r, int c)
{
    if (j.gather_slot) {
        const int sl = j.gather_slot[r];
        return sl >= 0 ? *reinterpret_cast<const uint4*>(j.in + (size_t)(sl / j.gather_k) * j.C + c)
                       : make_uint4(0, 0, 0, 0);
    }
    if (j.rows_valid > 0 && r >= j.rows_valid) return make_uint4(0, 0, 0, 0);
    return *reinterpret_cast<const uint4*>(j.in + (size_t)r * j.C + c);
}

// Stage the 128 x 128 bf16 tile at (r0, c0) into shared memory (gathered
// rows, zero rows past rows_valid).
__device__ __forceinline__ void nv_stage(const NvQuantJob& j, __nv_bfloat16 (*tile)[136], int r0, int c0)
{
    const int tid = threadIdx.x;
    uint4 u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = nv_chunk(j, r0 + (tid >> 4) + 16 * i, c0 + (tid & 15) * 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(&tile[(tid >> 4) + 16 * i][(tid & 15) * 8]) = u[i];
}

__global__ void __launch_bounds__(256) nv_amax_kernel(const NvQuantJob j, float* __restrict__ amax)
{
    __shared__ float wmax[8];
    const int rows = j.rows_dev ? *j.rows_dev : j.rows_max;
    const int ncb = j.C / 128;
    const int ntiles = (rows / 128) * ncb;
    const int tid = threadIdx.x;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int rb = t / ncb, cb = t - rb * ncb;
        float a = 0.f;
        uint4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = nv_chunk(j, rb * 128 + (tid >> 4) + 16 * i, cb * 128 + (tid & 15) * 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(h[q]);
                a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if ((tid & 31) == 0) wmax[tid >> 5] = a;
        __syncthreads();
        if (tid == 0) {
            float m = wmax[0];
            for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
            atomicMax(reinterpret_cast<unsigned int*>(amax) + nv_segment(j, rb * 128), __float_as_uint(m));
        }
        __syncthreads();   // wmax is free for the next tile
    }
}

// One 128 x 128 tile per iteration of a persistent block (256 threads).
//   ROWQ: codes q[rows][C/2], 16-value blocks along each row (K = C); atoms
//         sf[(rb * C/64 + c0/64 + j/4) * 512], byte atom_byte(m, j % 4).
//   COLQ: transposed codes, 16-row blocks down each column (K = rows), per
//         group of grp rows: column c of group g -> qc[((g C + c) grp + r) / 2]
//         for the group's row r (activations: one group of rows_cap rows;
//         expert-stacked weights [E][grp][C]: group = expert); atoms of
//         operand row g C + c over K = grp.
template <bool ROWQ, bool COLQ>
__global__ void __launch_bounds__(256) nv_tiles_kernel(const NvQuantJob j)
{
    __shared__ __align__(16) __nv_bfloat16 tile[128][136];
    const int rows = j.rows_dev ? *j.rows_dev : j.rows_max;
    const int C = j.C;
    const int ncb = C / 128;
    const int ntiles = (rows / 128) * ncb;
    const int tid = threadIdx.x;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int rb = t / ncb, cb = t - rb * ncb;
        const int r0 = rb * 128, c0 = cb * 128;
        const float S = nv_tensor_scale(j.amax[nv_segment(j, r0)]);
        nv_stage(j, tile, r0, c0);
        __syncthreads();
        if (ROWQ) {
            // thread -> row m = tid / 2 and the four 16-column blocks of one
            // 64-column chunk (its 32 code bytes and the chunk's atom word)
            const int m = tid >> 1, ch = tid & 1;
            uint32_t w[8], sw = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jb = 4 * ch + q;
                float v[16];
                const uint4 u0 = *reinterpret_cast<const uint4*>(&tile[m][16 * jb]);
                const uint4 u1 = *reinterpret_cast<const uint4*>(&tile[m][16 * jb + 8]);
                const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u0);
                const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f0 = __bfloat1622float2(h0[i]), f1 = __bfloat1622float2(h1[i]);
                    v[2 * i] = f0.x; v[2 * i + 1] = f0.y;
                    v[8 + 2 * i] = f1.x; v[8 + 2 * i + 1] = f1.y;
                }
                uint2 c;
                sw |= nv_encode16(v, S, c) << (8 * q);
                w[2 * q] = c.x;
                w[2 * q + 1] = c.y;
            }
            uint4* dst = reinterpret_cast<uint4*>(j.q + ((size_t)(r0 + m) * C + c0 + 64 * ch) / 2);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            *reinterpret_cast<uint32_t*>(j.sf + ((size_t)rb * (C / 64) + c0 / 64 + ch) * 512 + atom_byte(m, 0)) = sw;
        }
        if (COLQ) {
            // thread -> column c = tid % 128 and the four 16-row blocks of one
            // 64-row chunk (32 code bytes of the transpose and the chunk's
            // atom word); a warp reads 32 consecutive columns
            const int grp = j.grp, g = r0 / grp, lr = r0 - g * grp;
            const int c = tid & 127, ch = tid >> 7;
            uint32_t w[8], sw = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jb = 4 * ch + q;
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __bfloat162float(tile[16 * jb + i][c]);
                uint2 code;
                sw |= nv_encode16(v, S, code) << (8 * q);
                w[2 * q] = code.x;
                w[2 * q + 1] = code.y;
            }
            uint4* dst = reinterpret_cast<uint4*>(j.qc + (((size_t)g * C + c0 + c) * grp + lr + 64 * ch) / 2);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            *reinterpret_cast<uint32_t*>(j.sfc + (((size_t)g * C + c0) / 128 * (grp / 64) + lr / 64 + ch) * 512 +
                                         atom_byte(c, 0)) = sw;
        }
        __syncthreads();   // the tile buffer is free for the next tile
    }
}

// One warp per token: the row's largest magnitude, folded into the maximum
// of each expert the token is kept by (row below the expert's kept count).
__global__ void __launch_bounds__(256)
nv_token_amax_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ topk,
                     const int* __restrict__ row_of, const int* __restrict__ poff, const int* __restrict__ kept,
                     int T_, int H, int k, float* __restrict__ amax)
{
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T_) return;
    float a = 0.f;
    for (int c = lane * 8; c < H; c += 256) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(h[q]);
            a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (lane < k) {
        const int e = topk[(size_t)t * k + lane];
        const int row = row_of[(size_t)t * k + lane];
        if (row < poff[e] + kept[e]) atomicMax(reinterpret_cast<unsigned int*>(amax) + e, __float_as_uint(a));
    }
}

// Blocks [0, T): token t -> the row codes of its k permuted rows (K = H):
// lane l of a warp takes the 16-value block l of a 512-value column span.
// Blocks [T, T+E): the pad rows of expert e (zero codes, scale bytes 0).
__global__ void __launch_bounds__(128)
nv_permute_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ topk,
                  const int* __restrict__ row_of, const int* __restrict__ poff, const int* __restrict__ counts,
                  const float* __restrict__ amax, int T_, int H, int k, uint8_t* __restrict__ Xq,
                  uint8_t* __restrict__ sfX)
{
    const int b = blockIdx.x;
    const int KA = H / 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (b >= T_) {
        const int e = b - T_;
        for (int r = poff[e] + counts[e]; r < poff[e + 1]; ++r) {
            for (int v = threadIdx.x; v < H / 32; v += blockDim.x)
                reinterpret_cast<uint4*>(Xq + (size_t)r * (H / 2))[v] = make_uint4(0, 0, 0, 0);
            for (int ch = threadIdx.x; ch < KA; ch += blockDim.x)
                *reinterpret_cast<uint32_t*>(sfX + ((size_t)(r >> 7) * KA + ch) * 512 + atom_byte(r & 127, 0)) = 0u;
        }
        return;
    }
    int rows[kMaxK];
    float S[kMaxK];
    for (int j = 0; j < k; ++j) {
        rows[j] = row_of[(size_t)b * k + j];
        S[j] = nv_tensor_scale(amax[topk[(size_t)b * k + j]]);
    }
    for (int c0 = 512 * warp; c0 < H; c0 += 512 * (blockDim.x / 32)) {
        const int col = c0 + 16 * lane;
        if (col >= H) break;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)b * H + col);
        const uint4 u0 = src[0], u1 = src[1];
        float v[16];
        const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u0);
        const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f0 = __bfloat1622float2(h0[i]), f1 = __bfloat1622float2(h1[i]);
            v[2 * i] = f0.x; v[2 * i + 1] = f0.y;
            v[8 + 2 * i] = f1.x; v[8 + 2 * i + 1] = f1.y;
        }
        for (int j = 0; j < k; ++j) {
            const int r = rows[j];
            uint2 c;
            const uint32_t sb = nv_encode16(v, S[j], c);
            *reinterpret_cast<uint2*>(Xq + ((size_t)r * H + col) / 2) = c;
            sfX[((size_t)(r >> 7) * KA + col / 64) * 512 + atom_byte(r & 127, (col & 63) >> 4)] = (uint8_t)sb;
        }
    }
}

int nv_grid(const NvQuantJob& j)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    const long long tiles = (long long)(j.rows_max / 128) * (j.C / 128);
    const long long cap = 4ll * sms;
    return (int)(tiles < cap ? tiles : cap);
}

bool nv_job_ok(const NvQuantJob& j)
{
    if (!j.in || j.C <= 0 || j.C % 128 || j.rows_max % 128 || j.rows_cap % 128) return false;
    if (j.seg_off && j.nseg < 1) return false;
    if (j.qc && (j.grp <= 0 || j.grp % 128 || j.rows_max % j.grp)) return false;
    return true;
}

}  // namespace

cudaError_t launch_nv_amax(const NvQuantJob& j, float* amax, cudaStream_t s)
{
    if (!nv_job_ok(j) || !amax) return cudaErrorInvalidValue;
    const int grid = nv_grid(j);
    if (grid < 0) return cudaErrorInvalidValue;
    if (grid == 0) return cudaSuccess;
    nv_amax_kernel<<<grid, 256, 0, s>>>(j, amax);
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_nv_permute(const __nv_bfloat16* x, const int* topk, const int* row_of, const int* poff,
                              const int* counts, const int* kept, int T_, int H, int E, int k, float* amax,
                              uint8_t* Xq, uint8_t* sfX, cudaStream_t s)
{
    if (H % 128 || k > kMaxK) return cudaErrorInvalidValue;
    if (T_ > 0) {
        nv_token_amax_kernel<<<(T_ + 7) / 8, 256, 0, s>>>(x, topk, row_of, poff, kept, T_, H, k, amax);
        count_launches();
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    nv_permute_kernel<<<T_ + E, 128, 0, s>>>(x, topk, row_of, poff, counts, amax, T_, H, k, Xq, sfX);
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_nv_quant(const NvQuantJob& j, cudaStream_t s)
{
    if (!nv_job_ok(j) || !j.amax || (!j.q && !j.qc) || (j.q && !j.sf) || (j.qc && !j.sfc))
        return cudaErrorInvalidValue;
    const int grid = nv_grid(j);
    if (grid < 0) return cudaErrorInvalidValue;
    if (grid == 0) return cudaSuccess;
    if (j.q && j.qc) nv_tiles_kernel<true, true><<<grid, 256, 0, s>>>(j);
    else if (j.q) nv_tiles_kernel<true, false><<<grid, 256, 0, s>>>(j);
    else nv_tiles_kernel<false, true><<<grid, 256, 0, s>>>(j);
    count_launches();
    return cudaGetLastError();
}

}  // namespace moe
