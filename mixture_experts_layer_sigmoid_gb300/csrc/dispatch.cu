// dispatch.cu -- memory-bound stages of the MoE layer: Dispatch (permute),
// Combine, and their backward counterparts.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §2:
// Dispatch "permutes tokens by destination expert"; Combine "restores
// sequence order" and "can add a shared expert's output". §5 ("Kernel and
// shape optimization"): expert activations are emitted zero-padded to aligned
// sizes, here 128-row segments. Every kernel moves whole rows with 16-byte
// vector loads and stores and sums in fp32 in a fixed slot order, so results
// are deterministic (no floating-point atomics).
#include "internal.h"

namespace moe {
namespace {

// 16-byte vectors of 4 fp32 or 8 bf16 values.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void unpack(const uint4& q, float (&v)[4]) {
        v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
        v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
    }
    __device__ static void load(const float* p, float (&v)[4]) {
        float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    __device__ static void store(float* p, const float (&v)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void unpack(const uint4& q, float (&v)[8]) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x; v[2 * i + 1] = f.y;
        }
    }
    __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
        unpack(*reinterpret_cast<const uint4*>(p), v);
    }
    __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint4 q;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = q;
    }
};

// The 16-byte vectors at column vector v of a token's k rows, all loads in
// flight together (slots past k untouched). KM >= k is a compile-time bound
// (2, 4 or 8), so the slot arrays stay in registers.
template <typename T, int KM>
__device__ __forceinline__ void load_rows(const T* __restrict__ base, const int (&rows)[KM], int k,
                                          int H, int v, uint4 (&raw)[KM])
{
#pragma unroll
    for (int j = 0; j < KM; ++j)
        if (j < k) raw[j] = *reinterpret_cast<const uint4*>(base + (size_t)rows[j] * H + v * Vec<T>::N);
}

// Slot bound of a launch: the smallest of 2, 4, 8 that holds k.
inline int slot_bound(int k) { return k <= 2 ? 2 : (k <= 4 ? 4 : 8); }

constexpr int kRowThreads = 128;

// Zero the pad rows [poff[e] + counts[e], poff[e+1]) of expert e.
template <typename T>
__device__ void zero_pad_rows(T* buf, int H, int e, const int* poff, const int* counts)
{
    const int r0 = poff[e] + counts[e], r1 = poff[e + 1];
    const size_t nvec = (size_t)(r1 - r0) * H * sizeof(T) / 16;
    uint4* p = reinterpret_cast<uint4*>(buf + (size_t)r0 * H);
    for (size_t i = threadIdx.x; i < nvec; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
}

// Blocks [0, T): copy x[t] to its k rows. Blocks [T, T+E): zero pad rows.
template <typename T, int KM>
__global__ void __launch_bounds__(kRowThreads)
permute_kernel(const T* __restrict__ x, const int* __restrict__ row_of, const int* __restrict__ poff,
               const int* __restrict__ counts, int T_, int H, int k, T* __restrict__ Xp,
               const int* __restrict__ slot_live)
{
    const int b = blockIdx.x;
    if (b >= T_) { zero_pad_rows(Xp, H, b - T_, poff, counts); return; }
    constexpr int V = 16 / sizeof(T);
    int rows[KM];
    bool live[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        rows[j] = j < k ? row_of[(size_t)b * k + j] : 0;
        live[j] = j < k && (!slot_live || slot_live[rows[j]] >= 0);   // dropped rows: zeros
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)b * H);
    for (int v = threadIdx.x; v < H / V; v += kRowThreads) {
        uint4 q = src[v];
#pragma unroll
        for (int j = 0; j < KM; ++j)
            if (j < k) reinterpret_cast<uint4*>(Xp + (size_t)rows[j] * H)[v] = live[j] ? q : make_uint4(0, 0, 0, 0);
    }
}

// y[t] = sum_j gates[t, j] Yp[row_of(t, j)] (+ Ys[t]), fp32, slot order.
template <typename T, int KM>
__global__ void __launch_bounds__(kRowThreads)
combine_kernel(const T* __restrict__ Yp, const T* __restrict__ Ys, const int* __restrict__ row_of,
               const float* __restrict__ gates, int H, int k, T* __restrict__ y)
{
    constexpr int V = Vec<T>::N;
    const int t = blockIdx.x;
    int rows[KM];
    float g[KM];
    // gates == null: the routing weights were folded into the expert
    // activations, so the expert outputs are already weighted
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        rows[j] = j < k ? row_of[(size_t)t * k + j] : 0;
        g[j] = (gates && j < k) ? gates[(size_t)t * k + j] : 1.f;
    }
    for (int v = threadIdx.x; v < H / V; v += kRowThreads) {
        float acc[V], in[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        uint4 raw[KM];
        load_rows<T, KM>(Yp, rows, k, H, v, raw);
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            Vec<T>::unpack(raw[j], in);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(g[j], in[i], acc[i]);
        }
        if (Ys) {
            Vec<T>::load(Ys + (size_t)t * H + v * V, in);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += in[i];
        }
        Vec<T>::store(y + (size_t)t * H + v * V, acc);
    }
}

// Router logit gradient of one token's k selected experts from dg:
//   softmax: dz_j = g_j (dg_j - sum_i g_i dg_i)
//   sigmoid: dz_j = s_j (1 - s_j) (dg_j - sum_i g_i dg_i) / sum_i s_i
__device__ __forceinline__ void router_dz(const float* dg, const float* g, const float* sel, int k,
                                          int score, float* dz)
{
    float gd = 0.f, ssum = 0.f;
    for (int j = 0; j < k; ++j) {
        gd += g[j] * dg[j];
        ssum += sel[j];
    }
    for (int j = 0; j < k; ++j) {
        if (score == MOE_SCORE_SOFTMAX) {
            dz[j] = g[j] * (dg[j] - gd);
        } else {
            const float s = sel[j];
            dz[j] = s * (1.f - s) * (dg[j] - gd) / ssum;
        }
    }
}

// Backward of Combine for token t (blocks [0, T)):
//   dg_j = <dY_t, Yp[row_j]>,  dYp[row_j] = g_j dY_t,
// then the router logit gradient of the k selected experts:
//   softmax: dz_j = g_j (dg_j - sum_i g_i dg_i)
//   sigmoid: dz_j = s_j (1 - s_j) (dg_j - sum_i g_i dg_i) / sum_i s_i
// Blocks [T, T+E) zero the pad rows of dYp.
template <typename T, int KM>
__global__ void __launch_bounds__(kRowThreads)
gate_grad_kernel(const T* __restrict__ dY, const T* __restrict__ Yp, const int* __restrict__ row_of,
                 const float* __restrict__ gates, const float* __restrict__ selsc,
                 const int* __restrict__ poff, const int* __restrict__ counts, int T_, int H, int k,
                 int score, T* __restrict__ dYp, float* __restrict__ dz, const int* __restrict__ slot_live)
{
    const int b = blockIdx.x;
    if (b >= T_) { zero_pad_rows(dYp, H, b - T_, poff, counts); return; }
    constexpr int V = Vec<T>::N;
    __shared__ float red[kRowThreads / 32][kMaxK];
    const int t = b;
    int rows[KM];
    float g[kMaxK], gs[KM], dot[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        dot[j] = 0.f;
        rows[j] = j < k ? row_of[(size_t)t * k + j] : 0;
        g[j] = j < k ? gates[(size_t)t * k + j] : 0.f;
        // the output-gradient scale of the row (0 for a dropped assignment)
        gs[j] = (j < k && slot_live && slot_live[rows[j]] < 0) ? 0.f : g[j];
    }
    for (int v = threadIdx.x; v < H / V; v += kRowThreads) {
        float dy[V], yp[V], o[V];
        Vec<T>::load(dY + (size_t)t * H + v * V, dy);
        uint4 raw[KM];
        load_rows<T, KM>(Yp, rows, k, H, v, raw);
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j >= k) break;
            Vec<T>::unpack(raw[j], yp);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) { s = fmaf(dy[i], yp[i], s); o[i] = gs[j] * dy[i]; }
            dot[j] += s;
            Vec<T>::store(dYp + (size_t)rows[j] * H + v * V, o);
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j >= k) break;
        float s = dot[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) red[warp][j] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float dg[kMaxK];
        for (int j = 0; j < k; ++j) {
            float s = 0.f;
            for (int w = 0; w < kRowThreads / 32; ++w) s += red[w][j];
            dg[j] = s;
        }
        router_dz(dg, g, selsc + (size_t)t * k, k, score, dz + (size_t)t * k);
    }
}

// Folded routing weights: dg of token t's slot j is the sum of the fc2-dgrad
// epilogue's partial dot products <dh', h> over the 64-column units of its
// row (fixed order: lane-strided sums, then a butterfly), then dz as above.
// One warp per token.
__global__ void __launch_bounds__(256)
gate_dz_kernel(const float* __restrict__ dg_part, int nslots, const int* __restrict__ row_of,
               const float* __restrict__ gates, const float* __restrict__ selsc, int T_, int k,
               int score, float* __restrict__ dz)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T_) return;
    float dg[kMaxK], g[kMaxK];
    for (int j = 0; j < k; ++j) {
        const float* pr = dg_part + (size_t)row_of[(size_t)t * k + j] * nslots;
        float s = 0.f;
        for (int q = lane; q < nslots; q += 32) s += pr[q];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        dg[j] = s;
        g[j] = gates[(size_t)t * k + j];
    }
    if (lane == 0) router_dz(dg, g, selsc + (size_t)t * k, k, score, dz + (size_t)t * k);
}

// dWr[h][e] = sum over expert e's rows r of Xp[r][h] dz[slot(r)], in two
// passes so that a hot expert's rows are spread over many blocks. Row r of
// Xp is token slot(r) / k of x, so the values are read from x itself (T H
// elements, mostly from L2, instead of the R H of Xp).
// Pass 1, block (128-row tile, 64 columns h): 256 threads = 32 row phases x
// 8 column groups of 8 columns (one 16-byte vector each); each phase sums
// rows ph, ph + 32, ph + 64, ph + 96 of the tile (pad rows, slot -1, add 0),
// and the 32 phases are added in fixed order into part[tile][h].
template <typename T>
__global__ void __launch_bounds__(256)
router_wgrad_tile_kernel(const T* __restrict__ x, const int* __restrict__ slot_of,
                         const int* __restrict__ meta, const float* __restrict__ dz, int H, int k,
                         float* __restrict__ part)
{
    constexpr int V = 16 / sizeof(T);            // columns per vector
    constexpr int CG = 64 / V;                   // column groups per block
    constexpr int PH = 256 / CG;                 // row phases
    constexpr int RPT = kTileM / PH;             // rows per thread
    __shared__ float red[PH][64 + 1];
    __shared__ float dzs[kTileM];
    __shared__ int toks[kTileM];
    const int tile = blockIdx.x;
    if (tile >= meta[0]) return;                 // block-uniform
    const int cg = threadIdx.x % CG, ph = threadIdx.x / CG;
    const int h0 = blockIdx.y * 64 + cg * V;
    const int r0 = tile * kTileM;
    if (threadIdx.x < kTileM) {
        const int slot = slot_of[r0 + threadIdx.x];
        dzs[threadIdx.x] = slot >= 0 ? dz[slot] : 0.f;
        toks[threadIdx.x] = slot >= 0 ? slot / k : -1;
    }
    __syncthreads();
    float xv[RPT][V];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int tok = toks[ph + PH * i];
        if (h0 < H && tok >= 0) {
            Vec<T>::load(x + (size_t)tok * H + h0, xv[i]);
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j) xv[i][j] = 0.f;
        }
    }
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float d = dzs[ph + PH * i];
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(xv[i][j], d, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < V; ++j) red[ph][cg * V + j] = acc[j];
    __syncthreads();
    if (threadIdx.x < 64) {
        const int h = blockIdx.y * 64 + threadIdx.x;
        float v = 0.f;
        for (int p2 = 0; p2 < PH; ++p2) v += red[p2][threadIdx.x];
        if (h < H) part[(size_t)tile * H + h] = v;
    }
}

// Pass 2: dWr[h][e] = sum of part[tile][h] over expert e's tiles, in tile
// order (0 for an empty expert).
__global__ void __launch_bounds__(256)
router_wgrad_sum_kernel(const float* __restrict__ part, const int* __restrict__ poff, int H, int E,
                        float* __restrict__ dWr)
{
    const int h = blockIdx.x * 256 + threadIdx.x, e = blockIdx.y;
    if (h >= H) return;
    const int a = poff[e] / kTileM, z = poff[e + 1] / kTileM;
    float v = 0.f;
    for (int tile = a; tile < z; ++tile) v += part[(size_t)tile * H + h];
    dWr[(size_t)h * E + e] = v;
}

__global__ void transpose_kernel(const float* __restrict__ in, int rows, int cols, float* __restrict__ out)
{
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
        int r = r0 + i, c = c0 + threadIdx.x;
        tile[i][threadIdx.x] = (r < rows && c < cols) ? in[(size_t)r * cols + c] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        int c = c0 + i, r = r0 + threadIdx.x;
        if (c < cols && r < rows) out[(size_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

// dX[t] = sum_j dXp[row_j] + sum_j dz_j WrT[e_j] (+ dXs[t]), fp32, slot order.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
unpermute_reduce_kernel(const T* __restrict__ dXp, const T* __restrict__ dXs,
                        const int* __restrict__ row_of, const int* __restrict__ topk,
                        const float* __restrict__ dz, const float* __restrict__ WrT, int H, int k,
                        T* __restrict__ dX)
{
    constexpr int V = Vec<T>::N;
    const int t = blockIdx.x;
    int rows[kMaxK], ex[kMaxK];
    float d[kMaxK];
    for (int j = 0; j < k; ++j) {
        rows[j] = row_of[(size_t)t * k + j];
        ex[j] = topk[(size_t)t * k + j];
        d[j] = dz[(size_t)t * k + j];
    }
    for (int v = threadIdx.x; v < H / V; v += kRowThreads) {
        float acc[V], in[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        for (int j = 0; j < k; ++j) {
            Vec<T>::load(dXp + (size_t)rows[j] * H + v * V, in);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += in[i];
        }
        for (int j = 0; j < k; ++j) {
            const float4* w = reinterpret_cast<const float4*>(WrT + (size_t)ex[j] * H + v * V);
#pragma unroll
            for (int i = 0; i < V / 4; ++i) {
                float4 q = w[i];
                acc[4 * i + 0] = fmaf(d[j], q.x, acc[4 * i + 0]);
                acc[4 * i + 1] = fmaf(d[j], q.y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(d[j], q.z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(d[j], q.w, acc[4 * i + 3]);
            }
        }
        if (dXs) {
            Vec<T>::load(dXs + (size_t)t * H + v * V, in);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += in[i];
        }
        Vec<T>::store(dX + (size_t)t * H + v * V, acc);
    }
}

}  // namespace

template <typename T>
cudaError_t launch_permute(const T* x, const int* row_of, const int* poff, const int* counts,
                           int T_, int H, int E, int k, T* Xp, cudaStream_t s, const int* slot_live)
{
    switch (slot_bound(k)) {
    case 2: permute_kernel<T, 2><<<T_ + E, kRowThreads, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xp, slot_live); break;
    case 4: permute_kernel<T, 4><<<T_ + E, kRowThreads, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xp, slot_live); break;
    default: permute_kernel<T, 8><<<T_ + E, kRowThreads, 0, s>>>(x, row_of, poff, counts, T_, H, k, Xp, slot_live); break;
    }
    count_launches();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine(const T* Yp, const T* Ys, const int* row_of, const float* gates,
                           int T_, int H, int k, T* y, cudaStream_t s)
{
    switch (slot_bound(k)) {
    case 2: combine_kernel<T, 2><<<T_, kRowThreads, 0, s>>>(Yp, Ys, row_of, gates, H, k, y); break;
    case 4: combine_kernel<T, 4><<<T_, kRowThreads, 0, s>>>(Yp, Ys, row_of, gates, H, k, y); break;
    default: combine_kernel<T, 8><<<T_, kRowThreads, 0, s>>>(Yp, Ys, row_of, gates, H, k, y); break;
    }
    count_launches();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_gate_grad(const T* dY, const T* Yp, const int* row_of, const int* topk,
                             const float* gates, const float* selsc, const int* poff,
                             const int* counts, int T_, int H, int E, int k, int score, T* dYp,
                             float* dz, cudaStream_t s, const int* slot_live)
{
    (void)topk;
    switch (slot_bound(k)) {
    case 2: gate_grad_kernel<T, 2><<<T_ + E, kRowThreads, 0, s>>>(dY, Yp, row_of, gates, selsc, poff, counts,
                                                       T_, H, k, score, dYp, dz, slot_live); break;
    case 4: gate_grad_kernel<T, 4><<<T_ + E, kRowThreads, 0, s>>>(dY, Yp, row_of, gates, selsc, poff, counts,
                                                       T_, H, k, score, dYp, dz, slot_live); break;
    default: gate_grad_kernel<T, 8><<<T_ + E, kRowThreads, 0, s>>>(dY, Yp, row_of, gates, selsc, poff, counts,
                                                       T_, H, k, score, dYp, dz, slot_live); break;
    }
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_gate_dz(const float* dg_part, int nslots, const int* row_of, const float* gates,
                           const float* selsc, int T_, int k, int score, float* dz, cudaStream_t s)
{
    gate_dz_kernel<<<(T_ + 7) / 8, 256, 0, s>>>(dg_part, nslots, row_of, gates, selsc, T_, k, score, dz);
    count_launches();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_router_wgrad(const T* x, const int* slot_of, const int* poff, const int* meta,
                                int MT_max, const float* dz, int H, int E, int k, float* part,
                                float* dWr, cudaStream_t s)
{
    if (MT_max > 0) {
        dim3 grid1(MT_max, (H + 63) / 64);
        router_wgrad_tile_kernel<T><<<grid1, 256, 0, s>>>(x, slot_of, meta, dz, H, k, part);
    }
    dim3 grid2((H + 255) / 256, E);
    router_wgrad_sum_kernel<<<grid2, 256, 0, s>>>(part, poff, H, E, dWr);
    count_launches(MT_max > 0 ? 2 : 1);
    return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* in, int rows, int cols, float* out, cudaStream_t s)
{
    dim3 grid((cols + 31) / 32, (rows + 31) / 32);
    transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(in, rows, cols, out);
    count_launches();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_unpermute_reduce(const T* dXp, const T* dXs, const int* row_of,
                                    const int* topk, const float* dz, const float* WrT, int T_,
                                    int H, int k, T* dX, cudaStream_t s)
{
    unpermute_reduce_kernel<T><<<T_, kRowThreads, 0, s>>>(dXp, dXs, row_of, topk, dz, WrT, H, k, dX);
    count_launches();
    return cudaGetLastError();
}

#define MOE_INST(T)                                                                              \
    template cudaError_t launch_permute<T>(const T*, const int*, const int*, const int*, int, int, \
                                           int, int, T*, cudaStream_t, const int*);              \
    template cudaError_t launch_combine<T>(const T*, const T*, const int*, const float*, int, int, \
                                           int, T*, cudaStream_t);                               \
    template cudaError_t launch_gate_grad<T>(const T*, const T*, const int*, const int*,         \
                                             const float*, const float*, const int*, const int*, \
                                             int, int, int, int, int, T*, float*, cudaStream_t, \
                                             const int*);                                        \
    template cudaError_t launch_router_wgrad<T>(const T*, const int*, const int*, const int*,    \
                                                int, const float*, int, int, int, float*,        \
                                                float*, cudaStream_t);                           \
    template cudaError_t launch_unpermute_reduce<T>(const T*, const T*, const int*, const int*,  \
                                                    const float*, const float*, int, int, int,   \
                                                    T*, cudaStream_t);
MOE_INST(float)
MOE_INST(__nv_bfloat16)
#undef MOE_INST

}  // namespace moe
