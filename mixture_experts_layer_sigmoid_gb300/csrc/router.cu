// router.cu -- Route stage and the dispatch tables of the MoE layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §2
// ("Route"): token hidden states -> expert logits -> probabilities -> the
// top-k experts, producing routing weights and a token-expert assignment.
// §5 ("Selective precision"): the router runs in FP32.
//
// Kernels:
//   router_small_kernel (E <= 32) and router_kernel (tiled, larger E):
//                  logits z = x Wr + b (fp32 FMA, fixed summation order),
//                  warp-shuffle top-k on z (score order equals logit order for
//                  both softmax and sigmoid; equal values go to the lower
//                  expert index), renormalised gates, and a per-block expert
//                  histogram counted without atomics.
//   scan_kernel    per-expert counts, segment sizes padded to 128 rows, their
//                  exclusive scan, per-block bases, the 128-row tile -> expert
//                  table and the pad-row markers.
//   index_kernel   row_of(t, j) = block base + rank of t among the block's
//                  tokens that chose the same expert (stable, token order),
//                  and its inverse slot_of.
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// Rows of each half of H per chunk of the tiled router (EPL experts per lane).
constexpr int router_chunk_rows(int epl) { return (2048 / (epl * 32)) < 16 ? 2048 / (epl * 32) : 16; }

// (value, index) ordering: larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Router replay: expert of slot j of token t from the caller, clamped into
// [0, E); an index outside it is reported once in the status word.
__device__ __forceinline__ int replay_expert(const int* replay, size_t i, int E, DeviceStatus* status)
{
    int e = replay[i];
    if (e < 0 || e >= E) {
        if (status && atomicCAS(&status->code, 0, (int)MOE_ERR_INVALID_ARG) == 0) status->where = 1;
        e = e < 0 ? 0 : E - 1;
    }
    return e;
}

// Gates of the selected logits: softmax over them (max-shifted), or the
// sigmoid scores over their sum.
__device__ __forceinline__ void gates_of(const float* sel_z, int k, int score, float* sc, float& den)
{
    float m = sel_z[0];
    for (int j = 1; j < k; ++j) m = fmaxf(m, sel_z[j]);
    den = 0.f;
    for (int j = 0; j < k; ++j) {
        sc[j] = (score == MOE_SCORE_SOFTMAX) ? expf(sel_z[j] - m) : 1.f / (1.f + expf(-sel_z[j]));
        den += sc[j];
    }
}

// Top-k of one token held by a warp (lane l has the logits of experts
// l + 32 i in z[i], -inf past E): k rounds of a warp-shuffle argmax, larger
// logit first and the lower expert index on equal values (score order equals
// logit order for softmax and sigmoid), or the replayed experts; lane 0
// writes the token's experts, gates and selected scores, and sel[0..k).
template <int EPL>
__device__ __forceinline__ void warp_route_token(const float (&z)[EPL], int t, int E, int k, int score,
                                                 const int* replay, DeviceStatus* status, int lane,
                                                 int* topk, float* gates, float* selsc, int* sel)
{
    unsigned taken = 0;
    int sel_e[kMaxK];
    float sel_z[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j >= k) break;
        if (replay) {
            // the given expert's logit, from the lane that holds it
            const int e = replay_expert(replay, (size_t)t * k + j, E, lane == 0 ? status : nullptr);
            float zi = z[0];
#pragma unroll
            for (int i = 1; i < EPL; ++i)
                if ((e >> 5) == i) zi = z[i];
            sel_e[j] = e;
            sel_z[j] = __shfl_sync(0xffffffffu, zi, e & 31);
            continue;
        }
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && better(z[i], e, bv, bi)) { bv = z[i]; bi = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        sel_e[j] = bi;
        sel_z[j] = bv;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
        float sc[kMaxK], den;
        gates_of(sel_z, k, score, sc, den);
        for (int j = 0; j < k; ++j) {
            topk[(size_t)t * k + j] = sel_e[j];
            gates[(size_t)t * k + j] = sc[j] / den;
            selsc[(size_t)t * k + j] = sc[j];
            sel[j] = sel_e[j];
        }
    }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Router for E > 32. A block routes kRouterTokens = 32 tokens: warps 0-3 sum
// the logits over the first half of H and warps 4-7 over the second half,
// and thread (warp w, lane l) accumulates tokens 8 (w % 4) .. +8 against
// experts l + 32 i (8 x EPL fp32 FMA chains, h ascending within a half).
// Chunks of HC rows of Wr per half arrive through a two-stage cp.async ring;
// x chunks are register-prefetched and staged transposed in fp32, so two
// 16-byte shared loads give a thread its 8 tokens' values of one h. The two
// halves are added in fixed order, then one warp per token selects the top k.
template <typename T, int EPL, bool SPLIT>
__global__ void __launch_bounds__(256, EPL <= 4 ? 3 : 2)
router_kernel(const T* __restrict__ x, const float* __restrict__ Wr, const float* __restrict__ b,
              int T_, int H, int E, int k, int score, int* __restrict__ topk,
              float* __restrict__ gates, float* __restrict__ selsc, int* __restrict__ hist,
              const int* __restrict__ replay, DeviceStatus* __restrict__ status,
              float* __restrict__ zpart)
{
    constexpr int EW = EPL * 32;                          // padded expert width
    constexpr int HC = router_chunk_rows(EPL);           // rows of H per half per chunk
    constexpr int TQ = 8;                                 // tokens per thread
    constexpr int V = 16 / sizeof(T);                     // x values per 16-byte load
    constexpr int XSEG = HC / V;                          // 16-byte pieces per token row per half
    constexpr int XPIECES = 2 * kRouterTokens * XSEG;     // <= 256
    static_assert(XPIECES <= 256 && HC % V == 0, "x staging");
    static_assert(4 * HC * EW >= kRouterTokens * EW, "partial sums reuse the Wr ring");
    __shared__ __align__(16) float ws[2][2][HC][EW];      // [stage][half][h][expert]
    __shared__ __align__(16) float xs[2][2][HC][kRouterTokens];   // [stage][half][h][token]
    __shared__ int sel_s[kRouterTokens][kMaxK];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = warp >> 2, tq0 = (warp & 3) * TQ;
    const int t0 = blockIdx.x * kRouterTokens;
    const int Hh = H / 2;                 // H is a multiple of 128
    // split blockIdx.y of gridDim.y takes the y-th of gridDim.y equal ranges
    // of chunks of both halves (the split count divides the chunk count) and
    // leaves its partial logits in zpart, for router_finish_kernel to route; a
    // grid of one split routes here
    const int nchunk = Hh / HC / (SPLIT ? (int)gridDim.y : 1);
    if (SPLIT) {
        Wr += (size_t)blockIdx.y * nchunk * HC * E;
        x += (size_t)blockIdx.y * nchunk * HC;
    }
    const int E4 = E / 4;
    const bool vec_w = (E & 3) == 0;      // Wr rows are 16-byte aligned

    // This thread's 16-byte pieces of a Wr chunk (at most 4: 2 HC EW / 4 <= 1024
    // pieces per chunk), as offsets from the chunk's first row; with E not a
    // multiple of 4 the chunk is copied in 4-byte pieces instead.
    constexpr int kMaxPieces = (2 * HC * EW / 4 + 255) / 256;
    int goff[kMaxPieces], soff[kMaxPieces];
    int npieces = 0;
    if (vec_w) {
#pragma unroll
        for (int j = 0; j < kMaxPieces; ++j) {
            const int i = tid + 256 * j;
            goff[j] = soff[j] = 0;
            if (i < 2 * HC * E4) {
                const int hf = i / (HC * E4), r = (i / E4) % HC, c4 = i % E4;
                goff[j] = (hf * Hh + r) * E + 4 * c4;
                soff[j] = (hf * HC + r) * EW + 4 * c4;
                npieces = j + 1;
            }
        }
    }
    auto issue_w = [&](int c, int st) {
        const float* src = Wr + (size_t)c * HC * E;
        float* dst = &ws[st][0][0][0];
        if (vec_w) {
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j)
                if (j < npieces) cp_async16(dst + soff[j], src + goff[j]);
        } else {
            for (int i = tid; i < 2 * HC * E; i += 256) {
                const int hf = i / (HC * E), r = (i / E) % HC, e = i % E;
                cp_async4(dst + (hf * HC + r) * EW + e, src + (size_t)(hf * Hh + r) * E + e);
            }
        }
        cp_async_commit();
    };
    // x piece of this thread: (half, token, segment) of chunk c
    const int xhf = tid / (kRouterTokens * XSEG), xtok = (tid / XSEG) % kRouterTokens, xseg = tid % XSEG;
    const bool xload = tid < XPIECES && t0 + xtok < T_;
    auto load_x = [&](int c, uint4& u) {
        if (xload)
            u = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + xtok) * H + xhf * Hh + c * HC + xseg * V);
        else
            u = make_uint4(0, 0, 0, 0);
    };
    auto store_x = [&](int st, const uint4& u) {
        if (tid < XPIECES) {
            const T* p = reinterpret_cast<const T*>(&u);
#pragma unroll
            for (int i = 0; i < V; ++i) xs[st][xhf][xseg * V + i][xtok] = to_f32(p[i]);
        }
    };

    float acc[TQ][EPL];
#pragma unroll
    for (int q = 0; q < TQ; ++q)
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[q][i] = 0.f;

    uint4 xr;
    issue_w(0, 0);
    load_x(0, xr);
    for (int c = 0; c < nchunk; ++c) {
        const int st = c & 1;
        store_x(st, xr);
        if (c + 1 < nchunk) {
            issue_w(c + 1, st ^ 1);
            load_x(c + 1, xr);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
#pragma unroll
        for (int hh = 0; hh < HC; ++hh) {
            float wv[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) wv[i] = ws[st][half][hh][lane + 32 * i];
            const float4 xa = *reinterpret_cast<const float4*>(&xs[st][half][hh][tq0]);
            const float4 xb = *reinterpret_cast<const float4*>(&xs[st][half][hh][tq0 + 4]);
            const float xv[TQ] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int q = 0; q < TQ; ++q)
#pragma unroll
                for (int i = 0; i < EPL; ++i) acc[q][i] = fmaf(xv[q], wv[i], acc[q][i]);
        }
        __syncthreads();
    }

    // second half's sums through shared memory (the Wr ring is free now)
    float* part = &ws[0][0][0][0];        // [token][EW]
    if (half == 1) {
#pragma unroll
        for (int q = 0; q < TQ; ++q)
#pragma unroll
            for (int i = 0; i < EPL; ++i) part[(tq0 + q) * EW + lane + 32 * i] = acc[q][i];
    }
    __syncthreads();
    if (SPLIT) {
        if (half == 0) {
            float* zp = zpart + (size_t)blockIdx.y * T_ * E;
#pragma unroll
            for (int q = 0; q < TQ; ++q) {
                const int tt = tq0 + q, t = t0 + tt;
                if (t >= T_) break;               // warp-uniform
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E) zp[(size_t)t * E + e] = acc[q][i] + part[tt * EW + e];
                }
            }
        }
        return;
    }
    if (half == 0) {
#pragma unroll
        for (int q = 0; q < TQ; ++q) {
            const int tt = tq0 + q, t = t0 + tt;
            if (t >= T_) break;                   // warp-uniform
            float z[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                z[i] = (e < E) ? (acc[q][i] + part[tt * EW + e]) + (b ? b[e] : 0.f) : -INFINITY;
            }
            warp_route_token<EPL>(z, t, E, k, score, replay, status, lane, topk, gates, selsc, sel_s[tt]);
        }
    }
    __syncthreads();
    const int ntok = min(kRouterTokens, T_ - t0);
    for (int e = tid; e < E; e += 256) {
        int cnt = 0;
        for (int tt = 0; tt < ntok; ++tt)
            for (int j = 0; j < k; ++j) cnt += (sel_s[tt][j] == e);
        hist[(size_t)blockIdx.x * E + e] = cnt;
    }
}

// Second pass of a split router: the logits of a token are its splits'
// partial sums added in split order, plus the bias; one warp routes each token
// (kRouterTokens / 8 per warp) and the block counts its tokens' experts like
// router_kernel.
template <int EPL>
__global__ void __launch_bounds__(256)
router_finish_kernel(const float* __restrict__ zpart, int S, const float* __restrict__ b, int T_, int E,
                     int k, int score, int* __restrict__ topk, float* __restrict__ gates,
                     float* __restrict__ selsc, int* __restrict__ hist, const int* __restrict__ replay,
                     DeviceStatus* __restrict__ status)
{
    constexpr int TPW = kRouterTokens / 8;
    __shared__ int sel_s[kRouterTokens][kMaxK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRouterTokens;
#pragma unroll 1
    for (int q = 0; q < TPW; ++q) {
        const int tt = warp * TPW + q, t = t0 + tt;
        if (t >= T_) break;                       // warp-uniform
        float z[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                float v = zpart[(size_t)t * E + e];
                for (int sp = 1; sp < S; ++sp) v += zpart[((size_t)sp * T_ + t) * E + e];
                z[i] = v + (b ? b[e] : 0.f);
            } else {
                z[i] = -INFINITY;
            }
        }
        warp_route_token<EPL>(z, t, E, k, score, replay, status, lane, topk, gates, selsc, sel_s[tt]);
    }
    __syncthreads();
    const int ntok = min(kRouterTokens, T_ - t0);
    for (int e = threadIdx.x; e < E; e += 256) {
        int cnt = 0;
        for (int tt = 0; tt < ntok; ++tt)
            for (int j = 0; j < k; ++j) cnt += (sel_s[tt][j] == e);
        hist[(size_t)blockIdx.x * E + e] = cnt;
    }
}

// Router for E <= 32. A block routes kRouterTokens tokens: lane l of every
// warp owns token l, warp w sums the logits of all experts over the w-th
// NW-th of H (16-byte x loads, four in flight; each Wr row is read once per
// warp as a broadcast), then one thread per token adds the NW partial sums in
// warp order, selects the top k (largest logit, lower expert index on
// equality) and writes the gates.
template <typename T, int EMAX>
__global__ void __launch_bounds__((EMAX <= 16 ? 16 : 8) * 32, 1)
router_small_kernel(const T* __restrict__ x, const float* __restrict__ Wr, const float* __restrict__ b,
                    int T_, int H, int E, int k, int score, int* __restrict__ topk,
                    float* __restrict__ gates, float* __restrict__ selsc, int* __restrict__ hist,
                    const int* __restrict__ replay, DeviceStatus* __restrict__ status)
{
    constexpr int V = 16 / sizeof(T);
    constexpr int NW = EMAX <= 16 ? 16 : 8;
    __shared__ float part[NW][kRouterTokens][EMAX + 1];
    __shared__ int sel_s[kRouterTokens][kMaxK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouterTokens + lane;
    float acc[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[e] = 0.f;
    const int hs = H / NW;                       // H is a multiple of 128
    const int h_lo = warp * hs;
    const int nv = hs / V;
    auto fma_vec = [&](const uint4& u, int h0) {
        const T* p = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const float xv = to_f32(p[i]);
            const float* wrow = Wr + (size_t)(h0 + i) * E;
#pragma unroll
            for (int e = 0; e < EMAX; ++e)
                if (e < E) acc[e] = fmaf(xv, __ldg(wrow + e), acc[e]);
        }
    };
    if (t < T_) {
        const T* xr = x + (size_t)t * H + h_lo;
        int v = 0;
        for (; v + 4 <= nv; v += 4) {
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) u[q] = *reinterpret_cast<const uint4*>(xr + (v + q) * V);
#pragma unroll
            for (int q = 0; q < 4; ++q) fma_vec(u[q], h_lo + (v + q) * V);
        }
        for (; v < nv; ++v) fma_vec(*reinterpret_cast<const uint4*>(xr + v * V), h_lo + v * V);
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) part[warp][lane][e] = acc[e];
    __syncthreads();
    if (threadIdx.x < kRouterTokens) {
        const int tt = threadIdx.x;
        const int tok = blockIdx.x * kRouterTokens + tt;
        if (tok < T_) {
            float z[EMAX];
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) v += part[w][tt][e];
                z[e] = (e < E) ? v + (b ? b[e] : 0.f) : -INFINITY;
            }
            unsigned taken = 0;
            int sel_e[kMaxK];
            float sel_z[kMaxK];
            for (int j = 0; j < k; ++j) {
                if (replay) {
                    const int e = replay_expert(replay, (size_t)tok * k + j, E, status);
                    float ze = z[0];
#pragma unroll
                    for (int i = 1; i < EMAX; ++i)
                        if (e == i) ze = z[i];
                    sel_e[j] = e;
                    sel_z[j] = ze;
                    continue;
                }
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int e = 0; e < EMAX; ++e)
                    if (e < E && !((taken >> e) & 1u) && better(z[e], e, bv, bi)) { bv = z[e]; bi = e; }
                taken |= 1u << bi;
                sel_e[j] = bi;
                sel_z[j] = bv;
            }
            float sc[kMaxK], den;
            gates_of(sel_z, k, score, sc, den);
            for (int j = 0; j < k; ++j) {
                topk[(size_t)tok * k + j] = sel_e[j];
                gates[(size_t)tok * k + j] = sc[j] / den;
                selsc[(size_t)tok * k + j] = sc[j];
                sel_s[tt][j] = sel_e[j];
            }
        }
    }
    __syncthreads();
    const int tb = blockIdx.x * kRouterTokens;
    const int ntok = min(kRouterTokens, T_ - tb);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int tt = 0; tt < ntok; ++tt)
            for (int j = 0; j < k; ++j) c += (sel_s[tt][j] == e);
        hist[(size_t)blockIdx.x * E + e] = c;
    }
}

// Four threads per expert (kScanParts); part p of expert e sums and bases
// router blocks [p nblk / 4, (p + 1) nblk / 4), the parts in block order.
constexpr int kScanParts = 4;

__global__ void __launch_bounds__(kScanParts * kMaxE)
scan_kernel(const int* __restrict__ hist, int nblk, int E, int* __restrict__ counts,
            int* __restrict__ poff, int* __restrict__ blkbase, int* __restrict__ tile_tab,
            int* __restrict__ meta, int* __restrict__ slot_of, int* __restrict__ pair_tab,
            int* __restrict__ pair_off, int cap, int* __restrict__ kept, int* __restrict__ eorder,
            int* __restrict__ full_tab, int* __restrict__ full_off, int* __restrict__ tail_tab)
{
    __shared__ int sc[kMaxE];
    __shared__ int plen[kMaxE];
    __shared__ int part_sum[kScanParts][kMaxE];
    const int e = threadIdx.x % kMaxE, part = threadIdx.x / kMaxE;
    const int b0 = (int)((long long)nblk * part / kScanParts);
    const int b1 = (int)((long long)nblk * (part + 1) / kScanParts);
    int cp = 0;
    if (e < E)
        for (int blk = b0; blk < b1; ++blk) cp += hist[(size_t)blk * E + e];
    part_sum[part][e] = cp;
    __syncthreads();
    int c = 0, before = 0;            // the expert's count; this part's rows before b0
#pragma unroll
    for (int q = 0; q < kScanParts; ++q) {
        if (q < part) before += part_sum[q][e];
        c += part_sum[q][e];
    }
    const int pc = (c + kTileM - 1) / kTileM * kTileM;
    if (part == 0) sc[e] = plen[e] = (e < E) ? pc : 0;
    __syncthreads();
    // inclusive Hillis-Steele scan over kMaxE entries (part 0 threads)
    for (int off = 1; off < kMaxE; off <<= 1) {
        int v = (part == 0 && e >= off) ? sc[e - off] : 0;
        __syncthreads();
        if (part == 0) sc[e] += v;
        __syncthreads();
    }
    const int start = sc[e] - ((e < E) ? pc : 0);
    if (e < E) {
        int run = start + before;
        for (int blk = b0; blk < b1; ++blk) {
            blkbase[(size_t)blk * E + e] = run;
            run += hist[(size_t)blk * E + e];
        }
        if (part == 0) {
            counts[e] = c;
            // capacity-limited dropping: the segment keeps all c rows (the router
            // gradient needs them) but only the first min(c, cap) are computed
            if (kept) kept[e] = (cap >= 0 && c > cap) ? cap : c;
            poff[e] = start;
            for (int i = 0; i < pc / kTileM; ++i) tile_tab[start / kTileM + i] = e;
            for (int r = start + c; r < start + pc; ++r) slot_of[r] = -1;
        }
    }
    const int total = sc[kMaxE - 1];
    if (threadIdx.x == 0) {
        poff[E] = total;
        meta[0] = total / kTileM;
        meta[1] = total;
    }
    if (pair_tab) {
        // pairs of consecutive tiles of one expert (the last one may be alone)
        const int np = (e < E) ? (pc / kTileM + 1) / 2 : 0;
        __syncthreads();
        if (part == 0) sc[e] = np;
        __syncthreads();
        for (int off = 1; off < kMaxE; off <<= 1) {
            int v = (part == 0 && e >= off) ? sc[e - off] : 0;
            __syncthreads();
            if (part == 0) sc[e] += v;
            __syncthreads();
        }
        if (part == 0) {
            const int pstart = sc[e] - np;
            for (int i = 0; i < np; ++i) pair_tab[pstart + i] = start / kTileM + 2 * i;
            if (e < E) pair_off[e] = pstart;   // first pair of expert e
        }
        if (threadIdx.x == 0) {
            meta[2] = sc[kMaxE - 1];
            pair_off[E] = sc[kMaxE - 1];
        }
    }
    if (full_tab) {
        // the pairs of the experts with two tiles or more (an odd last tile
        // beside a ghost, so that a second launch does not read the expert's
        // weights again); the experts of one tile are listed apart
        const int nt = (e < E) ? pc / kTileM : 0;
        const int nf = nt >= 2 ? (nt + 1) / 2 : 0, tl = nt == 1;
        int* tails = part_sum[1];            // free again: the counts are summed
        __syncthreads();
        if (part == 0) {
            sc[e] = nf;
            tails[e] = tl;
        }
        __syncthreads();
        for (int off = 1; off < kMaxE; off <<= 1) {
            int v = 0, u = 0;
            if (part == 0 && e >= off) {
                v = sc[e - off];
                u = tails[e - off];
            }
            __syncthreads();
            if (part == 0) {
                sc[e] += v;
                tails[e] += u;
            }
            __syncthreads();
        }
        if (part == 0) {
            const int fstart = sc[e] - nf;
            for (int i = 0; i < nf; ++i) full_tab[fstart + i] = start / kTileM + 2 * i;
            if (e < E) full_off[e] = fstart;
            if (tl) tail_tab[tails[e] - 1] = start / kTileM;
        }
        if (threadIdx.x == 0) {
            meta[3] = sc[kMaxE - 1];
            meta[4] = tails[kMaxE - 1];
            full_off[E] = sc[kMaxE - 1];
        }
    }
    // experts by padded segment length, longest first (lower index first on
    // equal lengths): the order the weight-gradient GEMMs take them in
    if (eorder && part == 0 && e < E) {
        const int len = plen[e];
        int rank = 0;
        for (int o = 0; o < E; ++o) rank += (plen[o] > len) || (plen[o] == len && o < e);
        eorder[rank] = e;
    }
}

__global__ void __launch_bounds__(256)
index_kernel(const int* __restrict__ topk, const int* __restrict__ blkbase, int T_, int E, int k,
             int* __restrict__ row_of, int* __restrict__ slot_of, const int* __restrict__ poff,
             const int* __restrict__ kept, int* __restrict__ slot_live)
{
    __shared__ int sel[kRouterTokens * kMaxK];
    const int t0 = blockIdx.x * kRouterTokens;
    const int ntok = min(kRouterTokens, T_ - t0);
    for (int i = threadIdx.x; i < ntok * k; i += blockDim.x) sel[i] = topk[(size_t)t0 * k + i];
    __syncthreads();
    for (int p = threadIdx.x; p < ntok * k; p += blockDim.x) {
        const int tt = p / k;
        const int e = sel[p];
        int rank = 0;
        for (int u = 0; u < tt; ++u)
            for (int j = 0; j < k; ++j) rank += (sel[u * k + j] == e);
        const int row = blkbase[(size_t)blockIdx.x * E + e] + rank;
        const int slot = (t0 + tt) * k + (p % k);
        row_of[slot] = row;
        slot_of[row] = slot;
        if (slot_live && row < poff[e] + kept[e]) slot_live[row] = slot;
    }
}

// H splits of the tiled router: the largest count up to kRouterSplitMax that
// divides the number of chunks in each half of H. It depends on H and E alone, so a
// token's logits (and hence its routing) do not depend on the batch it comes
// in, on the entry point, or on the GPU's SM count.
int router_split_count(int H, int E)
{
    if (E <= 32) return 1;
    const int epl = E <= 64 ? 2 : (E <= 128 ? 4 : 8);
    const int nchunk = (H / 2) / router_chunk_rows(epl);
    for (int S = kRouterSplitMax; S > 1; --S)
        if (nchunk % S == 0) return S;
    return 1;
}

template <typename T, int EPL>
cudaError_t run_router_tiled(const T* x, const float* Wr, const float* b, int T_, int H, int E, int k,
                             int score, int* topk, float* gates, float* selsc, int* hist,
                             cudaStream_t s, const int* replay, DeviceStatus* status, float* zpart,
                             size_t zpart_floats)
{
    const int nblk = (T_ + kRouterTokens - 1) / kRouterTokens;
    const int S = router_split_count(H, E);
    if (S > 1 && (!zpart || zpart_floats < (size_t)S * T_ * E)) return cudaErrorInvalidValue;
    if (S == 1) {
        router_kernel<T, EPL, false><<<nblk, 256, 0, s>>>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc,
                                                          hist, replay, status, nullptr);
        count_launches();
        return cudaGetLastError();
    }
    router_kernel<T, EPL, true><<<dim3(nblk, S), 256, 0, s>>>(x, Wr, b, T_, H, E, k, score, topk, gates,
                                                              selsc, hist, replay, status, zpart);
    router_finish_kernel<EPL><<<nblk, 256, 0, s>>>(zpart, S, b, T_, E, k, score, topk, gates, selsc, hist,
                                                   replay, status);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_router(const T* x, const float* Wr, const float* b, int T_, int H, int E, int k,
                          int score, int* topk, float* gates, float* selsc, int* hist,
                          cudaStream_t s,
                          const int* replay, DeviceStatus* status, float* zpart, size_t zpart_floats)
{
    const int nblk = (T_ + kRouterTokens - 1) / kRouterTokens;
    if (E <= 8)
        router_small_kernel<T, 8><<<nblk, 512, 0, s>>>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist,
                                                               replay, status);
    else if (E <= 16)
        router_small_kernel<T, 16><<<nblk, 512, 0, s>>>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist,
                                                               replay, status);
    else if (E <= 32)
        router_small_kernel<T, 32><<<nblk, 256, 0, s>>>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist,
                                                               replay, status);
    else if (E <= 64)
        return run_router_tiled<T, 2>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist, s, replay, status,
                                      zpart, zpart_floats);
    else if (E <= 128)
        return run_router_tiled<T, 4>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist, s, replay, status,
                                      zpart, zpart_floats);
    else
        return run_router_tiled<T, 8>(x, Wr, b, T_, H, E, k, score, topk, gates, selsc, hist, s, replay, status,
                                      zpart, zpart_floats);
    count_launches();
    return cudaGetLastError();
}
template cudaError_t launch_router<float>(const float*, const float*, const float*, int, int, int,
                                          int, int, int*, float*, float*, int*, cudaStream_t, const int*,
                                          DeviceStatus*, float*, size_t);
template cudaError_t launch_router<__nv_bfloat16>(const __nv_bfloat16*, const float*, const float*,
                                                  int, int, int, int, int, int*, float*, float*,
                                                  int*, cudaStream_t, const int*, DeviceStatus*, float*,
                                                  size_t);

size_t router_zpart_floats(int T, int H, int E)
{
    const int S = router_split_count(H, E);
    return S > 1 ? (size_t)S * T * E : 0;
}

cudaError_t launch_scan(const int* hist, int nblk, int E, int* counts, int* poff, int* blkbase,
                        int* tile_tab, int* meta, int* slot_of, cudaStream_t s, int* pair_tab,
                        int* pair_off, int cap, int* kept, int* eorder, int* full_tab,
                        int* full_off, int* tail_tab)
{
    if (pair_tab && !pair_off) return cudaErrorInvalidValue;
    if (full_tab && (!full_off || !tail_tab)) return cudaErrorInvalidValue;
    scan_kernel<<<1, kScanParts * kMaxE, 0, s>>>(hist, nblk, E, counts, poff, blkbase, tile_tab, meta,
                                                 slot_of, pair_tab, pair_off, cap, kept, eorder,
                                                 full_tab, full_off, tail_tab);
    count_launches();
    return cudaGetLastError();
}

cudaError_t launch_index(const int* topk, const int* blkbase, int T_, int E, int k, int* row_of,
                         int* slot_of, cudaStream_t s, const int* poff, const int* kept, int* slot_live)
{
    if (slot_live && (!poff || !kept)) return cudaErrorInvalidValue;
    const int nblk = (T_ + kRouterTokens - 1) / kRouterTokens;
    index_kernel<<<nblk, 256, 0, s>>>(topk, blkbase, T_, E, k, row_of, slot_of, poff, kept, slot_live);
    count_launches();
    return cudaGetLastError();
}

}  // namespace moe
