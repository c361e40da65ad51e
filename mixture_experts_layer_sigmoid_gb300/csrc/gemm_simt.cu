// gemm_simt.cu -- fp32 grouped GEMM on the CUDA cores, for the MOE_FP32
// configuration (fp32 storage, fp32 FMA arithmetic; the tensor cores have no
// full-precision fp32 mode).
//
// Same problem description (GemmDesc) and epilogues as the bf16 tensor-core
// engine: "Expert Computation" of "Scalable Training of Mixture-of-Experts
// Models with Megatron Core", §2 (all experts' GEMMs in one launch over
// ragged per-expert row segments).
//
// Tile: 64 x 64 outputs per accumulator, K chunk 16, 256 threads with 4 x 4
// outputs each. Each output is owned by one thread and summed in a fixed
// order, so results are deterministic.
#include "internal.h"
#include "epilogue.cuh"

namespace moe {
namespace {

constexpr int BMs = 64, BNs = 64, BKs = 16;

template <int NACC>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const GemmDesc d)
{
    __shared__ float As[BKs][BMs + 4];
    __shared__ float Bs[NACC][BKs][BNs + 4];
    const float* A0 = static_cast<const float*>(d.A0);
    const float* A1 = static_cast<const float*>(d.A1);
    const float* B0 = static_cast<const float*>(d.B0);
    const float* B1 = static_cast<const float*>(d.B1);

    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int n0 = blockIdx.x * BNs;
    int e = 0, row0 = 0, m0 = 0, k_lo = 0, k_hi = 0, valid_end = 0, alloc_end = 0, Ktot = 0;
    if (d.sched == SCHED_ROWS) {
        row0 = blockIdx.y * BMs;
        if (d.dense_rows > 0) {
            if (row0 >= d.dense_rows) return;
            valid_end = alloc_end = d.dense_rows;
        } else {
            const int t128 = row0 / kTileM;
            if (t128 >= d.meta[0]) return;
            e = d.tile_tab[t128];
            valid_end = d.poff[e] + d.counts[e];
            alloc_end = d.poff[e + 1];
        }
        Ktot = (d.dual == DUAL_K) ? 2 * d.K : d.K;
    } else {
        m0 = blockIdx.y * BMs;
        e = blockIdx.z;
        if (d.dense_rows > 0) { k_lo = 0; k_hi = d.dense_rows; }
        else { k_lo = d.poff[e]; k_hi = d.poff[e] + d.counts[e]; }
        Ktot = k_hi - k_lo;
    }

    float acc[NACC][4][4];
#pragma unroll
    for (int a = 0; a < NACC; ++a)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[a][i][j] = 0.f;

    for (int kc = 0; kc < Ktot; kc += BKs) {
        // A tile -> As[kk][m]
        for (int idx = tid; idx < BMs * BKs; idx += 256) {
            float v = 0.f;
            if (d.sched == SCHED_ROWS) {
                const int m = idx / BKs, kk = idx % BKs;
                const int kg = kc + kk;
                const float* src = A0;
                int kl = kg;
                if (d.dual == DUAL_K && kg >= d.K) { src = A1; kl = kg - d.K; }
                const int r = row0 + m;
                if (r < d.a_rows) v = src[(size_t)r * d.lda + kl];
                As[kk][m] = v;
            } else {
                const int kk = idx / BMs, m = idx % BMs;
                const int r = k_lo + kc + kk;
                if (r < k_hi && m0 + m < d.M_out) v = A0[(size_t)r * d.lda + m0 + m];
                As[kk][m] = v;
            }
        }
        // B tile(s) -> Bs[a][kk][n]
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
            for (int idx = tid; idx < BKs * BNs; idx += 256) {
                float v = 0.f;
                int kk, n;
                if (d.sched == SCHED_ROWS && d.b_kmajor) { n = idx / BKs; kk = idx % BKs; }
                else { kk = idx / BNs; n = idx % BNs; }
                const int ng = n0 + n;
                if (ng < d.N) {
                    if (d.sched == SCHED_ROWS) {
                        const int kg = kc + kk;
                        const float* src = (NACC == 2 && a == 1) ? B1 : B0;
                        int kl = kg;
                        if (d.dual == DUAL_K && kg >= d.K) { src = B1; kl = kg - d.K; }
                        const float* base = src + (size_t)e * d.b_estride;
                        v = d.b_kmajor ? base[(size_t)ng * d.ldb + kl] : base[(size_t)kl * d.ldb + ng];
                    } else {
                        const float* src = (NACC == 2 && a == 1) ? B1 : B0;
                        const int r = k_lo + kc + kk;
                        if (r < k_hi) v = src[(size_t)r * d.ldb + ng];
                    }
                }
                Bs[a][kk][n] = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BKs; ++kk) {
            float av[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
                float bv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = Bs[a][kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[a][i][j] = fmaf(av[i], bv[j], acc[a][i][j]);
            }
        }
        __syncthreads();
    }

    float* O0 = static_cast<float*>(d.O0);
    float* O1 = static_cast<float*>(d.O1);
    float* O2 = static_cast<float*>(d.O2);
    const float* X0 = static_cast<const float*>(d.X0);
    const float* X1 = static_cast<const float*>(d.X1);
    const bool fold = d.gates != nullptr && d.sched == SCHED_ROWS;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // folded routing weight of this row; dg partial over this tile's 64 columns
        const int row_i = row0 + ty * 4 + i;
        const float grow = (fold && d.sched == SCHED_ROWS && row_i < valid_end) ? d.gates[d.slot_of[row_i]] : 1.f;
        float dgp = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = n0 + tx * 4 + j;
            if (col >= d.N) continue;
            if (d.sched == SCHED_WGRAD) {
                const int m = m0 + ty * 4 + i;
                if (m >= d.M_out) continue;
                const size_t o = (size_t)e * d.o_estride + (size_t)m * d.ldo + col;
                O0[o] = acc[0][i][j];
                if (NACC == 2) O1[o] = acc[NACC - 1][i][j];
                continue;
            }
            const int row = row0 + ty * 4 + i;
            if (row >= alloc_end) continue;
            const bool valid = row < valid_end;
            const size_t o = (size_t)row * d.ldo + col;
            if (d.epi == EPI_SWIGLU_FWD) {
                SwigluFwd r(acc[0][i][j], acc[NACC - 1][i][j]);
                O0[o] = valid ? r.a : 0.f;
                O1[o] = valid ? r.u : 0.f;
                O2[o] = valid ? r.h * grow : 0.f;
            } else if (d.epi == EPI_SWIGLU_BWD) {
                if (valid && fold) {
                    SwigluBwdFold r(acc[0][i][j], grow, X0[o], X1[o]);
                    O0[o] = r.dA;
                    O1[o] = r.dU;
                    dgp = fmaf(acc[0][i][j], r.h, dgp);
                    if (O2) O2[o] = r.h * grow;
                } else if (valid) {
                    SwigluBwd r(acc[0][i][j], X0[o], X1[o]);
                    O0[o] = r.dA;
                    O1[o] = r.dU;
                } else {
                    O0[o] = 0.f;
                    O1[o] = 0.f;
                    if (fold && O2) O2[o] = 0.f;
                }
            } else {
                O0[o] = valid ? acc[0][i][j] : 0.f;
            }
        }
        if (fold && d.epi == EPI_SWIGLU_BWD) {
            // the 16 threads of a half-warp (tx) share these rows
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) dgp += __shfl_xor_sync(0xffffffffu, dgp, off);
            if (tx == 0 && row_i < alloc_end) d.dg_part[(size_t)row_i * d.dg_ld + n0 / 64] = dgp;
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt_f32(const GemmDesc& d, int max_m_tiles, cudaStream_t s)
{
    dim3 grid((d.N + BNs - 1) / BNs, 1, 1);
    if (d.sched == SCHED_ROWS) {
        const int rows = d.dense_rows > 0 ? d.dense_rows : max_m_tiles * kTileM;
        grid.y = (rows + BMs - 1) / BMs;
    } else {
        grid.y = (d.M_out + BMs - 1) / BMs;
        grid.z = d.E;
    }
    if (grid.y == 0 || grid.z == 0) return cudaSuccess;
    if (d.dual == DUAL_N)
        gemm_simt_kernel<2><<<grid, 256, 0, s>>>(d);
    else
        gemm_simt_kernel<1><<<grid, 256, 0, s>>>(d);
    count_launches();
    return cudaGetLastError();
}

}  // namespace moe
