// gemm_fp8.cu -- persistent grouped GEMM on blockwise-scaled FP8 (E4M3)
// operands with fp32 accumulation, for the MOE_FP8_BLOCK layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): blockwise FP8 with 1x128 activation/gradient
// tiles and 128x128 weight blocks. In each GEMM C = A B the operand A
// (rows = output rows) carries one fp32 scale per row and 128-deep K block,
// B one per 128x128 block, so
//   C[r][n] = sum_kb sA[r][kb] sB[kb][n/128] (sum_{k in kb} qA[r][k] qB[k][n]).
// Both operands are stored K-major in E4M3.
//
// One CTA per SM, 6 warps: warp 0 TMA producer (stages of A 128x128 B and
// B 128x128 B, 128-byte swizzle); warp 1 TMEM allocator and single-thread
// issuer of tcgen05.mma.kind::f8f6f4 (4 x K=32 per k block) into one of two
// TMEM partial buffers; warps 2-5 promote each finished k block into fp32
// registers (one output row per thread, 128 columns) with its two scales and,
// at the end of the tile, run the fused epilogue from the registers.
#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

constexpr int QBM = 128, QBK = 128, QBN = 128;   // tile M, K block, MMA N
constexpr int kQThreads = 192;
constexpr int kQStage = QBM * QBK + QBN * QBK;    // 32 KB
constexpr int kQStages = 6;
constexpr int kQSmem = 1024 + kQStages * kQStage + 256;
constexpr int kQGroupN = 16;

// f8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D, K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int N, int M)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct QTile {
    int e, m, n, row0, kblocks, kb0, valid_end, alloc_end;
};

template <int DUAL, int SCHED>
__device__ __forceinline__ void qtile_counts(const GemmDesc& d, int& num_m, int& num_n, int& total)
{
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;
    num_n = d.N / NW;
    if (SCHED == SCHED_ROWS) {
        num_m = d.meta[0];
        total = num_m * num_n;
    } else {
        num_m = d.M_out / QBM;
        total = d.E * num_m * num_n;
    }
}

template <int DUAL, int SCHED>
__device__ __forceinline__ QTile qdecode(const GemmDesc& d, int w, int num_m, int num_n)
{
    QTile t;
    if (SCHED == SCHED_ROWS) {
        const int group = w / (num_m * kQGroupN);
        const int r = w - group * num_m * kQGroupN;
        const int gsz = min(kQGroupN, num_n - group * kQGroupN);
        t.m = r / gsz;
        t.n = group * kQGroupN + r % gsz;
        t.e = d.tile_tab[t.m];
        t.row0 = t.m * QBM;
        t.valid_end = d.poff[t.e] + d.counts[t.e];
        t.alloc_end = d.poff[t.e + 1];
        t.kblocks = ((DUAL == DUAL_K) ? 2 * d.K : d.K) / QBK;
        t.kb0 = 0;
    } else {
        const int per = num_m * num_n;
        t.e = w / per;
        const int r = w % per;
        t.m = r % num_m;
        t.n = r / num_m;
        t.row0 = d.poff[t.e];
        t.kb0 = t.row0 / QBK;
        t.kblocks = (d.poff[t.e + 1] - t.row0) / QBK;
        t.valid_end = t.alloc_end = 0;
    }
    return t;
}

__device__ __forceinline__ void st32(__nv_bfloat16* dst, const float* v)
{
    uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
        p[q] = u;
    }
}
__device__ __forceinline__ void ld32(const __nv_bfloat16* src, float* v)
{
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u = p[q];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[8 * q + 2 * i] = f.x;
            v[8 * q + 2 * i + 1] = f.y;
        }
    }
}

template <int EPI, int SCHED, int DUAL>
__global__ void __launch_bounds__(kQThreads, 1)
gemm_fp8_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
                const GemmDesc d)
{
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;
    constexpr uint32_t IDESC = idesc_e4m3(QBN, QBM);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQStages * kQStage);
    // full[S], empty[S], pfull[2], pempty[2], final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kQStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kQStages + s); };
    auto pfull_bar = [&](int b) { return bar0 + 8u * (2 * kQStages + b); };
    auto pempty_bar = [&](int b) { return bar0 + 8u * (2 * kQStages + 2 + b); };
    const uint32_t final_bar = bar0 + 8u * (2 * kQStages + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(pfull_bar(b), 1);
            ptx::mbar_init(pempty_bar(b), 4);
        }
        ptx::mbar_init(final_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&mA0);
        ptx::prefetch_tmap(&mB0);
        if (DUAL != DUAL_NONE) {
            ptx::prefetch_tmap(&mA1);
            ptx::prefetch_tmap(&mB1);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 2 * QBN);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int num_m, num_n, total;
    qtile_counts<DUAL, SCHED>(d, num_m, num_n, total);
    auto wait_uniform = [&](uint32_t bar, uint32_t parity, int where) -> bool {
        int ok = 1;
        if (lane == 0) ok = ptx::wait_bounded(bar, parity, abort_flag, d.status, where) ? 1 : 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        uint32_t it = 0;
        const int kb_half = d.K / QBK;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
            const QTile t = qdecode<DUAL, SCHED>(d, w, num_m, num_n);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % kQStages;
                const uint32_t ph = (it / kQStages) & 1u;
                if (!wait_uniform(empty_bar(s), ph ^ 1u, 11)) { ok = false; break; }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(full_bar(s), kQStage);
                    const uint32_t a_dst = ptx::smem_u32(smem + s * kQStage);
                    const uint32_t b_dst = a_dst + QBM * QBK;
                    if (SCHED == SCHED_ROWS) {
                        const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                        const int kx = (second ? kb - kb_half : kb) * QBK;
                        ptx::tma_load_2d(a_dst, second ? &mA1 : &mA0, full_bar(s), kx, t.row0);
                        if (DUAL == DUAL_N) {
                            ptx::tma_load_2d(b_dst, &mB0, full_bar(s), kx, t.e * d.N + t.n * NW);
                            ptx::tma_load_2d(b_dst + 64 * QBK, &mB1, full_bar(s), kx, t.e * d.N + t.n * NW);
                        } else {
                            ptx::tma_load_2d(b_dst, second ? &mB1 : &mB0, full_bar(s), kx,
                                             t.e * d.N + t.n * NW);
                        }
                    } else {
                        const int kx = (t.kb0 + kb) * QBK;
                        ptx::tma_load_2d(a_dst, &mA0, full_bar(s), kx, t.m * QBM);
                        if (DUAL == DUAL_N) {
                            ptx::tma_load_2d(b_dst, &mB0, full_bar(s), kx, t.n * NW);
                            ptx::tma_load_2d(b_dst + 64 * QBK, &mB1, full_bar(s), kx, t.n * NW);
                        } else {
                            ptx::tma_load_2d(b_dst, &mB0, full_bar(s), kx, t.n * NW);
                        }
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer
        uint32_t it = 0, pc = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
            const QTile t = qdecode<DUAL, SCHED>(d, w, num_m, num_n);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it, ++pc) {
                const int s = it % kQStages;
                const uint32_t ph = (it / kQStages) & 1u;
                const int pb = pc & 1;
                const uint32_t pph = (pc >> 1) & 1u;
                if (!wait_uniform(pempty_bar(pb), pph ^ 1u, 12)) { ok = false; break; }
                if (!wait_uniform(full_bar(s), ph, 13)) { ok = false; break; }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_addr = ptx::smem_u32(smem + s * kQStage);
                    const uint32_t b_addr = a_addr + QBM * QBK;
                    const uint32_t dt = tmem_base + (uint32_t)(pb * QBN);
#pragma unroll
                    for (int k = 0; k < QBK / 32; ++k)
                        mma_e4m3(dt, ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024),
                                 ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024), IDESC, k > 0 ? 1u : 0u);
                    ptx::tc_commit(empty_bar(s));
                    ptx::tc_commit(pfull_bar(pb));
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            ptx::tc_commit(final_bar);
            volatile int never = 0;
            ptx::wait_bounded(final_bar, 0, &never, d.status, 14);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- promotion + epilogue
        const int q = warp & 3;
        const int r_in = q * 32 + lane;
        uint32_t pc = 0;
        const int kb_half = d.K / QBK;
        for (int w = blockIdx.x; w < total; w += gridDim.x) {
            const QTile t = qdecode<DUAL, SCHED>(d, w, num_m, num_n);
            float acc[QBN];
#pragma unroll
            for (int j = 0; j < QBN; ++j) acc[j] = 0.f;
            const int arow = (SCHED == SCHED_ROWS) ? t.row0 + r_in : t.m * QBM + r_in;
            bool ok = true;
            for (int kb = 0; kb < t.kblocks; ++kb, ++pc) {
                // scales of this k block (A: per row; B: per 128-column block)
                float sa, sb0, sb1;
                if (SCHED == SCHED_ROWS) {
                    const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                    const int kk = second ? kb - kb_half : kb;
                    sa = (second ? d.SA1 : d.SA0)[(size_t)arow * d.lds_a + kk];
                    const int nb = (t.n * NW) / 128;
                    const size_t bi = ((size_t)t.e * (d.N / 128) + nb) * (d.K / 128) + kk;
                    sb0 = (second ? d.SB1 : d.SB0)[bi];
                    sb1 = (DUAL == DUAL_N) ? d.SB1[bi] : sb0;
                } else {
                    const int kg = t.kb0 + kb;
                    sa = d.SA0[(size_t)arow * d.lds_a + kg];
                    const int nb = (t.n * NW) / 128;
                    sb0 = d.SB0[(size_t)nb * d.lds_b + kg];
                    sb1 = (DUAL == DUAL_N) ? d.SB1[(size_t)nb * d.lds_b + kg] : sb0;
                }
                const int pb = pc & 1;
                const uint32_t pph = (pc >> 1) & 1u;
                if (!wait_uniform(pfull_bar(pb), pph, 15)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(pb * QBN);
#pragma unroll
                for (int c = 0; c < QBN / 32; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + c * 32, r);
                    ptx::tmem_ld_wait();
                    const float sc = sa * ((c * 32 < NW) ? sb0 : sb1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[c * 32 + i] = fmaf(__uint_as_float(r[i]), sc, acc[c * 32 + i]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(pempty_bar(pb));
            }
            if (!ok) break;
            // ---- epilogue from registers
            if (SCHED == SCHED_WGRAD) {
                const int m = t.m * QBM + r_in;
                if (DUAL == DUAL_N) {
                    __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + (size_t)t.e * d.o_estride + (size_t)m * d.ldo + t.n * NW;
                    __nv_bfloat16* O1 = static_cast<__nv_bfloat16*>(d.O1) + (size_t)t.e * d.o_estride + (size_t)m * d.ldo + t.n * NW;
                    st32(O0, acc); st32(O0 + 32, acc + 32);
                    st32(O1, acc + 64); st32(O1 + 32, acc + 96);
                } else {
                    __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + (size_t)t.e * d.o_estride + (size_t)m * d.ldo + t.n * NW;
#pragma unroll
                    for (int c = 0; c < 4; ++c) st32(O0 + 32 * c, acc + 32 * c);
                }
            } else {
                const int row = t.row0 + r_in;
                if (row < t.alloc_end) {
                    const bool valid = row < t.valid_end;
                    const size_t o = (size_t)row * d.ldo + t.n * NW;
                    if (EPI == EPI_SWIGLU_FWD) {
                        float a[64], u[64], hv[64];
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            if (valid) {
                                SwigluFwd r(acc[i], acc[64 + i]);
                                a[i] = r.a; u[i] = r.u; hv[i] = r.h;
                            } else {
                                a[i] = u[i] = hv[i] = 0.f;
                            }
                        }
                        __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + o;
                        __nv_bfloat16* O1 = static_cast<__nv_bfloat16*>(d.O1) + o;
                        __nv_bfloat16* O2 = static_cast<__nv_bfloat16*>(d.O2) + o;
                        st32(O0, a); st32(O0 + 32, a + 32);
                        st32(O1, u); st32(O1 + 32, u + 32);
                        st32(O2, hv); st32(O2 + 32, hv + 32);
                    } else if (EPI == EPI_SWIGLU_BWD) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float av[32], uv[32], da[32], du[32];
                            if (valid) {
                                ld32(static_cast<const __nv_bfloat16*>(d.X0) + o + 32 * c, av);
                                ld32(static_cast<const __nv_bfloat16*>(d.X1) + o + 32 * c, uv);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    SwigluBwd r(acc[32 * c + i], av[i], uv[i]);
                                    da[i] = r.dA; du[i] = r.dU;
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i) da[i] = du[i] = 0.f;
                            }
                            st32(static_cast<__nv_bfloat16*>(d.O0) + o + 32 * c, da);
                            st32(static_cast<__nv_bfloat16*>(d.O1) + o + 32 * c, du);
                        }
                    } else {
                        if (!valid) {
#pragma unroll
                            for (int j = 0; j < QBN; ++j) acc[j] = 0.f;
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) st32(static_cast<__nv_bfloat16*>(d.O0) + o + 32 * c, acc + 32 * c);
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, 2 * QBN);
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 g_enc8 = nullptr;
std::once_flag g_enc8_once;
bool enc8()
{
    std::call_once(g_enc8_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_enc8 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_enc8 != nullptr;
}

// Row-major byte matrix rows x cols (row stride ld bytes), boxes of
// box_rows x 128 bytes, 128-byte swizzle, out-of-bounds reads 0.
bool map8(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld, int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    return g_enc8(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int SCHED, int DUAL>
cudaError_t qrun(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;
    constexpr int BROWS = (DUAL == DUAL_N) ? 64 : QBN;
    CUtensorMap mA0, mA1, mB0, mB1;
    bool ok = true;
    long long units;
    if (SCHED == SCHED_ROWS) {
        ok &= map8(&mA0, d.A0, d.a_rows, d.K, d.lda, QBM);
        ok &= map8(&mA1, d.A1 ? d.A1 : d.A0, d.a_rows, d.K, d.lda, QBM);
        ok &= map8(&mB0, d.B0, d.b_rows, d.K, d.ldb, BROWS);
        ok &= map8(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.K, d.ldb, BROWS);
        units = (long long)max_m_tiles * (d.N / NW);
    } else {
        // A: [M_out][rows_cap], B: [N][rows_cap] (transposed operands)
        ok &= map8(&mA0, d.A0, d.M_out, d.rows_cap, d.lda, QBM);
        mA1 = mA0;
        ok &= map8(&mB0, d.B0, d.N, d.rows_cap, d.ldb, BROWS);
        ok &= map8(&mB1, d.B1 ? d.B1 : d.B0, d.N, d.rows_cap, d.ldb, BROWS);
        units = (long long)d.E * (d.M_out / QBM) * (d.N / NW);
    }
    if (!ok) return cudaErrorInvalidValue;
    if (units <= 0) return cudaSuccess;
    const int grid = (int)(units < num_sms ? units : num_sms);
    gemm_fp8_kernel<EPI, SCHED, DUAL><<<grid, kQThreads, kQSmem, s>>>(mA0, mA1, mB0, mB1, d);
    return cudaGetLastError();
}

template <int EPI, int SCHED, int DUAL>
cudaError_t qattr()
{
    return cudaFuncSetAttribute(gemm_fp8_kernel<EPI, SCHED, DUAL>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
}

}  // namespace

cudaError_t gemm_fp8_prepare(int device)
{
    (void)device;
    if (!enc8()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    acc(qattr<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N>());
    acc(qattr<EPI_STORE, SCHED_ROWS, DUAL_NONE>());
    acc(qattr<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE>());
    acc(qattr<EPI_STORE, SCHED_ROWS, DUAL_K>());
    acc(qattr<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE>());
    acc(qattr<EPI_WGRAD, SCHED_WGRAD, DUAL_N>());
    return e;
}

cudaError_t launch_gemm_fp8(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    if (!enc8()) return cudaErrorNotSupported;
    if (d.sched == SCHED_ROWS) {
        switch (d.epi) {
        case EPI_SWIGLU_FWD: return qrun<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD: return qrun<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            return d.dual == DUAL_K ? qrun<EPI_STORE, SCHED_ROWS, DUAL_K>(d, max_m_tiles, num_sms, s)
                                    : qrun<EPI_STORE, SCHED_ROWS, DUAL_NONE>(d, max_m_tiles, num_sms, s);
        default: return cudaErrorInvalidValue;
        }
    }
    return d.dual == DUAL_N ? qrun<EPI_WGRAD, SCHED_WGRAD, DUAL_N>(d, max_m_tiles, num_sms, s)
                            : qrun<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
