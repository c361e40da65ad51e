// gemm_tc.cu -- persistent grouped GEMM on the sm_103a tensor cores (bf16
// operands, fp32 accumulation) for every expert GEMM of the MoE layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §2
// ("Expert Computation": Grouped GEMM executes all local experts together)
// and §5 ("Kernel and shape optimization": expert activations padded with
// zero rows to aligned sizes, so every 128-row tile belongs to one expert).
//
// One CTA per SM, 6 warps:
//   warp 0     TMA producer: 128-byte-swizzled tiles of A and B into a ring
//              of shared-memory stages (mbarrier full/empty pairs);
//   warp 1     TMEM allocator and single-thread tcgen05.mma issuer; each
//              k block is 4 MMAs of 128 x BN x 16 into a TMEM accumulator;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//              output row), fused SwiGLU / SwiGLU-backward / store, 16-byte
//              global stores. Two TMEM accumulators let the epilogue of tile
//              i overlap the main loop of tile i+1.
// Tiles are enumerated identically by all three roles from device-side tables
// (tile -> expert, padded segment offsets), so the host never reads routing
// results and the launch is graph-capturable.
//
// Scheduling:
//   SCHED_ROWS  M = padded permuted rows (or a dense row range); fixed K.
//               fc1 (+SwiGLU), fc2, fc2 dgrad (+SwiGLU backward), fc1 dgrad.
//   SCHED_WGRAD per expert, output M_out x N, K = the expert's padded rows
//               (empty experts give zeros). Both operands are MN-major.
#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

constexpr int TBM = 128;       // MMA M
constexpr int TBK = 64;        // K block (128 bytes of bf16)
constexpr int STRIPE = 64 * 128;  // bytes of one 64-wide MN stripe of a 64-deep k block
constexpr int kThreads = 192;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kGroupN = 16;    // n tiles per raster group (row-scheduled GEMMs)

template <int BN>
struct TcCfg {
    static constexpr int A_BYTES = TBM * TBK * 2;
    static constexpr int B_BYTES = BN * TBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = kSmemBudget / STAGE;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM = 1024 + STAGES * STAGE + 256;
};

struct Tile {
    int e, m, n, row0, kblocks, valid_end, alloc_end;
};

template <int BN, int DUAL, int SCHED>
__device__ __forceinline__ void tile_counts(const GemmDesc& d, int& num_m, int& num_n, int& total)
{
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;   // output columns per tile
    if (SCHED == SCHED_ROWS) {
        num_m = d.dense_rows > 0 ? (d.dense_rows + TBM - 1) / TBM : d.meta[0];
        num_n = d.N / NW;
        total = num_m * num_n;
    } else {
        num_m = d.M_out / TBM;
        num_n = d.N / NW;
        total = d.E * num_m * num_n;
    }
}

template <int BN, int DUAL, int SCHED>
__device__ __forceinline__ Tile decode_tile(const GemmDesc& d, int w, int num_m, int num_n)
{
    Tile t;
    if (SCHED == SCHED_ROWS) {
        // Groups of kGroupN n-tiles: consecutive tiles share the A rows (one
        // 128-row tile against kGroupN weight column tiles), and consecutive
        // groups of them walk the m tiles, which share the expert's weights.
        const int group = w / (num_m * kGroupN);
        const int r = w - group * num_m * kGroupN;
        const int gsz = min(kGroupN, num_n - group * kGroupN);
        t.m = r / gsz;
        t.n = group * kGroupN + r % gsz;
        t.row0 = t.m * TBM;
        if (d.dense_rows > 0) {
            t.e = 0;
            t.valid_end = t.alloc_end = d.dense_rows;
        } else {
            t.e = d.tile_tab[t.m];
            t.valid_end = d.poff[t.e] + d.counts[t.e];
            t.alloc_end = d.poff[t.e + 1];
        }
        t.kblocks = ((DUAL == DUAL_K) ? 2 * d.K : d.K) / TBK;
    } else {
        const int per = num_m * num_n;
        t.e = w / per;
        const int r = w % per;
        t.m = r % num_m;
        t.n = r / num_m;
        if (d.dense_rows > 0) {
            t.row0 = 0;
            t.kblocks = (d.dense_rows + TBK - 1) / TBK;
        } else {
            t.row0 = d.poff[t.e];
            t.kblocks = (d.poff[t.e + 1] - d.poff[t.e]) / TBK;
        }
        t.valid_end = t.alloc_end = 0;
    }
    return t;
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float (&v)[32])
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
__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src, float (&v)[32])
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
__device__ __forceinline__ void zero32(float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
}
__device__ __forceinline__ void tmem_load32f(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    ptx::tmem_ld32(taddr, r);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int BN, bool B_MN, int DUAL, int EPI, int SCHED>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
               const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
               const GemmDesc d)
{
    using C = TcCfg<BN>;
    constexpr bool A_MN = (SCHED == SCHED_WGRAD);
    constexpr uint32_t IDESC = ptx::idesc_bf16<BN, A_MN, B_MN>();
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
    // bars: full[STAGES], empty[STAGES], accf[2], acce[2], final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t final_bar = bar0 + 8u * (2 * C::STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), 4);
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
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int num_m, num_n, total;
    tile_counts<BN, DUAL, SCHED>(d, num_m, num_n, total);

    // Each role runs its loop with the whole warp; lane 0 waits and issues, and
    // the wait's outcome is broadcast so the warp stays converged.
    auto wait_uniform = [&](uint32_t bar, uint32_t parity, int where) -> bool {
        int ok = 1;
        if (lane == 0) ok = ptx::wait_bounded(bar, parity, abort_flag, d.status, where) ? 1 : 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        uint32_t it = 0;
        const int kb_half = d.K / TBK;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
            const Tile t = decode_tile<BN, DUAL, SCHED>(d, w, num_m, num_n);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1u;
                if (!wait_uniform(empty_bar(s), ph ^ 1u, 1)) { ok = false; break; }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(full_bar(s), C::STAGE);
                    const uint32_t a_dst = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    if (SCHED == SCHED_ROWS) {
                        const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                        const int kx = (second ? kb - kb_half : kb) * TBK;
                        ptx::tma_load_2d(a_dst, second ? &mA1 : &mA0, full_bar(s), kx, t.row0);
                        if (B_MN) {
#pragma unroll
                            for (int s2 = 0; s2 < BN / 64; ++s2) {
                                const bool hi = (DUAL == DUAL_N) && s2 >= BN / 128;
                                const int x = (DUAL == DUAL_N) ? t.n * NW + 64 * (s2 % (BN / 128))
                                                               : t.n * NW + 64 * s2;
                                ptx::tma_load_2d(b_dst + s2 * STRIPE, hi ? &mB1 : &mB0, full_bar(s), x,
                                                 t.e * d.K + kb * TBK);
                            }
                        } else {
                            ptx::tma_load_2d(b_dst, second ? &mB1 : &mB0, full_bar(s), kx,
                                             t.e * d.N + t.n * NW);
                        }
                    } else {
                        const int krow = t.row0 + kb * TBK;
#pragma unroll
                        for (int s2 = 0; s2 < TBM / 64; ++s2)
                            ptx::tma_load_2d(a_dst + s2 * STRIPE, &mA0, full_bar(s), t.m * TBM + 64 * s2, krow);
#pragma unroll
                        for (int s2 = 0; s2 < BN / 64; ++s2) {
                            const bool hi = (DUAL == DUAL_N) && s2 >= BN / 128;
                            const int x = (DUAL == DUAL_N) ? t.n * NW + 64 * (s2 % (BN / 128))
                                                           : t.n * NW + 64 * s2;
                            ptx::tma_load_2d(b_dst + s2 * STRIPE, hi ? &mB1 : &mB0, full_bar(s), x, krow);
                        }
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        uint32_t it = 0, tc = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++tc) {
            const Tile t = decode_tile<BN, DUAL, SCHED>(d, w, num_m, num_n);
            const int a = tc & 1;
            const uint32_t aph = (tc >> 1) & 1u;
            if (!wait_uniform(acce_bar(a), aph ^ 1u, 2)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(a * BN);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1u;
                if (!wait_uniform(full_bar(s), ph, 3)) { ok = false; break; }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_addr = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < TBK / 16; ++k) {
                        const uint64_t ad = A_MN ? ptx::smem_desc_sw128(a_addr + k * 2048, STRIPE, 1024)
                                                 : ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
                        const uint64_t bd = B_MN ? ptx::smem_desc_sw128(b_addr + k * 2048, STRIPE, 1024)
                                                 : ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
                        ptx::tc_mma_f16(d_tmem, ad, bd, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(empty_bar(s));
                }
                __syncwarp();
            }
            if (ok && lane == 0) ptx::tc_commit(accf_bar(a));
            __syncwarp();
        }
        // every MMA issued by this warp has completed before TMEM is freed
        if (lane == 0) {
            ptx::tc_commit(final_bar);
            volatile int never = 0;
            ptx::wait_bounded(final_bar, 0, &never, d.status, 4);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int r_in = q * 32 + lane;         // row of the tile owned by this thread
        uint32_t tc = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++tc) {
            const Tile t = decode_tile<BN, DUAL, SCHED>(d, w, num_m, num_n);
            const int a = tc & 1;
            const uint32_t aph = (tc >> 1) & 1u;
            if (!wait_uniform(accf_bar(a), aph, 5)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN);
            float v0[32], v1[32];
            if (SCHED == SCHED_WGRAD) {
                const int m = t.m * TBM + r_in;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    if (t.kblocks > 0) tmem_load32f(taddr + c * 32, v0);
                    else zero32(v0);
                    int col, which = 0;
                    if (DUAL == DUAL_N) { which = c / (NW / 32); col = t.n * NW + (c % (NW / 32)) * 32; }
                    else col = t.n * NW + c * 32;
                    __nv_bfloat16* O = static_cast<__nv_bfloat16*>(which ? d.O1 : d.O0);
                    store32_bf16(O + (size_t)t.e * d.o_estride + (size_t)m * d.ldo + col, v0);
                }
            } else {
                const int row = t.row0 + r_in;
                const bool in_alloc = row < t.alloc_end;
                const bool valid = row < t.valid_end;
                if (EPI == EPI_SWIGLU_FWD) {
#pragma unroll 1
                    for (int c = 0; c < NW / 32; ++c) {
                        tmem_load32f(taddr + c * 32, v0);
                        tmem_load32f(taddr + NW + c * 32, v1);
                        if (in_alloc) {
                            float hv[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                if (valid) {
                                    SwigluFwd r(v0[i], v1[i]);
                                    v0[i] = r.a; v1[i] = r.u; hv[i] = r.h;
                                } else {
                                    v0[i] = 0.f; v1[i] = 0.f; hv[i] = 0.f;
                                }
                            }
                            const size_t o = (size_t)row * d.ldo + t.n * NW + c * 32;
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O0) + o, v0);
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O1) + o, v1);
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O2) + o, hv);
                        }
                    }
                } else if (EPI == EPI_SWIGLU_BWD) {
#pragma unroll 1
                    for (int c = 0; c < NW / 32; ++c) {
                        tmem_load32f(taddr + c * 32, v0);
                        if (in_alloc) {
                            const size_t o = (size_t)row * d.ldo + t.n * NW + c * 32;
                            if (valid) {
                                float av[32], uv[32];
                                load32_bf16(static_cast<const __nv_bfloat16*>(d.X0) + o, av);
                                load32_bf16(static_cast<const __nv_bfloat16*>(d.X1) + o, uv);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    SwigluBwd r(v0[i], av[i], uv[i]);
                                    v0[i] = r.dA; v1[i] = r.dU;
                                }
                            } else {
                                zero32(v0);
                                zero32(v1);
                            }
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O0) + o, v0);
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O1) + o, v1);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < NW / 32; ++c) {
                        tmem_load32f(taddr + c * 32, v0);
                        if (in_alloc) {
                            if (!valid) zero32(v0);
                            const size_t o = (size_t)row * d.ldo + t.n * NW + c * 32;
                            store32_bf16(static_cast<__nv_bfloat16*>(d.O0) + o, v0);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(a));
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Row-major bf16 matrix of `rows` x `cols` (row stride `ld` elements) read in
// boxes of box_rows x 64 with the 128-byte swizzle; out-of-bounds rows read 0.
bool make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
              int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool B_MN, int DUAL, int EPI, int SCHED>
cudaError_t set_attr()
{
    return cudaFuncSetAttribute(gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN>::SMEM);
}

template <int BN, bool B_MN, int DUAL, int EPI, int SCHED>
cudaError_t run(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;
    CUtensorMap mA0, mA1, mB0, mB1;
    bool ok = true;
    long long total;
    if (SCHED == SCHED_ROWS) {
        // A: [a_rows][K] read as 128-row boxes. B: per-expert blocks stacked.
        ok &= make_map(&mA0, d.A0, d.a_rows, d.K, d.lda, TBM);
        ok &= make_map(&mA1, d.A1 ? d.A1 : d.A0, d.a_rows, d.K, d.lda, TBM);
        if (B_MN) {   // B[e*K + k][n]
            ok &= make_map(&mB0, d.B0, d.b_rows, d.N, d.ldb, 64);
            ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, 64);
        } else {      // B[e*N + n][k]
            ok &= make_map(&mB0, d.B0, d.b_rows, d.K, d.ldb, BN);
            ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.K, d.ldb, BN);
        }
        const long long m_tiles = d.dense_rows > 0 ? (d.dense_rows + TBM - 1) / TBM : max_m_tiles;
        total = m_tiles * (d.N / NW);
    } else {
        // A: [rows][M_out], B: [rows][N], read as 64-row boxes of 64 columns.
        ok &= make_map(&mA0, d.A0, d.a_rows, d.M_out, d.lda, 64);
        mA1 = mA0;
        ok &= make_map(&mB0, d.B0, d.b_rows, DUAL == DUAL_N ? d.N : d.N, d.ldb, 64);
        ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, 64);
        total = (long long)d.E * (d.M_out / TBM) * (d.N / NW);
    }
    if (!ok) return cudaErrorInvalidValue;
    if (total <= 0) return cudaSuccess;
    const int grid = (int)(total < num_sms ? total : num_sms);
    gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED><<<grid, kThreads, TcCfg<BN>::SMEM, s>>>(mA0, mA1, mB0, mB1, d);
    return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_tc_prepare(int device)
{
    (void)device;
    if (!get_encode()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    acc(set_attr<256, true, DUAL_N, EPI_SWIGLU_FWD, SCHED_ROWS>());
    acc(set_attr<256, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>());
    acc(set_attr<128, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>());
    acc(set_attr<256, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>());
    acc(set_attr<128, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>());
    acc(set_attr<256, false, DUAL_K, EPI_STORE, SCHED_ROWS>());
    acc(set_attr<128, false, DUAL_K, EPI_STORE, SCHED_ROWS>());
    acc(set_attr<256, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>());
    acc(set_attr<128, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>());
    acc(set_attr<256, true, DUAL_N, EPI_WGRAD, SCHED_WGRAD>());
    return e;
}

cudaError_t launch_gemm_tc_bf16(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    if (!get_encode()) return cudaErrorNotSupported;
    const bool n256 = (d.N % 256) == 0;
    if (d.sched == SCHED_ROWS) {
        switch (d.epi) {
        case EPI_SWIGLU_FWD:
            return run<256, true, DUAL_N, EPI_SWIGLU_FWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            if (d.dual == DUAL_K)
                return n256 ? run<256, false, DUAL_K, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                            : run<128, false, DUAL_K, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
            return n256 ? run<256, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                        : run<128, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD:
            return n256 ? run<256, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                        : run<128, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (d.dual == DUAL_N) return run<256, true, DUAL_N, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s);
    return n256 ? run<256, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s)
                : run<128, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
