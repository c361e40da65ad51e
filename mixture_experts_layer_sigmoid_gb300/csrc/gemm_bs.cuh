// gemm_bs.cuh -- persistent grouped GEMM on block-scaled operands: MXFP8 (E4M3 values, one
// UE8M0 power-of-two scale per 32 consecutive values along K, for both A and
// B) with fp32 accumulation, for the MOE_MXFP8 layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): MXFP8, the default FP8 recipe on Blackwell,
// with 1x32 granularity. The tensor cores apply the scales inside the MMA
// (tcgen05.mma.kind::mxf8f6f4.block_scale): each MMA of K = 32 multiplies
// the products of row m of A and column n of B by 2^(eA[m] + eB[n]) before
// accumulating, so the whole K loop accumulates in tensor memory, with no
// per-block promotion in registers (the blockwise-FP8 engine's limit).
//
// Ten warps per CTA: warp 0 loads each 128-deep k block (A: 128 rows x 128
// bytes, B: 256 rows, 128-byte swizzle; the operands' scale atoms, 512 bytes
// each, as 4 x 128-byte boxes; all by TMA); warp 1 allocates tensor memory and one
// thread issues, per k block, tcgen05.cp of the scale atoms into a ring of
// tensor-memory columns and four N = 256 MMAs (K = 32 each, the scale
// sub-block chosen by the instruction descriptor's scale-factor IDs);
// warps 2-9 wait for a finished tile, copy its 128 x 256 fp32 accumulator
// into registers (two warps per TMEM lane quarter, 128 columns each), release
// it to the next tile and run the fused epilogue from registers.
//
// CTA pairs (clusters of two, the default wherever the row units come in
// pairs): the even CTA issues M = 256 MMAs (cta_group::2) with A rows 0-127
// from its own shared memory and 128-255 from its peer's and B's 256 columns
// split between the two, so each SM loads 32 KB + 1.5 KB per k block instead
// of 48 KB + 1.5 KB; every CTA stages its own A scale atom and both B atoms,
// and tcgen05.cp.cta_group::2 moves each CTA's atoms into its own tensor
// memory, where its 128 rows of the accumulator live.
//
// Scale atoms (quant_mx.cu): an operand read as [rows][K] keeps, per 128-row
// tile and 128-deep K block, 512 bytes whose byte 16 (m % 32) + 4 (m / 32) + j
// is the scale of tile row m and 32-deep sub-block j. tcgen05.cp.32x128b.warpx4
// puts the atom's 32 rows of 16 bytes into every TMEM lane quarter, four
// 32-bit columns each: lane 32 q + r, column c + j holds the scales of rows
// r + 32 j, one byte per sub-block.
//
// NVFP4 operands (the NV template argument; gemm_nv.cu): E2M1 values packed
// two per byte, one unsigned E4M3 scale per 16 values along K
// (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X, K = 64 per MMA),
// always K-major. A k block is the same 128 bytes of each row (256 values,
// four MMAs); every MMA takes its own scale atoms, copied to its own tensor
// memory columns, and the epilogue divides the accumulator by the two
// operands' fp32 tensor scales (nv.cuh). Instantiated once per format:
// gemm_mx.cu (MXFP8) and gemm_nv.cu (NVFP4).
#pragma once
#include "internal.h"
#include "epilogue.cuh"
#include "mx.cuh"
#include "nv.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

constexpr int XBM = 128, XBK = 128, XBN = 256;   // rows per CTA, K block (bytes), MMA N
constexpr int kXThreads = 320;
constexpr int kXSmemMax = 232448;
constexpr int kXGroupN = 16;
constexpr int kAccCols = 256;                    // the accumulator

// STG: bytes of epilogue staging for TMA stores (8 warps x one 32-row x
// 128-byte buffer, which leaves the CTA-pair engine a fifth operand stage;
// two per warp for the SwiGLU backward, whose dA and dU leave together)
//
// NV: NVFP4 operands. A k block is still 128 bytes of each row (256 E2M1
// values, four MMAs of K = 64), and each MMA takes its own scale atoms (one
// per 16-value sub-block, .scale_vec::4X): 4 A atoms and 2 x 4 B atoms per
// stage, 48 tensor-memory columns.
template <bool PAIR, int STG = 0, bool NV = false>
struct XCfg {
    static constexpr int A_BYTES = XBM * XBK;
    static constexpr int B_ROWS = PAIR ? XBN / 2 : XBN;  // B rows (n) staged by this CTA
    static constexpr int B_BYTES = B_ROWS * XBK;
    // A atom(s), then the B atoms of the two 128-column parts
    static constexpr int SF_BYTES = (NV ? 12 : 3) * 512;
    static constexpr int SF_REGION = NV ? 6144 : 2048;   // (padded to keep 1 KB alignment)
    static constexpr int SF_COLS = NV ? 48 : 12;         // tensor-memory scale columns per stage
    static constexpr int STAGE = A_BYTES + B_BYTES + SF_REGION;
    static constexpr int STAGES = (kXSmemMax - 1024 - 256 - STG) / STAGE;
    static constexpr int SMEM = 1024 + STAGES * STAGE + STG + 256;
};
constexpr int kStoreStaging = 8 * 4096;
// every epilogue stores through staging
template <int EPI, int SCHED>
constexpr int staging_bytes()
{
    return EPI == EPI_SWIGLU_BWD ? 2 * kStoreStaging
                                 : (SCHED == SCHED_WGRAD || SCHED == SCHED_ROWS) ? kStoreStaging : 0;
}
static_assert(kAccCols + XCfg<true>::SF_COLS * XCfg<true>::STAGES <= 512, "tensor memory");
static_assert(kAccCols + XCfg<false>::SF_COLS * XCfg<false>::STAGES <= 512, "tensor memory");
static_assert(kAccCols + XCfg<true, 0, true>::SF_COLS * XCfg<true, 0, true>::STAGES <= 512, "tensor memory");
static_assert(kAccCols + XCfg<false, 0, true>::SF_COLS * XCfg<false, 0, true>::STAGES <= 512, "tensor memory");

// kind::mxf8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D,
// UE8M0 scales (bit 23), A K-major, B K-major or MN-major (bit 16), the
// scale-factor IDs of A (bits 29-30) and B (bits 4-5) select the byte of
// each 32-bit scale column (the 32-deep sub-block).
__host__ __device__ constexpr uint32_t idesc_mx(int N, int M, bool b_mn, int sf_id)
{
    return ((uint32_t)sf_id << 4) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// kind::mxf4nvf4 instruction descriptor: E2M1 A and B (format 1 in bits 7-9
// and 10-12), fp32 D, UE4M3 scales (bit 23 clear), both K-major; with
// .scale_vec::4X each 32-bit scale column holds the four 16-value sub-blocks
// of one MMA (scale-factor IDs 0).
__host__ __device__ constexpr uint32_t idesc_nv(int N, int M)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_nv(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_nv_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mx_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// 32 rows x 16 bytes of shared memory -> every TMEM lane quarter, 4 columns
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// the same in both CTAs of a pair: each CTA's shared memory -> its own TMEM
__device__ __forceinline__ void tmem_cp_atom_pair(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory descriptor of 16-byte rows stored contiguously (no swizzle:
// 8-row core matrices 128 bytes apart)
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v)
{
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
// 8 fp32 -> 8 bf16 in one 16-byte store
__device__ __forceinline__ void st8(__nv_bfloat16* dst, const float* v)
{
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(dst) = u;
}
// eight consecutive accumulators (four packed pairs) starting at pair p
__device__ __forceinline__ void get8(const uint64_t* acc, int p, float* v)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2(acc[p + i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// NVFP4: fold a warp's largest magnitude into amax[e] (non-negative floats
// order like their bit patterns)
__device__ __forceinline__ void warp_amax(float m, float* amax, int e)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax) + e, __float_as_uint(m));
}

struct XTile {
    int e, m, n, row0, kblocks, klast, valid_end, alloc_end;   // klast: MMAs in the last k block
};

template <int DUAL, int SCHED, bool PAIR>
__device__ __forceinline__ void xtile_counts(const GemmDesc& d, int& num_m, int& num_n, int& total)
{
    constexpr int NW = (DUAL == DUAL_N) ? XBN / 2 : XBN;
    num_n = (d.N + NW - 1) / NW;
    if (SCHED == SCHED_ROWS) {
        if (d.dense_rows > 0) {   // one dense group of rows (the shared expert)
            const int tiles = (d.dense_rows + XBM - 1) / XBM;
            num_m = PAIR ? (tiles + 1) / 2 : tiles;
        } else {
            num_m = PAIR ? d.meta[2] : d.meta[0];
        }
        total = num_m * num_n;
    } else {
        num_m = d.M_out / (PAIR ? 2 * XBM : XBM);
        total = d.E * num_m * num_n;
    }
}

// Row-scheduled tiles go expert by expert; within an expert, groups of
// kXGroupN column tiles walk its row units (a 128-row tile, or a pair of one
// expert's consecutive tiles, the second possibly a "ghost" past the segment
// that is never stored). Weight-gradient tiles take the experts longest
// first (the order the scan wrote) and walk each expert's (m, n) grid with
// the smaller count fastest.
template <int DUAL, int SCHED, bool PAIR, bool NV = false>
__device__ __forceinline__ XTile xdecode(const GemmDesc& d, int w, int num_m, int num_n, int rank)
{
    constexpr int KE = NV ? 2 * XBK : XBK;   // K values per k block
    XTile t;
    t.klast = 4;
    if (SCHED == SCHED_ROWS) {
        int u0 = 0, nu = num_m;
        if (d.dense_rows == 0) {
            const int q = w / num_n;
            const int e = d.tile_tab[PAIR ? d.pair_tab[q] : q];
            u0 = PAIR ? d.pair_off[e] : d.poff[e] / XBM;
            nu = (PAIR ? d.pair_off[e + 1] : d.poff[e + 1] / XBM) - u0;
        }
        w -= u0 * num_n;
        const int group = w / (nu * kXGroupN);
        const int r = w - group * nu * kXGroupN;
        const int gsz = min(kXGroupN, num_n - group * kXGroupN);
        const int mu = u0 + r / gsz;
        t.n = group * kXGroupN + r % gsz;
        if (d.dense_rows > 0) {
            // a pair's second tile may lie past the rows ("ghost"): not stored
            t.m = PAIR ? 2 * mu + rank : mu;
            t.e = 0;
            t.valid_end = t.alloc_end = d.dense_rows;
        } else {
            const int first = PAIR ? d.pair_tab[mu] : mu;
            t.m = first + rank;
            t.e = d.tile_tab[first];
            t.valid_end = d.poff[t.e] + d.counts[t.e];
            t.alloc_end = d.poff[t.e + 1];
        }
        t.row0 = t.m * XBM;
        t.kblocks = ((DUAL == DUAL_K) ? 2 * d.K : d.K) / KE;
    } else {
        const int per = num_m * num_n;
        const int eo = w / per;
        t.e = d.expert_order ? d.expert_order[eo] : eo;
        const int r = w - eo * per;
        int mu;
        if (num_n < num_m) {
            t.n = r % num_n;
            mu = r / num_n;
        } else {
            mu = r % num_m;
            t.n = r / num_m;
        }
        t.m = PAIR ? 2 * mu + rank : mu;
        // K = the dense rows (padded to the operands' rows_cap), or the
        // expert's padded segment (a multiple of 128 rows; with NVFP4 the
        // last 256-row k block may hold only two 64-row MMAs)
        const int krows = d.dense_rows > 0 ? d.dense_rows : d.poff[t.e + 1] - d.poff[t.e];
        t.row0 = d.dense_rows > 0 ? 0 : d.poff[t.e];
        if (NV) {
            const int chunks = (krows + 63) / 64;
            t.kblocks = (chunks + 3) / 4;
            t.klast = chunks - 4 * (t.kblocks - 1);
        } else {
            t.kblocks = (krows + XBK - 1) / XBK;
        }
        t.valid_end = t.alloc_end = 0;
    }
    return t;
}

template <int EPI, int SCHED, int DUAL, bool B_MN, bool PAIR, bool NV>
__global__ void __launch_bounds__(kXThreads, 1)
gemm_mx_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
               const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
               const __grid_constant__ CUtensorMap mSA0, const __grid_constant__ CUtensorMap mSA1,
               const __grid_constant__ CUtensorMap mSB0, const __grid_constant__ CUtensorMap mSB1,
               const __grid_constant__ CUtensorMap mO0, const __grid_constant__ CUtensorMap mO1,
               const __grid_constant__ CUtensorMap mO2, const GemmDesc d)
{
    using C = XCfg<PAIR, staging_bytes<EPI, SCHED>(), NV>;
    constexpr int NW = (DUAL == DUAL_N) ? XBN / 2 : XBN;   // output columns per tile
    static_assert(!B_MN || (SCHED == SCHED_ROWS && DUAL != DUAL_K), "MN-major B: forward GEMMs");
    static_assert(!(NV && B_MN), "4-bit operands are read K-major");
    constexpr int KE = NV ? 2 * XBK : XBK;    // K values per k block
    constexpr int CH = NV ? 64 : XBK;         // K values per scale atom
    constexpr int AS = KE / CH;               // scale atoms per k block and 128 rows
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t staging = ptx::smem_u32(smem + C::STAGES * C::STAGE);   // 1024-aligned
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + staging_bytes<EPI, SCHED>());
    // full[S], empty[S], accf, acce, final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
    const int unit0 = PAIR ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
    const int nunits = PAIR ? (int)ptx::nclusters_x() : (int)gridDim.x;
    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t accf_bar = bar0 + 8u * (2 * C::STAGES);
    const uint32_t acce_bar = bar0 + 8u * (2 * C::STAGES + 1);
    const uint32_t final_bar = bar0 + 8u * (2 * C::STAGES + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        ptx::mbar_init(accf_bar, 1);
        ptx::mbar_init(acce_bar, PAIR ? 16 : 8);   // the epilogue warps (of both CTAs)
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
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&mSA0);
        ptx::prefetch_tmap(&mSB0);
    }
    if (warp == 1) {
        if (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // peer barriers initialised before any remote signal
    else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int num_m, num_n, total;
    xtile_counts<DUAL, SCHED, PAIR>(d, num_m, num_n, total);
    auto wait_uniform = [&](uint32_t bar, uint32_t parity, int where) -> bool {
        int ok = 1;
        if (lane == 0) ok = ptx::wait_bounded(bar, parity, abort_flag, d.status, where) ? 1 : 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    auto load = [&](uint32_t dst, const CUtensorMap* m, int s, int x, int y) {
        if (PAIR) ptx::tma_load_2d_pair(dst, m, ptx::mapa_shared(full_bar(s), 0), x, y);
        else ptx::tma_load_2d(dst, m, full_bar(s), x, y);
    };
    // the 128-row tiles of B's two 128-column parts (part 1: the same columns
    // of B1 for DUAL_N, else the next 128 columns) and whether part 1 exists
    auto bparts = [&](const XTile& t, int& nb_lo, int& nb_hi, bool& hi_ok) {
        nb_lo = (DUAL == DUAL_N) ? t.n : 2 * t.n;
        nb_hi = (DUAL == DUAL_N) ? t.n : 2 * t.n + 1;
        hi_ok = (DUAL == DUAL_N) || nb_hi < d.N / 128;
    };

    if (warp == 0) {
        // ---------------------------------------------------- loads
        uint32_t it = 0;
        const int kb_half = d.K / KE;
        bool ok = true;
        for (int w = unit0; ok && w < total; w += nunits) {
            const XTile t = xdecode<DUAL, SCHED, PAIR, NV>(d, w, num_m, num_n, rank);
            int nb_lo, nb_hi;
            bool hi_ok;
            bparts(t, nb_lo, nb_hi, hi_ok);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1u;
                if (!wait_uniform(empty_bar(s), ph ^ 1u, 21)) { ok = false; break; }
                if (lane == 0) {
                    if (rank == 0)
                        ptx::mbar_arrive_expect_tx(full_bar(s),
                                                   (PAIR ? 2 : 1) * (C::A_BYTES + C::B_BYTES + C::SF_BYTES));
                    const uint32_t a_dst = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    const uint32_t sf_dst = b_dst + C::B_BYTES;
                    int kx, arow, brow;
                    const CUtensorMap* am = &mA0;
                    const CUtensorMap* bm = &mB0;
                    const CUtensorMap* sam = &mSA0;
                    const CUtensorMap* sbm = &mSB0;
                    int a_atom, b_atom_lo, b_atom_hi;
                    // kx: the k block's first byte of each row; atoms: index of
                    // the first of its AS scale atoms per 128 operand rows
                    if (SCHED == SCHED_ROWS) {
                        const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                        const int kk = second ? kb - kb_half : kb;
                        kx = kk * XBK;
                        arow = t.row0;
                        brow = t.e * d.N + t.n * NW;
                        if (second) { am = &mA1; bm = &mB1; sam = &mSA1; sbm = &mSB1; }
                        const int KA = d.K / CH;
                        const int ebase = t.e * (d.N / 128);
                        a_atom = t.m * KA + AS * kk;
                        b_atom_lo = (ebase + nb_lo) * KA + AS * kk;
                        b_atom_hi = (ebase + (hi_ok ? nb_hi : nb_lo)) * KA + AS * kk;
                    } else {
                        const int krow = t.row0 + kb * KE;   // first K row (token) of the block
                        kx = NV ? krow / 2 : krow;
                        arow = t.m * XBM;
                        brow = t.n * NW;
                        const int KA = d.rows_cap / CH;
                        a_atom = t.m * KA + krow / CH;
                        b_atom_lo = nb_lo * KA + krow / CH;
                        b_atom_hi = (hi_ok ? nb_hi : nb_lo) * KA + krow / CH;
                    }
                    load(a_dst, am, s, kx, arow);
                    // B "part 0" = tile columns [0, 128) (DUAL_N: B0 columns), "part 1" =
                    // [128, 256) (DUAL_N: the same columns of B1). A pair's CTA r stages
                    // part r; a single CTA stages [part 0 | part 1].
                    const CUtensorMap* p0 = (DUAL == DUAL_N) ? &mB0 : bm;
                    const CUtensorMap* p1 = (DUAL == DUAL_N) ? &mB1 : bm;
                    const int r1 = (DUAL == DUAL_N) ? brow : brow + 128;
                    if (B_MN) {
                        const int n0 = t.n * NW;
                        const int c1 = (DUAL == DUAL_N) ? n0 : n0 + 128;
                        const int krow = t.e * d.K + kx;
                        if (PAIR) {
                            load(b_dst, rank ? p1 : p0, s, rank ? c1 : n0, krow);
                        } else {
                            load(b_dst, p0, s, n0, krow);
                            load(b_dst + 128 * XBK, p1, s, c1, krow);
                        }
                    } else if (PAIR) {
                        load(b_dst, rank ? p1 : p0, s, kx, rank ? r1 : brow);
                        load(b_dst + 64 * XBK, rank ? p1 : p0, s, kx, (rank ? r1 : brow) + 64);
                    } else {
                        load(b_dst, p0, s, kx, brow);
                        load(b_dst + 128 * XBK, p1, s, kx, r1);
                        load(b_dst + 64 * XBK, p0, s, kx, brow + 64);
                        load(b_dst + 192 * XBK, p1, s, kx, r1 + 64);
                    }
                    // scale atoms: this CTA's A rows, and both B parts (the MMA reads
                    // the scales of all 256 B columns in each CTA's tensor memory)
                    const CUtensorMap* sb1 = (DUAL == DUAL_N) ? &mSB1 : sbm;
                    load(sf_dst, sam, s, 0, 4 * a_atom);
                    load(sf_dst + 512 * AS, sbm, s, 0, 4 * b_atom_lo);
                    load(sf_dst + 1024 * AS, sb1, s, 0, 4 * b_atom_hi);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (rank == 0) {
            constexpr int MM = PAIR ? 2 * XBM : XBM;
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int w = unit0; ok && w < total; w += nunits) {
                const XTile t = xdecode<DUAL, SCHED, PAIR, NV>(d, w, num_m, num_n, rank);
                if (t.kblocks == 0) continue;              // an expert without rows: zeros
                if (!wait_uniform(acce_bar, (tc & 1u) ^ 1u, 22)) { ok = false; break; }
                ptx::tc_fence_after();
                for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                    const int s = it % C::STAGES;
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    if (!wait_uniform(full_bar(s), ph, 23)) { ok = false; break; }
                    ptx::tc_fence_after();
                    if (NV && lane == 0) {
                        // per MMA k (K = 64): its A atom -> columns 4k of the
                        // stage's 48, its two B atoms -> 16 + 8k (the low
                        // 128 columns) and 20 + 8k (the high 128)
                        const uint32_t a_addr = ptx::smem_u32(smem + s * C::STAGE);
                        const uint32_t b_addr = a_addr + C::A_BYTES;
                        const uint32_t sf_addr = b_addr + C::B_BYTES;
                        const uint32_t sf0 = tmem_base + (uint32_t)(kAccCols + C::SF_COLS * s);
                        const int nm = (kb == t.kblocks - 1) ? t.klast : 4;
                        for (int k = 0; k < nm; ++k) {
                            const uint32_t ta = sf0 + 4u * k, tb = sf0 + 16u + 8u * k;
                            if (PAIR) {
                                tmem_cp_atom_pair(ta, smem_desc_plain(sf_addr + 512 * k));
                                tmem_cp_atom_pair(tb, smem_desc_plain(sf_addr + 2048 + 512 * k));
                                tmem_cp_atom_pair(tb + 4, smem_desc_plain(sf_addr + 4096 + 512 * k));
                            } else {
                                tmem_cp_atom(ta, smem_desc_plain(sf_addr + 512 * k));
                                tmem_cp_atom(tb, smem_desc_plain(sf_addr + 2048 + 512 * k));
                                tmem_cp_atom(tb + 4, smem_desc_plain(sf_addr + 4096 + 512 * k));
                            }
                        }
                        for (int k = 0; k < nm; ++k) {
                            const uint64_t ad = ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
                            const uint64_t bd = ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
                            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                            const uint32_t ta = sf0 + 4u * k, tb = sf0 + 16u + 8u * k;
                            if (PAIR) mma_nv_pair(tmem_base, ad, bd, idesc_nv(XBN, MM), ta, tb, acc);
                            else mma_nv(tmem_base, ad, bd, idesc_nv(XBN, MM), ta, tb, acc);
                        }
                        if (PAIR) ptx::tc_commit_pair(empty_bar(s), 3);
                        else ptx::tc_commit(empty_bar(s));
                    } else if (lane == 0) {
                        const uint32_t a_addr = ptx::smem_u32(smem + s * C::STAGE);
                        const uint32_t b_addr = a_addr + C::A_BYTES;
                        const uint32_t sf_addr = b_addr + C::B_BYTES;
                        const uint32_t sfa = tmem_base + (uint32_t)(kAccCols + C::SF_COLS * s);
                        const uint32_t sfb = sfa + 4;
                        if (PAIR) {
                            tmem_cp_atom_pair(sfa, smem_desc_plain(sf_addr));
                            tmem_cp_atom_pair(sfb, smem_desc_plain(sf_addr + 512));
                            tmem_cp_atom_pair(sfb + 4, smem_desc_plain(sf_addr + 1024));
                        } else {
                            tmem_cp_atom(sfa, smem_desc_plain(sf_addr));
                            tmem_cp_atom(sfb, smem_desc_plain(sf_addr + 512));
                            tmem_cp_atom(sfb + 4, smem_desc_plain(sf_addr + 1024));
                        }
#pragma unroll
                        for (int k = 0; k < XBK / 32; ++k) {
                            const uint64_t ad = ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
                            // MN-major: 32 rows of 128 bytes per K=32 step, stripes of
                            // 128 columns 16 KB apart (one stripe per CTA in a pair)
                            const uint64_t bd = B_MN ? ptx::smem_desc_sw128(b_addr + k * 4096, 128 * XBK, 1024)
                                                     : ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
                            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                            if (PAIR) mma_mx_pair(tmem_base, ad, bd, idesc_mx(XBN, MM, B_MN, k), sfa, sfb, acc);
                            else mma_mx(tmem_base, ad, bd, idesc_mx(XBN, MM, B_MN, k), sfa, sfb, acc);
                        }
                        if (PAIR) ptx::tc_commit_pair(empty_bar(s), 3);
                        else ptx::tc_commit(empty_bar(s));
                    }
                    __syncwarp();
                }
                if (ok && lane == 0) {
                    if (PAIR) ptx::tc_commit_pair(accf_bar, 3);
                    else ptx::tc_commit(accf_bar);
                }
                __syncwarp();
                ++tc;
            }
            // every MMA issued by this warp has completed before TMEM is freed
            if (lane == 0) {
                if (PAIR) ptx::tc_commit_pair(final_bar, 3);
                else ptx::tc_commit(final_bar);
            }
        }
        // (in a pair, the odd CTA's TMEM is written by its peer's MMAs)
        if (lane == 0) {
            volatile int never = 0;
            ptx::wait_bounded(final_bar, 0, &never, d.status, 24);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- accumulator + epilogue
        const int q = warp & 3;                  // TMEM lane quarter
        const int hh = (warp - 2) >> 2;          // 64-column half of each part
        const int r_in = q * 32 + lane;          // row of the CTA's 128
        // This thread takes part-0 columns [64hh, +64) of its row into acc
        // pairs 0-31 and part-1 columns [64hh, +64) into pairs 32-63; part 0 is
        // tile columns [0, 128) (DUAL_N: B0), part 1 [128, 256) (DUAL_N: B1).
        uint32_t tc = 0;
        for (int w = unit0; w < total; w += nunits) {
            const XTile t = xdecode<DUAL, SCHED, PAIR, NV>(d, w, num_m, num_n, rank);
            const int arow = (SCHED == SCHED_ROWS) ? t.row0 + r_in : t.m * XBM + r_in;
            const bool arow_ok = (SCHED == SCHED_ROWS) ? arow < d.a_rows : true;
            (void)arow_ok;
            int nb_lo, nb_hi;
            bool hi_ok;
            bparts(t, nb_lo, nb_hi, hi_ok);
            const int col_lo = (DUAL == DUAL_N) ? t.n * NW + 64 * hh : nb_lo * 128 + 64 * hh;
            const int col_hi = (DUAL == DUAL_N) ? col_lo : nb_hi * 128 + 64 * hh;
            uint64_t acc[64];
            if (t.kblocks > 0) {
                // NVFP4: the MMAs summed code x block-scale products; divide
                // out the two operands' tensor scales
                float gsc = 1.f;
                if (NV) {
                    const int ge = d.dense_rows > 0 ? 0 : t.e;
                    gsc = nv_unscale(d.gA[ge], d.gB[ge]);
                }
                auto us = [&](uint32_t u) { return NV ? __float_as_uint(__uint_as_float(u) * gsc) : u; };
                if (!wait_uniform(accf_bar, tc & 1u, 25)) break;
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + 64u * hh;
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(taddr + (c < 4 ? 16 * c : 128 + 16 * (c - 4)), r0);
                    tmem_ld16(taddr + (c < 4 ? 16 * (c + 1) : 128 + 16 * (c - 3)), r1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        acc[8 * c + i] = pack2(us(r0[2 * i]), us(r0[2 * i + 1]));
                        acc[8 * (c + 1) + i] = pack2(us(r1[2 * i]), us(r1[2 * i + 1]));
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                // relaxed: the accumulator has been read (tcgen05.wait::ld)
                if (lane == 0) {
                    if (PAIR) ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(acce_bar, 0));
                    else ptx::mbar_arrive_relaxed(acce_bar);
                }
                ++tc;
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[j] = 0ull;
            }
            // ---- epilogue from registers (pairs 0-31: part-0 columns, 32-63: part 1)
            float v[8], x[8];
            // this warp's 32 rows x (64 part-0 + 64 part-1) columns go out by TMA:
            // bf16 into two 128-byte-swizzled staging buffers (16-byte chunk j of
            // row r at chunk j ^ (r % 8)), one bulk store each; zero rows where
            // `zero` (pad rows of a segment)
            auto store_staged = [&](int y, bool zero) {
                const uint32_t stg = staging + (uint32_t)(warp - 2) * 4096u;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    if (part == 1 && !hi_ok) break;
                    if (lane == 0) ptx::bulk_wait_read<0>();   // the buffer's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        get8(acc, 32 * part + 4 * j, v);
                        uint4 u4;
                        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u4);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            h2[i] = zero ? __floats2bfloat162_rn(0.f, 0.f) : __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                        const uint32_t addr = stg + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(u4.x), "r"(u4.y),
                                     "r"(u4.z), "r"(u4.w)
                                     : "memory");
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (part == 0) ptx::tma_store_2d(&mO0, stg, col_lo, y);
                        else ptx::tma_store_2d(DUAL == DUAL_N ? &mO1 : &mO0, stg, col_hi, y);
                        ptx::bulk_commit();
                    }
                }
            };
            if (SCHED == SCHED_WGRAD) {
                store_staged(t.e * d.M_out + t.m * XBM + q * 32, false);
            } else if (EPI == EPI_STORE) {
                // segments are 128-row aligned: a warp's 32 rows are all inside the
                // tile's expert or (a pair's ghost half) all past it
                if (t.row0 + q * 32 < t.alloc_end) store_staged(t.row0 + q * 32, arow >= t.valid_end);
            } else if (EPI == EPI_SWIGLU_FWD) {
                // a, u, then h = silu(a) u (g h with the routing weight folded in)
                // of this warp's 32 rows x 64 columns, one after the other through
                // the warp's staging buffer; h's MX row codes (fc2's A operand)
                // from this thread
                if (t.row0 + q * 32 < t.alloc_end) {
                    const bool valid = arow < t.valid_end;
                    const float grow = (d.gates && valid) ? d.gates[d.slot_of[arow]] : 1.f;
                    const int y = t.row0 + q * 32;
                    const uint32_t stg = staging + (uint32_t)(warp - 2) * 4096u;
                    auto put = [&](uint32_t buf, int j, const float* f) {
                        uint4 u4;
                        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u4);
#pragma unroll
                        for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
                        const uint32_t addr = buf + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(u4.x), "r"(u4.y),
                                     "r"(u4.z), "r"(u4.w)
                                     : "memory");
                    };
#pragma unroll
                    for (int part = 0; part < 2; ++part) {   // a (part-0 columns), then u
                        if (lane == 0) ptx::bulk_wait_read<0>();   // the buffer's previous store has read it
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            get8(acc, 32 * part + 4 * j, v);
                            if (!valid) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) v[i] = 0.f;
                            }
                            put(stg, j, v);
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(part ? &mO1 : &mO0, stg, col_lo, y);
                            ptx::bulk_commit();
                        }
                    }
                    if (lane == 0) ptx::bulk_wait_read<0>();
                    __syncwarp();
                    float hmax = 0.f;   // NVFP4: the largest stored |h|
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        float hb[32];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int j = 4 * blk + jj;
                            float hv[8];
                            get8(acc, 4 * j, v);
                            get8(acc, 32 + 4 * j, x);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                hv[i] = valid ? SwigluFwd(v[i], x[i]).h * grow : 0.f;
                                hb[8 * jj + i] = __bfloat162float(__float2bfloat16_rn(hv[i]));
                                if (NV) hmax = fmaxf(hmax, fabsf(hb[8 * jj + i]));
                            }
                            put(stg, j, hv);
                        }
                        if (d.Qrows) {
                            uint4 c0, c1;
                            const int e = encode32(hb, c0, c1);
                            const int col = col_lo + 32 * blk;
                            uint4* dst = reinterpret_cast<uint4*>(d.Qrows + (size_t)arow * d.N + col);
                            dst[0] = c0;
                            dst[1] = c1;
                            d.Qatoms[((size_t)(arow >> 7) * (d.N / 128) + (col >> 7)) * 512 +
                                     atom_byte(arow & 127, (col & 127) >> 5)] = (uint8_t)(e + 127);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&mO2, stg, col_lo, y);
                        ptx::bulk_commit();
                    }
                    if (NV && d.amaxO) warp_amax(hmax, d.amaxO, d.dense_rows > 0 ? 0 : t.e);
                }
            } else if (EPI == EPI_SWIGLU_BWD) {
                // dA, dU of this warp's 32 rows x (64 part-0 + 64 part-1) columns,
                // from dh (the accumulator) and the saved a, u, through the two
                // staging buffers (folded gates: g h for the fc2 weight gradient
                // and the partial dot products dg = <dh', h> too)
                if (t.row0 + q * 32 < t.alloc_end) {
                    const bool valid = arow < t.valid_end;
                    const bool fold = d.gates != nullptr;
                    const float grow = (fold && valid) ? d.gates[d.slot_of[arow]] : 1.f;
                    const int y = t.row0 + q * 32;
                    const size_t orow = (size_t)arow * d.ldo;
                    const uint32_t stg = staging + (uint32_t)(warp - 2) * 8192u;
                    float gmax = 0.f, hmax = 0.f;   // NVFP4: the largest stored |dA|, |dU| and |g h|
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1 && !hi_ok) break;
                        if (lane == 0) ptx::bulk_wait_read<0>();   // both buffers free
                        __syncwarp();
                        const int col = part ? col_hi : col_lo;
                        const size_t o = orow + col;
                        const __nv_bfloat16* X0 = static_cast<const __nv_bfloat16*>(d.X0) + o;
                        const __nv_bfloat16* X1 = static_cast<const __nv_bfloat16*>(d.X1) + o;
                        __nv_bfloat16* O2 = fold && d.O2 ? static_cast<__nv_bfloat16*>(d.O2) + o : nullptr;
                        float dgp = 0.f;
#pragma unroll
                        for (int j0 = 0; j0 < 8; j0 += 2) {
                            uint4 ua[2], uu[2];
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                ua[j] = valid ? *reinterpret_cast<const uint4*>(X0 + 8 * (j0 + j)) : make_uint4(0, 0, 0, 0);
                                uu[j] = valid ? *reinterpret_cast<const uint4*>(X1 + 8 * (j0 + j)) : make_uint4(0, 0, 0, 0);
                            }
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                uint4 oa, ou, oh;
                                const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&ua[j]);
                                const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uu[j]);
                                __nv_bfloat162* da2 = reinterpret_cast<__nv_bfloat162*>(&oa);
                                __nv_bfloat162* du2 = reinterpret_cast<__nv_bfloat162*>(&ou);
                                __nv_bfloat162* dh2 = reinterpret_cast<__nv_bfloat162*>(&oh);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float2 dh = unpack2(acc[32 * part + 4 * (j0 + j) + i]);
                                    const float2 av = __bfloat1622float2(a2[i]);
                                    const float2 uv = __bfloat1622float2(u2[i]);
                                    // pad rows (a = u = 0) give dA = dU = 0
                                    if (fold) {
                                        const SwigluBwdFold r0(dh.x, grow, av.x, uv.x);
                                        const SwigluBwdFold r1(dh.y, grow, av.y, uv.y);
                                        dgp = fmaf(dh.x, r0.h, dgp);
                                        dgp = fmaf(dh.y, r1.h, dgp);
                                        da2[i] = __floats2bfloat162_rn(r0.dA, r1.dA);
                                        du2[i] = __floats2bfloat162_rn(r0.dU, r1.dU);
                                        dh2[i] = __floats2bfloat162_rn(r0.h * grow, r1.h * grow);
                                    } else {
                                        const SwigluBwd r0(dh.x, av.x, uv.x);
                                        const SwigluBwd r1(dh.y, av.y, uv.y);
                                        da2[i] = __floats2bfloat162_rn(r0.dA, r1.dA);
                                        du2[i] = __floats2bfloat162_rn(r0.dU, r1.dU);
                                    }
                                    if (NV) {
                                        const float2 fa = __bfloat1622float2(da2[i]), fu = __bfloat1622float2(du2[i]);
                                        gmax = fmaxf(gmax, fmaxf(fmaxf(fabsf(fa.x), fabsf(fa.y)),
                                                                 fmaxf(fabsf(fu.x), fabsf(fu.y))));
                                        if (fold) {
                                            const float2 fh = __bfloat1622float2(dh2[i]);
                                            hmax = fmaxf(hmax, fmaxf(fabsf(fh.x), fabsf(fh.y)));
                                        }
                                    }
                                }
                                const int jc = j0 + j;
                                const uint32_t sw = (uint32_t)lane * 128u + (uint32_t)((jc ^ (lane & 7)) * 16);
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + sw), "r"(oa.x),
                                             "r"(oa.y), "r"(oa.z), "r"(oa.w)
                                             : "memory");
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + 4096u + sw),
                                             "r"(ou.x), "r"(ou.y), "r"(ou.z), "r"(ou.w)
                                             : "memory");
                                if (O2) *reinterpret_cast<uint4*>(O2 + 8 * jc) = oh;
                            }
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&mO0, stg, col, y);
                            ptx::tma_store_2d(&mO1, stg + 4096u, col, y);
                            ptx::bulk_commit();
                        }
                        if (fold) d.dg_part[(size_t)arow * d.dg_ld + col / 64] = dgp;   // 0 past the computed rows
                    }
                    const int ge = d.dense_rows > 0 ? 0 : t.e;
                    if (NV && d.amaxO) warp_amax(gmax, d.amaxO, ge);
                    if (NV && fold && d.amaxO2) warp_amax(hmax, d.amaxO2, ge);
                }
            }
        }
    }

    if (staging_bytes<EPI, SCHED>() && warp >= 2 && lane == 0) ptx::bulk_wait_all();   // stores complete before exit
    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // both CTAs done with TMEM and with remote signals
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if (PAIR) ptx::tmem_dealloc_pair(tmem_base, 512);
        else ptx::tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 g_encx = nullptr;
std::once_flag g_encx_once;
bool encx()
{
    std::call_once(g_encx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encx = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encx != nullptr;
}

// Row-major byte matrix rows x cols (row stride ld bytes), boxes of
// box_rows x 128 bytes, 128-byte swizzle, out-of-bounds reads 0.
bool mapx(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld, int box_rows)
{
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    return g_encx(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 output rows x cols (row stride ld elements), written in
// 32-row x 64-column boxes with the 128-byte swizzle.
bool map_out(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld)
{
    if (!ptr) {   // unused output map: any valid map will do
        static __nv_bfloat16 dummy[64] __attribute__((aligned(16)));
        ptr = dummy;
        rows = 1;
        cols = 64;
        ld = 64;
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, rows < 32 ? (cuuint32_t)rows : 32u};
    cuuint32_t es[2] = {1u, 1u};
    return g_encx(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms as a [natoms * 4][128] byte tensor read in boxes of `per`
// consecutive atoms (128 x 4 per rows).
bool map_atoms(CUtensorMap* m, const void* ptr, long long natoms, int per = 1)
{
    cuuint64_t dims[2] = {128u, (cuuint64_t)natoms * 4};
    cuuint64_t strides[1] = {128u};
    cuuint32_t box[2] = {128u, 4u * (cuuint32_t)per};
    cuuint32_t es[2] = {1u, 1u};
    return g_encx(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int SCHED, int DUAL, bool B_MN, bool NV>
int xpair_slots()
{
    // computed once (thread-safe initialisation of a function-local static)
    static const int slots = [] {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kXThreads, 1, 1);
        cfg.dynamicSmemBytes = XCfg<true, staging_bytes<EPI, SCHED>(), NV>::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_mx_kernel<EPI, SCHED, DUAL, B_MN, true, NV>, &cfg) != cudaSuccess)
            n = 0;
        cudaGetLastError();
        return n;
    }();
    return slots;
}

template <int EPI, int SCHED, int DUAL, bool B_MN, bool PAIR, bool NV>
cudaError_t xrun(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    constexpr int NW = (DUAL == DUAL_N) ? XBN / 2 : XBN;
    constexpr int CH = NV ? 64 : XBK;   // K values per scale atom
    constexpr int AS = NV ? 4 : 1;      // atoms per k block and 128 rows
    constexpr int VB = NV ? 2 : 1;      // values per code byte
    CUtensorMap mA0, mA1, mB0, mB1, mSA0, mSA1, mSB0, mSB1, mO0, mO1, mO2;
    bool ok = true;
    long long units;
    const long long num_n = (d.N + NW - 1) / NW;
    if (!d.XA0 || !d.XB0 || (DUAL != DUAL_NONE && !d.XB1) || (DUAL == DUAL_K && !d.XA1))
        return cudaErrorInvalidValue;
    if (NV && (!d.gA || !d.gB)) return cudaErrorInvalidValue;
    constexpr int BKROWS = PAIR ? 64 : 64;   // K-major B boxes of 64 rows
    if (SCHED == SCHED_ROWS) {
        const long long KA = d.K / CH;
        ok &= mapx(&mA0, d.A0, d.a_rows, d.K / VB, d.lda / VB, XBM);
        ok &= mapx(&mA1, d.A1 ? d.A1 : d.A0, d.a_rows, d.K / VB, d.lda / VB, XBM);
        // atoms of A: one row of atoms per 128-row tile of the permuted rows
        ok &= map_atoms(&mSA0, d.XA0, (d.a_rows / XBM) * KA, AS);
        ok &= map_atoms(&mSA1, d.XA1 ? d.XA1 : d.XA0, (d.a_rows / XBM) * KA, AS);
        // atoms of B: operand rows e N + n, K blocks of d.K
        const long long b_nrows = (long long)(d.b_rows / d.K) * d.N;   // E * N
        ok &= map_atoms(&mSB0, d.XB0, (B_MN ? b_nrows : d.b_rows) / 128 * KA, AS);
        ok &= map_atoms(&mSB1, d.XB1 ? d.XB1 : d.XB0, (B_MN ? b_nrows : d.b_rows) / 128 * KA, AS);
        if (B_MN) {   // [E*K][N] codes, 128-column x 128-row boxes
            ok &= mapx(&mB0, d.B0, d.b_rows, d.N, d.ldb, XBK);
            ok &= mapx(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, XBK);
        } else {      // [E*N][K] codes
            ok &= mapx(&mB0, d.B0, d.b_rows, d.K / VB, d.ldb / VB, BKROWS);
            ok &= mapx(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.K / VB, d.ldb / VB, BKROWS);
        }
        const long long m_tiles = d.dense_rows > 0 ? (d.dense_rows + XBM - 1) / XBM : max_m_tiles;
        units = (PAIR ? (m_tiles + 1) / 2 : m_tiles) * num_n;
    } else {
        // A: [M_out][rows_cap], B: [N][rows_cap] (transposed operands)
        const long long KA = d.rows_cap / CH;
        ok &= mapx(&mA0, d.A0, d.M_out, d.rows_cap / VB, d.lda / VB, XBM);
        mA1 = mA0;
        ok &= mapx(&mB0, d.B0, d.N, d.rows_cap / VB, d.ldb / VB, BKROWS);
        ok &= mapx(&mB1, d.B1 ? d.B1 : d.B0, d.N, d.rows_cap / VB, d.ldb / VB, BKROWS);
        ok &= map_atoms(&mSA0, d.XA0, (d.M_out / 128) * KA, AS);
        mSA1 = mSA0;
        ok &= map_atoms(&mSB0, d.XB0, (d.N / 128) * KA, AS);
        ok &= map_atoms(&mSB1, d.XB1 ? d.XB1 : d.XB0, (d.N / 128) * KA, AS);
        units = (long long)d.E * (d.M_out / (PAIR ? 2 * XBM : XBM)) * num_n;
        ok &= map_out(&mO0, d.O0, (long long)d.E * d.M_out, d.N, d.ldo);
        ok &= map_out(&mO1, (DUAL == DUAL_N) ? d.O1 : d.O0, (long long)d.E * d.M_out, d.N, d.ldo);
    }
    if (SCHED == SCHED_ROWS) {
        // a dense group's outputs hold its rows alone (the operand codes are padded)
        const long long orows = d.dense_rows > 0 ? d.dense_rows : d.a_rows;
        ok &= map_out(&mO0, d.O0, orows, d.N, d.ldo);
        ok &= map_out(&mO1, EPI != EPI_STORE ? d.O1 : nullptr, orows, d.N, d.ldo);
        ok &= map_out(&mO2, EPI == EPI_SWIGLU_FWD ? d.O2 : nullptr, orows, d.N, d.ldo);
    } else {
        mO2 = mO0;
    }
    if (!ok) return cudaErrorInvalidValue;
    if (units <= 0) return cudaSuccess;
    if (!PAIR) {
        const int grid = (int)(units < num_sms ? units : num_sms);
        gemm_mx_kernel<EPI, SCHED, DUAL, B_MN, false, NV><<<grid, kXThreads, XCfg<false, staging_bytes<EPI, SCHED>(), NV>::SMEM, s>>>(
            mA0, mA1, mB0, mB1, mSA0, mSA1, mSB0, mSB1, mO0, mO1, mO2, d);
        count_launches();
        return cudaGetLastError();
    }
    const int slots = xpair_slots<EPI, SCHED, DUAL, B_MN, NV>();
    if (slots <= 0) return cudaErrorLaunchOutOfResources;
    const long long clusters = units < slots ? units : slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kXThreads, 1, 1);
    cfg.dynamicSmemBytes = XCfg<true, staging_bytes<EPI, SCHED>(), NV>::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches();
    return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<EPI, SCHED, DUAL, B_MN, true, NV>, mA0, mA1, mB0, mB1, mSA0,
                              mSA1, mSB0, mSB1, mO0, mO1, mO2, d);
}

// CTA pairs where the row units come in pairs of one expert's tiles (and
// always for the weight gradients, whose output rows come in 256s).
template <int EPI, int SCHED, int DUAL, bool B_MN, bool NV>
cudaError_t xrun_any(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    const bool pair = (SCHED == SCHED_WGRAD) ? d.M_out % (2 * XBM) == 0
                      : d.dense_rows > 0 ? d.dense_rows > XBM
                                         : (d.pair_tab != nullptr && d.prefer_pair);
    if (pair) return xrun<EPI, SCHED, DUAL, B_MN, true, NV>(d, max_m_tiles, num_sms, s);
    return xrun<EPI, SCHED, DUAL, B_MN, false, NV>(d, max_m_tiles, num_sms, s);
}

template <int EPI, int SCHED, int DUAL, bool B_MN, bool NV>
cudaError_t xattr()
{
    cudaError_t e = cudaFuncSetAttribute(gemm_mx_kernel<EPI, SCHED, DUAL, B_MN, false, NV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         XCfg<false, staging_bytes<EPI, SCHED>(), NV>::SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_mx_kernel<EPI, SCHED, DUAL, B_MN, true, NV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 XCfg<true, staging_bytes<EPI, SCHED>(), NV>::SMEM);
    return e;
}

}  // namespace
}  // namespace moe
