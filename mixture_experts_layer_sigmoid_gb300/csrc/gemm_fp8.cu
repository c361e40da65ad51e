// gemm_fp8.cu -- persistent grouped GEMM on blockwise-scaled FP8 (E4M3)
// operands with fp32 accumulation, for the MOE_FP8_BLOCK layer.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
// (Platform-specific recipes): blockwise FP8 with 1x128 activation/gradient
// tiles and 128x128 weight blocks. In each GEMM C = A B the operand A
// (rows = output rows) carries one fp32 scale per row and 128-deep K block,
// B one per 128x128 block, so
//   C[r][n] = sum_kb sA[r][kb] sB[kb][n/128] (sum_{k in kb} qA[r][k] qB[k][n]).
// A is stored K-major in E4M3; B is K-major, or (forward GEMMs, B_MN) the
// weights' natural [E][K][N] codes read MN-major, so a weight matrix is
// quantised in one orientation and serves both the forward GEMM (MN-major)
// and the data-gradient GEMM (K-major); its 128x128 block scales are then
// read as [E][K/128][N/128].
//
// Ten warps per CTA: warp 0 TMA producer (stages of A 128x128 B and this
// CTA's share of B, 128-byte swizzle); warp 1 TMEM allocator and, in the
// even CTA, single-thread issuer of tcgen05.mma.kind::f8f6f4 (N = 256, 4 x
// K=32 per k block) into one of two 256-column TMEM partial buffers; warps
// 2-9 promote each finished k block into fp32 registers with its two scales
// (two warps per TMEM lane quarter, 128 columns per thread, packed f32x2
// FMAs) and, at the end of the tile, run the fused epilogue from registers.
// They release a partial buffer with a relaxed mbarrier arrive: a release
// arrive would first wait for their outstanding scale loads and stores, and
// that wait, once per k block, cost more than the MMAs themselves.
// PAIR (in the template, not dispatched: see qrun_any): clusters of two CTAs
// issue M = 256 MMAs (A rows split between the CTAs, B columns split between
// them), so each SM loads 32 KB per 128-deep k block for 128 x 256 x 128 MACs.
#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

constexpr int QBM = 128, QBK = 128, QBN = 256;   // rows per CTA, K block, MMA N
constexpr int kQThreads = 320;
constexpr int kQSmemMax = 232448;
constexpr int kQGroupN = 16;
// MMA unit per partial buffer: false -> one N = 256 MMA per k block into two
// 256-column TMEM buffers; true -> two N = 128 halves into four 128-column
// buffers (deeper, but each half re-reads the A tile from shared memory).
constexpr bool kSplitN = false;
constexpr int kPBuf = kSplitN ? 4 : 2;
constexpr int kPCols = kSplitN ? 128 : 256;
constexpr int kUnitsPerKb = kSplitN ? 2 : 1;

template <bool PAIR>
struct QCfg {
    static constexpr int A_BYTES = QBM * QBK;
    static constexpr int B_ROWS = PAIR ? QBN / 2 : QBN;   // B rows (n) staged by this CTA
    static constexpr int STAGE = A_BYTES + B_ROWS * QBK;
    static constexpr int STAGES = (kQSmemMax - 1024 - 256) / STAGE;
    static constexpr int SMEM = 1024 + STAGES * STAGE + 256;
};

// f8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D, A K-major,
// B K-major or MN-major (bit 16).
__host__ __device__ constexpr uint32_t idesc_e4m3(int N, int M, bool b_mn)
{
    return (1u << 4) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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
__device__ __forceinline__ void mma_e4m3_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
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

// Packed pairs of fp32 accumulators: acc += v * s on both halves at once.
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t v, uint64_t s)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(v), "l"(s));
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

struct QTile {
    int e, m, n, row0, kblocks, kb0, valid_end, alloc_end;
};

template <int DUAL, int SCHED, bool PAIR>
__device__ __forceinline__ void qtile_counts(const GemmDesc& d, int& num_m, int& num_n, int& total)
{
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;
    num_n = (d.N + NW - 1) / NW;
    if (SCHED == SCHED_ROWS) {
        num_m = PAIR ? d.meta[2] : d.meta[0];
        total = num_m * num_n;
    } else {
        num_m = d.M_out / (PAIR ? 2 * QBM : QBM);
        total = d.E * num_m * num_n;
    }
}

// Row-scheduled tiles go expert by expert; within an expert, groups of
// kQGroupN column tiles walk its row units (one unit = a 128-row tile, or a
// pair of one expert's consecutive tiles, the second possibly a "ghost" past
// the segment that is never stored); weight-gradient tiles walk each
// expert's (m, n) grid m-fastest.
template <int DUAL, int SCHED, bool PAIR>
__device__ __forceinline__ QTile qdecode(const GemmDesc& d, int w, int num_m, int num_n, int rank)
{
    QTile t;
    if (SCHED == SCHED_ROWS) {
        // expert by expert (each expert's units x num_n tiles are contiguous in w)
        const int q = w / num_n;
        const int e = d.tile_tab[PAIR ? d.pair_tab[q] : q];
        const int u0 = PAIR ? d.pair_off[e] : d.poff[e] / QBM;
        const int nu = (PAIR ? d.pair_off[e + 1] : d.poff[e + 1] / QBM) - u0;
        w -= u0 * num_n;
        const int group = w / (nu * kQGroupN);
        const int r = w - group * nu * kQGroupN;
        const int gsz = min(kQGroupN, num_n - group * kQGroupN);
        const int mu = u0 + r / gsz;
        t.n = group * kQGroupN + r % gsz;
        const int first = PAIR ? d.pair_tab[mu] : mu;
        t.m = first + rank;
        t.e = d.tile_tab[first];
        t.row0 = t.m * QBM;
        t.valid_end = d.poff[t.e] + d.counts[t.e];
        t.alloc_end = d.poff[t.e + 1];
        t.kblocks = ((DUAL == DUAL_K) ? 2 * d.K : d.K) / QBK;
        t.kb0 = 0;
    } else {
        const int per = num_m * num_n;
        t.e = w / per;
        const int r = w - t.e * per;
        const int mu = r % num_m;
        t.m = PAIR ? 2 * mu + rank : mu;
        t.n = r / num_m;
        t.row0 = d.poff[t.e];
        t.kb0 = t.row0 / QBK;
        t.kblocks = (d.poff[t.e + 1] - t.row0) / QBK;
        t.valid_end = t.alloc_end = 0;
    }
    return t;
}

template <int EPI, int SCHED, int DUAL, bool PAIR, bool B_MN>
__global__ void __launch_bounds__(kQThreads, 1)
gemm_fp8_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
                const GemmDesc d)
{
    using C = QCfg<PAIR>;
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;   // output columns per tile
    static_assert(!B_MN || (SCHED == SCHED_ROWS && DUAL != DUAL_K && !kSplitN), "MN-major B: forward GEMMs");
    constexpr uint32_t IDESC = idesc_e4m3(kPCols, PAIR ? 2 * QBM : QBM, B_MN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
    // full[S], empty[S], pfull[4], pempty[4], final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 9);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
    const int unit0 = PAIR ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
    const int nunits = PAIR ? (int)ptx::nclusters_x() : (int)gridDim.x;
    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto pfull_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
    auto pempty_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 4 + b); };
    const uint32_t final_bar = bar0 + 8u * (2 * C::STAGES + 8);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 4; ++b) {
            ptx::mbar_init(pfull_bar(b), 1);
            // the warps promoting one buffer, in each CTA
            ptx::mbar_init(pempty_bar(b), (kSplitN ? 4 : 8) * (PAIR ? 2 : 1));
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
        if (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 2 * QBN);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 2 * QBN);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // peer barriers initialised before any remote signal
    else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int num_m, num_n, total;
    qtile_counts<DUAL, SCHED, PAIR>(d, num_m, num_n, total);
    auto wait_uniform = [&](uint32_t bar, uint32_t parity, int where) -> bool {
        int ok = 1;
        if (lane == 0) ok = ptx::wait_bounded(bar, parity, abort_flag, d.status, where) ? 1 : 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    auto load = [&](uint32_t dst, const CUtensorMap* m, int s, int x, int y) {
        if (PAIR) ptx::tma_load_2d_pair(dst, m, ptx::mapa_shared(full_bar(s), 0), x, y);
        else ptx::tma_load_2d(dst, m, full_bar(s), x, y);
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        uint32_t it = 0;
        const int kb_half = d.K / QBK;
        bool ok = true;
        for (int w = unit0; ok && w < total; w += nunits) {
            const QTile t = qdecode<DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1u;
                if (!wait_uniform(empty_bar(s), ph ^ 1u, 11)) { ok = false; break; }
                if (lane == 0) {
                    if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(s), (PAIR ? 2 : 1) * C::STAGE);
                    const uint32_t a_dst = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    int kx, arow, brow;
                    const CUtensorMap* am = &mA0;
                    const CUtensorMap* bm = &mB0;
                    if (SCHED == SCHED_ROWS) {
                        const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                        kx = (second ? kb - kb_half : kb) * QBK;
                        arow = t.row0;
                        brow = t.e * d.N + t.n * NW;
                        if (second) { am = &mA1; bm = &mB1; }
                    } else {
                        kx = (t.kb0 + kb) * QBK;
                        arow = t.m * QBM;
                        brow = t.n * NW;
                    }
                    load(a_dst, am, s, kx, arow);
                    // B "part 0" = tile columns [0, 128) (DUAL_N: B0 columns),
                    // "part 1" = [128, 256) (DUAL_N: the same columns of B1).
                    // A pair's CTA r stages part r (128 rows). A single CTA stages
                    // [part0 | part1] for N = 256 MMAs, or, with split halves,
                    // [part0 rows 0-63 | part1 rows 0-63 | part0 rows 64-127 |
                    // part1 rows 64-127] so that half h reads 128 contiguous rows
                    // at offset h x 16 KB: the same columns as a pair's half h.
                    const CUtensorMap* p0 = (DUAL == DUAL_N) ? &mB0 : bm;
                    const CUtensorMap* p1 = (DUAL == DUAL_N) ? &mB1 : bm;
                    const int r1 = (DUAL == DUAL_N) ? brow : brow + 128;
                    if (B_MN) {
                        // MN-major: each part is one 128-column x 128-deep stripe of
                        // the expert's [K][N] codes, at column n0 (part 1: DUAL_N, the
                        // same columns of B1; otherwise the next 128 columns)
                        const int n0 = t.n * NW;
                        const int c1 = (DUAL == DUAL_N) ? n0 : n0 + 128;
                        const int krow = t.e * d.K + kx;
                        if (PAIR) {
                            load(b_dst, rank ? p1 : p0, s, rank ? c1 : n0, krow);
                        } else {
                            load(b_dst, p0, s, n0, krow);
                            load(b_dst + 128 * QBK, p1, s, c1, krow);
                        }
                    } else if (PAIR) {
                        load(b_dst, rank ? p1 : p0, s, kx, rank ? r1 : brow);
                    } else {
                        load(b_dst, p0, s, kx, brow);
                        load(b_dst + (kSplitN ? 64 : 128) * QBK, p1, s, kx, r1);
                        load(b_dst + (kSplitN ? 128 : 64) * QBK, p0, s, kx, brow + 64);
                        load(b_dst + 192 * QBK, p1, s, kx, r1 + 64);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        if (rank == 0) {
            // --------------------------------------------------- MMA issuer
            uint32_t it = 0, pc = 0;
            bool ok = true;
            for (int w = unit0; ok && w < total; w += nunits) {
                const QTile t = qdecode<DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
                for (int kb = 0; kb < t.kblocks; ++kb, ++it, ++pc) {
                    const int s = it % C::STAGES;
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    if (!wait_uniform(full_bar(s), ph, 13)) { ok = false; break; }
                    const uint32_t a_addr = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
                    // the k block's MMA unit(s), into partial buffers u % kPBuf
#pragma unroll
                    for (int h = 0; h < kUnitsPerKb; ++h) {
                        const uint32_t u = kUnitsPerKb * pc + (uint32_t)h;
                        const int pb = (int)(u % kPBuf);
                        if (!wait_uniform(pempty_bar(pb), ((u / kPBuf) & 1u) ^ 1u, 12)) { ok = false; break; }
                        ptx::tc_fence_after();
                        if (lane == 0) {
                            const uint32_t dt = tmem_base + (uint32_t)(pb * kPCols);
                            const uint32_t bh = b_addr + (uint32_t)h * (PAIR ? 64 * QBK : 128 * QBK);
#pragma unroll
                            for (int k = 0; k < QBK / 32; ++k) {
                                const uint64_t ad = ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
                                // MN-major: 32 rows of 128 bytes per K=32 step, stripes of
                                // 128 columns 16 KB apart
                                const uint64_t bd = B_MN ? ptx::smem_desc_sw128(bh + k * 4096, 128 * QBK, 1024)
                                                         : ptx::smem_desc_sw128(bh + k * 32, 16, 1024);
                                if (PAIR) mma_e4m3_pair(dt, ad, bd, IDESC, k > 0 ? 1u : 0u);
                                else mma_e4m3(dt, ad, bd, IDESC, k > 0 ? 1u : 0u);
                            }
                            if (PAIR) ptx::tc_commit_pair(pfull_bar(pb), 3);
                            else ptx::tc_commit(pfull_bar(pb));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (lane == 0) {
                        if (PAIR) ptx::tc_commit_pair(empty_bar(s), 3);
                        else ptx::tc_commit(empty_bar(s));
                    }
                    __syncwarp();
                }
            }
            // every MMA issued by this warp has completed before TMEM is freed
            if (lane == 0) {
                if (PAIR) ptx::tc_commit_pair(final_bar, 3);
                else ptx::tc_commit(final_bar);
            }
        }
        if (lane == 0) {
            volatile int never = 0;
            ptx::wait_bounded(final_bar, 0, &never, d.status, 14);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- promotion + epilogue
        const int q = warp & 3;                  // TMEM lane quarter
        const int hh = (warp - 2) >> 2;          // MMA half owned by this warp
        const int r_in = q * 32 + lane;          // row of the CTA's 128
        // This thread accumulates MMA half hh of its row: part-0 columns
        // [64hh, +64) in acc pairs 0-31 ("lo") and part-1 columns [64hh, +64)
        // in pairs 32-63 ("hi"). Part 0 is tile columns [0, 128) (DUAL_N: B0),
        // part 1 tile columns [128, 256) (DUAL_N: the same columns of B1).
        const int kb_half = d.K / QBK;
        uint32_t pc = 0;
        for (int w = unit0; w < total; w += nunits) {
            const QTile t = qdecode<DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
            const int arow = (SCHED == SCHED_ROWS) ? t.row0 + r_in : t.m * QBM + r_in;
            const bool arow_ok = (SCHED == SCHED_ROWS) ? arow < d.a_rows : true;
            // 128-wide B column blocks of the two parts, and the output columns
            const int nb_lo = (DUAL == DUAL_N) ? t.n : 2 * t.n;
            const int nb_hi = (DUAL == DUAL_N) ? t.n : 2 * t.n + 1;
            const bool hi_ok = (DUAL == DUAL_N) || nb_hi < d.N / 128;
            const int col_lo = (DUAL == DUAL_N) ? t.n * NW + 64 * hh : nb_lo * 128 + 64 * hh;
            const int col_hi = (DUAL == DUAL_N) ? col_lo : nb_hi * 128 + 64 * hh;
            if (EPI == EPI_SWIGLU_BWD && arow_ok && arow < t.alloc_end) {
                // the saved a, u of this thread's columns, into L2 ahead of the epilogue
                const __nv_bfloat16* X0 = static_cast<const __nv_bfloat16*>(d.X0) + (size_t)arow * d.ldo;
                const __nv_bfloat16* X1 = static_cast<const __nv_bfloat16*>(d.X1) + (size_t)arow * d.ldo;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(X0 + col_lo));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(X1 + col_lo));
                if (hi_ok) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(X0 + col_hi));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(X1 + col_hi));
                }
            }
            uint64_t acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0ull;
            bool ok = true;
            // the scales of k block kb (A: this thread's row; B: the two parts' blocks)
            auto scales = [&](int kb, float& sa, float& sb_lo, float& sb_hi) {
                sa = sb_lo = sb_hi = 0.f;
                if (SCHED == SCHED_ROWS) {
                    const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                    const int kk = second ? kb - kb_half : kb;
                    if (arow_ok) sa = (second ? d.SA1 : d.SA0)[(size_t)arow * d.lds_a + kk];
                    const size_t kbs = d.K / 128;
                    const size_t e0 = (size_t)t.e * (d.N / 128);
                    if (B_MN) {
                        // natural block layout [E][K/128][N/128]
                        const float* sbrow = d.SB0 + ((size_t)t.e * kbs + kk) * (d.N / 128);
                        sb_lo = sbrow[nb_lo];
                        if (DUAL == DUAL_N) sb_hi = d.SB1[((size_t)t.e * kbs + kk) * (d.N / 128) + nb_hi];
                        else if (hi_ok) sb_hi = sbrow[nb_hi];
                    } else if (DUAL == DUAL_N) {
                        sb_lo = d.SB0[(e0 + nb_lo) * kbs + kk];
                        sb_hi = d.SB1[(e0 + nb_hi) * kbs + kk];
                    } else {
                        const float* SB = second ? d.SB1 : d.SB0;
                        sb_lo = SB[(e0 + nb_lo) * kbs + kk];
                        if (hi_ok) sb_hi = SB[(e0 + nb_hi) * kbs + kk];
                    }
                } else {
                    const int kg = t.kb0 + kb;
                    sa = d.SA0[(size_t)arow * d.lds_a + kg];
                    if (DUAL == DUAL_N) {
                        sb_lo = d.SB0[(size_t)nb_lo * d.lds_b + kg];
                        sb_hi = d.SB1[(size_t)nb_hi * d.lds_b + kg];
                    } else {
                        sb_lo = d.SB0[(size_t)nb_lo * d.lds_b + kg];
                        if (hi_ok) sb_hi = d.SB0[(size_t)nb_hi * d.lds_b + kg];
                    }
                }
            };
            float nsa = 0.f, nsb_lo = 0.f, nsb_hi = 0.f;   // one k block ahead
            if (t.kblocks > 0) scales(0, nsa, nsb_lo, nsb_hi);
            for (int kb = 0; kb < t.kblocks; ++kb, ++pc) {
                const float sa = nsa, sb_lo = nsb_lo, sb_hi = nsb_hi;
                if (kb + 1 < t.kblocks) scales(kb + 1, nsa, nsb_lo, nsb_hi);
                const float s_lo = sa * sb_lo, s_hi = sa * sb_hi;
                const uint64_t s2_lo = pack2(__float_as_uint(s_lo), __float_as_uint(s_lo));
                const uint64_t s2_hi = pack2(__float_as_uint(s_hi), __float_as_uint(s_hi));
                const uint32_t u = kUnitsPerKb * pc + (kSplitN ? (uint32_t)hh : 0u);
                const int pb = (int)(u % kPBuf);
                if (!wait_uniform(pfull_bar(pb), (u / kPBuf) & 1u, 15)) { ok = false; break; }
                ptx::tc_fence_after();
                // this thread's part-0 and part-1 columns within the buffer
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(pb * kPCols) +
                                       (kSplitN ? 0u : 64u * hh);
                constexpr int kHiOff = kSplitN ? 64 : 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t r[16];
                    tmem_ld16(taddr + (c < 4 ? 16 * c : kHiOff + 16 * (c - 4)), r);
                    ptx::tmem_ld_wait();
                    const uint64_t s2 = c < 4 ? s2_lo : s2_hi;
#pragma unroll
                    for (int i = 0; i < 8; ++i) fma2(acc[8 * c + i], pack2(r[2 * i], r[2 * i + 1]), s2);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR) ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(pempty_bar(pb), 0));
                    else ptx::mbar_arrive_relaxed(pempty_bar(pb));
                }
            }
            if (!ok) break;
            // ---- epilogue from registers (pairs 0-31: part-0 columns, 32-63: part 1)
            float v[8], x[8];
            if (SCHED == SCHED_WGRAD) {
                const size_t ob = (size_t)t.e * d.o_estride + (size_t)arow * d.ldo;
                __nv_bfloat16* Olo = static_cast<__nv_bfloat16*>(d.O0) + ob + col_lo;
                __nv_bfloat16* Ohi = static_cast<__nv_bfloat16*>(DUAL == DUAL_N ? d.O1 : d.O0) + ob + col_hi;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    get8(acc, 4 * j, v);
                    st8(Olo + 8 * j, v);
                }
                if (hi_ok) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        get8(acc, 32 + 4 * j, v);
                        st8(Ohi + 8 * j, v);
                    }
                }
            } else if (arow < t.alloc_end) {
                const bool valid = arow < t.valid_end;
                const size_t orow = (size_t)arow * d.ldo;
                // routing weight of the row when it is folded into h
                const float grow = (d.gates && valid) ? d.gates[d.slot_of[arow]] : 1.f;
                if (EPI == EPI_SWIGLU_FWD) {
                    __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + orow + col_lo;
                    __nv_bfloat16* O1 = static_cast<__nv_bfloat16*>(d.O1) + orow + col_lo;
                    __nv_bfloat16* O2 = static_cast<__nv_bfloat16*>(d.O2) + orow + col_lo;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float hv[8];
                        get8(acc, 4 * j, v);
                        get8(acc, 32 + 4 * j, x);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (valid) {
                                const SwigluFwd r(v[i], x[i]);
                                hv[i] = r.h * grow;
                            } else {
                                v[i] = x[i] = hv[i] = 0.f;
                            }
                        }
                        st8(O0 + 8 * j, v);
                        st8(O1 + 8 * j, x);
                        st8(O2 + 8 * j, hv);
                    }
                } else if (EPI == EPI_SWIGLU_BWD) {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1 && !hi_ok) break;
                        const size_t o = orow + (part ? col_hi : col_lo);
                        const __nv_bfloat16* X0 = static_cast<const __nv_bfloat16*>(d.X0) + o;
                        const __nv_bfloat16* X1 = static_cast<const __nv_bfloat16*>(d.X1) + o;
                        __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + o;
                        __nv_bfloat16* O1 = static_cast<__nv_bfloat16*>(d.O1) + o;
                        const bool fold = d.gates != nullptr;
                        // folded gates: g h (the fc2 weight-gradient operand), from registers
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
                                }
                                *reinterpret_cast<uint4*>(O0 + 8 * (j0 + j)) = oa;
                                *reinterpret_cast<uint4*>(O1 + 8 * (j0 + j)) = ou;
                                if (O2) *reinterpret_cast<uint4*>(O2 + 8 * (j0 + j)) = oh;
                            }
                        }
                        if (fold) {
                            const int col = part ? col_hi : col_lo;
                            d.dg_part[(size_t)arow * d.dg_ld + col / 64] = dgp;   // 0 past the computed rows
                        }
                    }
                } else {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1 && !hi_ok) break;
                        __nv_bfloat16* O0 = static_cast<__nv_bfloat16*>(d.O0) + orow + (part ? col_hi : col_lo);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            get8(acc, 32 * part + 4 * j, v);
                            if (!valid) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) v[i] = 0.f;
                            }
                            st8(O0 + 8 * j, v);
                        }
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // both CTAs done with TMEM and with remote signals
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if (PAIR) ptx::tmem_dealloc_pair(tmem_base, 2 * QBN);
        else ptx::tmem_dealloc(tmem_base, 2 * QBN);
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

template <int EPI, int SCHED, int DUAL, bool B_MN>
int qpair_slots()
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
        cfg.blockDim = dim3(kQThreads, 1, 1);
        cfg.dynamicSmemBytes = QCfg<true>::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_fp8_kernel<EPI, SCHED, DUAL, true, B_MN>, &cfg) != cudaSuccess)
            n = 0;
        cudaGetLastError();
        return n;
    }();
    return slots;
}

template <int EPI, int SCHED, int DUAL, bool PAIR, bool B_MN>
cudaError_t qrun(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    using C = QCfg<PAIR>;
    constexpr int NW = (DUAL == DUAL_N) ? QBN / 2 : QBN;
    // B box rows: a pair's CTA stages its 128-row part in one box; a single
    // CTA stages both parts as four 64-row boxes
    constexpr int BROWS = PAIR ? 128 : 64;
    CUtensorMap mA0, mA1, mB0, mB1;
    bool ok = true;
    long long units;
    const long long num_n = (d.N + NW - 1) / NW;
    if (SCHED == SCHED_ROWS) {
        ok &= map8(&mA0, d.A0, d.a_rows, d.K, d.lda, QBM);
        ok &= map8(&mA1, d.A1 ? d.A1 : d.A0, d.a_rows, d.K, d.lda, QBM);
        if (B_MN) {   // [E*K][N] codes, 128-column x 128-row boxes
            ok &= map8(&mB0, d.B0, d.b_rows, d.N, d.ldb, QBK);
            ok &= map8(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, QBK);
        } else {      // [E*N][K] codes
            ok &= map8(&mB0, d.B0, d.b_rows, d.K, d.ldb, BROWS);
            ok &= map8(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.K, d.ldb, BROWS);
        }
        const long long m_units = PAIR ? (max_m_tiles + 1) / 2 : max_m_tiles;
        units = m_units * num_n;
    } else {
        // A: [M_out][rows_cap], B: [N][rows_cap] (transposed operands)
        ok &= map8(&mA0, d.A0, d.M_out, d.rows_cap, d.lda, QBM);
        mA1 = mA0;
        ok &= map8(&mB0, d.B0, d.N, d.rows_cap, d.ldb, BROWS);
        ok &= map8(&mB1, d.B1 ? d.B1 : d.B0, d.N, d.rows_cap, d.ldb, BROWS);
        units = (long long)d.E * (d.M_out / (PAIR ? 2 * QBM : QBM)) * num_n;
    }
    if (!ok) return cudaErrorInvalidValue;
    if (units <= 0) return cudaSuccess;
    if (!PAIR) {
        const int grid = (int)(units < num_sms ? units : num_sms);
        gemm_fp8_kernel<EPI, SCHED, DUAL, false, B_MN><<<grid, kQThreads, C::SMEM, s>>>(mA0, mA1, mB0, mB1, d);
        count_launches();
        return cudaGetLastError();
    }
    const int slots = qpair_slots<EPI, SCHED, DUAL, B_MN>();
    if (slots <= 0) return cudaErrorLaunchOutOfResources;
    const long long clusters = units < slots ? units : slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches();
    return cudaLaunchKernelEx(&cfg, gemm_fp8_kernel<EPI, SCHED, DUAL, true, B_MN>, mA0, mA1, mB0, mB1, d);
}

// Single CTAs for every FP8 GEMM. The engine releases a TMEM partial buffer
// once per 128-deep k block, and in a CTA pair that release crosses to the
// peer CTA's barrier; on the Qwen3-shaped FP8 layer single CTAs took the row
// GEMMs 8-12% and the weight-gradient GEMMs 1-3% below the pair times (step
// 17.77 -> 16.85 ms), although a pair loads less per SM. The pair
// instantiation (qrun<..., true>) stays available to the template.
template <int EPI, int SCHED, int DUAL, bool B_MN = false>
cudaError_t qrun_any(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    return qrun<EPI, SCHED, DUAL, false, B_MN>(d, max_m_tiles, num_sms, s);
}

template <int EPI, int SCHED, int DUAL, bool B_MN = false>
cudaError_t qattr()
{
    return cudaFuncSetAttribute(gemm_fp8_kernel<EPI, SCHED, DUAL, false, B_MN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, QCfg<false>::SMEM);
}

}  // namespace

cudaError_t gemm_fp8_prepare(int device)
{
    (void)device;
    if (!enc8()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    acc(qattr<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, true>());
    acc(qattr<EPI_STORE, SCHED_ROWS, DUAL_NONE, true>());
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
        // forward GEMMs read the weights' natural codes MN-major (b_kmajor 0),
        // the data-gradient GEMMs K-major (b_kmajor 1)
        case EPI_SWIGLU_FWD:
            if (d.b_kmajor) return cudaErrorInvalidValue;
            return qrun_any<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, true>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD:
            if (!d.b_kmajor) return cudaErrorInvalidValue;
            return qrun_any<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            if (d.dual == DUAL_K)
                return d.b_kmajor ? qrun_any<EPI_STORE, SCHED_ROWS, DUAL_K>(d, max_m_tiles, num_sms, s)
                                  : cudaErrorInvalidValue;
            return d.b_kmajor ? cudaErrorInvalidValue
                              : qrun_any<EPI_STORE, SCHED_ROWS, DUAL_NONE, true>(d, max_m_tiles, num_sms, s);
        default: return cudaErrorInvalidValue;
        }
    }
    return d.dual == DUAL_N ? qrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_N>(d, max_m_tiles, num_sms, s)
                            : qrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
