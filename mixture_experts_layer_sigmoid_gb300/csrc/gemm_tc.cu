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
constexpr int kGroupN = 16;    // n tiles per raster group (row-scheduled GEMMs) ...
constexpr int kGroupSpan = 16; // ... or fewer, so that the units sharing a weight tile
                               // are at most this many tiles apart (experts of <= 8 units)

constexpr int kSmemMax = 232448;               // 227 KB per CTA
constexpr int kStaging = 4 * 2 * 4096;          // per epilogue warp: 2 x (32 rows x 128 B)

template <int BN, bool PAIR>
struct TcCfg {
    static constexpr int A_BYTES = TBM * TBK * 2;            // this CTA's 128 rows of A
    static constexpr int B_COLS = PAIR ? BN / 2 : BN;        // this CTA's share of B
    static constexpr int B_BYTES = B_COLS * TBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = (kSmemMax - 1024 - 256 - kStaging) / STAGE;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM = 1024 + STAGES * STAGE + kStaging + 256;
};

struct Tile {
    int e, m, n, row0, kblocks, valid_end, alloc_end;
};

// Scheduling units: single CTAs work on 128-row tiles; CTA pairs on 256-row
// units (two 128-row tiles, one per CTA).
template <int BN, int DUAL, int SCHED, bool PAIR>
__device__ __forceinline__ void tile_counts(const GemmDesc& d, int& num_m, int& num_n, int& total)
{
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;   // output columns per tile
    if (SCHED == SCHED_ROWS) {
        const int tiles = d.dense_rows > 0 ? (d.dense_rows + TBM - 1) / TBM : d.meta[0];
        if (d.dense_rows > 0) num_m = PAIR ? (tiles + 1) / 2 : tiles;
        else if (PAIR) num_m = d.meta[d.row_set == ROWSET_FULL_PAIRS ? 3 : 2];
        else num_m = d.row_set == ROWSET_TAILS ? d.meta[4] : tiles;
        num_n = d.N / NW;
        total = num_m * num_n;
    } else {
        num_m = d.M_out / (PAIR ? 2 * TBM : TBM);
        num_n = d.N / NW;
        total = d.E * num_m * num_n;
    }
}

template <int BN, int DUAL, int SCHED, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const GemmDesc& d, int w, int num_m, int num_n, int rank)
{
    Tile t;
    if (SCHED == SCHED_ROWS) {
        // Groups of G n-tiles: consecutive units share the A rows (one row
        // unit against G weight column tiles), and consecutive groups of them
        // walk the row units, which share the weights. Routed rows go expert
        // by expert (each expert's block of units x num_n tiles is contiguous
        // in w), so an expert's weight column group and its rows stay in L2
        // while its units pass over them. An expert of few units (its rows
        // stay in L2 across groups) takes narrow groups, so that the nu units
        // reading one weight tile run within kGroupSpan consecutive tiles of
        // each other instead of drifting into the next wave; a large one takes
        // kGroupN, which reads its rows once per kGroupN weight tiles.
        // (A launch over the one-tile experts has one unit per expert.)
        const bool tails = !PAIR && d.row_set == ROWSET_TAILS;
        int group, r, u0 = 0, nu = num_m;
        if (d.dense_rows == 0) {
            const int q = w / num_n;                        // some unit of w's expert
            if (tails) {
                u0 = q;
                nu = 1;
            } else {
                const int e = d.tile_tab[PAIR ? d.pair_tab[q] : q];
                u0 = PAIR ? d.pair_off[e] : d.poff[e] / TBM;
                nu = (PAIR ? d.pair_off[e + 1] : d.poff[e + 1] / TBM) - u0;
            }
            w -= u0 * num_n;
        }
        const int G = nu <= kGroupSpan / 2 ? max(1, kGroupSpan / nu) : kGroupN;
        group = w / (nu * G);
        r = w - group * nu * G;
        const int gsz = min(G, num_n - group * G);
        const int mu = u0 + r / gsz;
        t.n = group * G + r % gsz;
        if (d.dense_rows > 0) {
            t.m = PAIR ? 2 * mu + rank : mu;
            t.e = 0;
            t.valid_end = t.alloc_end = d.dense_rows;
        } else {
            // a pair's second tile may lie past its expert's segment ("ghost"):
            // its rows are beyond alloc_end, so nothing of it is stored
            const int first = PAIR ? d.pair_tab[mu] : (tails ? d.tail_tab[mu] : mu);
            t.m = first + rank;
            t.e = d.tile_tab[first];
            t.valid_end = d.poff[t.e] + d.counts[t.e];
            t.alloc_end = d.poff[t.e + 1];
        }
        t.row0 = t.m * TBM;
        t.kblocks = ((DUAL == DUAL_K) ? 2 * d.K : d.K) / TBK;
    } else {
        // Experts longest first (the order the scan wrote), so the persistent
        // units start the longest tiles together and stay in step over them;
        // within an expert the smaller of the m and n tile counts runs fastest,
        // so the units working at once cover all of that dimension against a
        // few slices of the other and read each of those once.
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
        if (d.dense_rows > 0) {
            t.row0 = 0;
            t.kblocks = (d.dense_rows + TBK - 1) / TBK;
        } else {
            // K stops at the 64-row block holding the expert's last computed
            // row: the rest of the segment is zero padding
            t.row0 = d.poff[t.e];
            t.kblocks = (d.counts[t.e] + TBK - 1) / TBK;
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
__device__ __forceinline__ void zero32(float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
}
// 64 consecutive TMEM columns of this warp's 32 lanes: both 32-column loads
// in flight, one wait
__device__ __forceinline__ void tmem_load64f(uint32_t taddr, float (&v0)[32], float (&v1)[32])
{
    uint32_t r0[32], r1[32];
    ptx::tmem_ld32(taddr, r0);
    ptx::tmem_ld32(taddr + 32, r1);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v0[i] = __uint_as_float(r0[i]);
        v1[i] = __uint_as_float(r1[i]);
    }
}

// PAIR: launched as clusters of 2; the even CTA issues M=256 MMAs whose A
// rows 0-127 / 128-255 and B columns are split between the two CTAs'
// shared memory, and each CTA reads its own 128 rows of the accumulator.
template <int BN, bool B_MN, int DUAL, int EPI, int SCHED, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
               const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
               const __grid_constant__ CUtensorMap mO0, const __grid_constant__ CUtensorMap mO1,
               const __grid_constant__ CUtensorMap mO2, const GemmDesc d)
{
    using C = TcCfg<BN, PAIR>;
    constexpr bool A_MN = (SCHED == SCHED_WGRAD);
    constexpr uint32_t IDESC = ptx::idesc_bf16<BN, A_MN, B_MN, PAIR ? 2 * TBM : TBM>();
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t staging = ptx::smem_u32(smem + C::STAGES * C::STAGE);   // 1024-aligned
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + kStaging);
    // bars: full[STAGES], empty[STAGES], accf[2], acce[2], final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
    const int unit0 = PAIR ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
    const int nunits = PAIR ? (int)ptx::nclusters_x() : (int)gridDim.x;
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
            ptx::mbar_init(acce_bar(a), PAIR ? 8 : 4);
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
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // peer barriers initialised before any remote signal
    else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // a launch over the one-tile experts may follow this grid early: it
    // shares no output with it (see the end of the kernel)
    if (PAIR) ptx::griddep_launch_dependents();

    int num_m, num_n, total;
    tile_counts<BN, DUAL, SCHED, PAIR>(d, num_m, num_n, total);

    // Each role runs its loop with the whole warp; lane 0 waits and issues, and
    // the wait's outcome is broadcast so the warp stays converged.
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
        const int kb_half = d.K / TBK;
        bool ok = true;
        for (int w = unit0; ok && w < total; w += nunits) {
            const Tile t = decode_tile<BN, DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
            for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1u;
                if (!wait_uniform(empty_bar(s), ph ^ 1u, 1)) { ok = false; break; }
                if (lane == 0) {
                    if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(s), (PAIR ? 2 : 1) * C::STAGE);
                    const uint32_t a_dst = ptx::smem_u32(smem + s * C::STAGE);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    // this CTA's B columns: a DUAL_N pair splits [B0 | B1] between
                    // the CTAs; otherwise the CTA takes its half of the BN columns
                    const CUtensorMap* bmap = (DUAL == DUAL_N && (PAIR ? rank == 1 : false)) ? &mB1 : &mB0;
                    const int bcol0 = t.n * NW + ((PAIR && DUAL != DUAL_N) ? rank * C::B_COLS : 0);
                    if (SCHED == SCHED_ROWS) {
                        const bool second = (DUAL == DUAL_K) && kb >= kb_half;
                        const int kx = (second ? kb - kb_half : kb) * TBK;
                        load(a_dst, second ? &mA1 : &mA0, s, kx, t.row0);
                        if (B_MN) {
#pragma unroll
                            for (int s2 = 0; s2 < C::B_COLS / 64; ++s2) {
                                const CUtensorMap* m = bmap;
                                int x = bcol0 + 64 * s2;
                                if (!PAIR && DUAL == DUAL_N) {
                                    m = s2 >= BN / 128 ? &mB1 : &mB0;
                                    x = t.n * NW + 64 * (s2 % (BN / 128));
                                }
                                load(b_dst + s2 * STRIPE, m, s, x, t.e * d.K + kb * TBK);
                            }
                        } else {
                            load(b_dst, second ? &mB1 : &mB0, s, kx, t.e * d.N + bcol0);
                        }
                    } else {
                        const int krow = t.row0 + kb * TBK;
#pragma unroll
                        for (int s2 = 0; s2 < TBM / 64; ++s2)
                            load(a_dst + s2 * STRIPE, &mA0, s, t.m * TBM + 64 * s2, krow);
#pragma unroll
                        for (int s2 = 0; s2 < C::B_COLS / 64; ++s2) {
                            const CUtensorMap* m = bmap;
                            int x = bcol0 + 64 * s2;
                            if (!PAIR && DUAL == DUAL_N) {
                                m = s2 >= BN / 128 ? &mB1 : &mB0;
                                x = t.n * NW + 64 * (s2 % (BN / 128));
                            }
                            load(b_dst + s2 * STRIPE, m, s, x, krow);
                        }
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        if (rank == 0) {
            // --------------------------------------------------- MMA issuer
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int w = unit0; ok && w < total; w += nunits, ++tc) {
                const Tile t = decode_tile<BN, DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
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
                            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                            if (PAIR) ptx::tc_mma_f16_pair(d_tmem, ad, bd, IDESC, acc);
                            else ptx::tc_mma_f16(d_tmem, ad, bd, IDESC, acc);
                        }
                        if (PAIR) ptx::tc_commit_pair(empty_bar(s), 3);
                        else ptx::tc_commit(empty_bar(s));
                    }
                    __syncwarp();
                }
                if (ok && lane == 0) {
                    if (PAIR) ptx::tc_commit_pair(accf_bar(a), 3);
                    else ptx::tc_commit(accf_bar(a));
                }
                __syncwarp();
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
            ptx::wait_bounded(final_bar, 0, &never, d.status, 4);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int r_in = q * 32 + lane;         // row of the tile owned by this thread
        // Two 32-row x 128-byte staging buffers per warp, laid out with the
        // 128-byte swizzle of the output tensor maps (16-byte chunk j of row r
        // at chunk j ^ (r % 8)); lane 0 stores them with TMA.
        const uint32_t stg = staging + (uint32_t)q * 8192u;
        uint32_t nstore = 0;
        auto stage_store = [&](const CUtensorMap* m, const float (&a)[32], const float (&b)[32], int x, int y) {
            const uint32_t buf = stg + (nstore & 1u) * 4096u;
            if (nstore >= 2 && lane == 0) ptx::bulk_wait_read<1>();   // this buffer's previous store
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float* src = (j < 4) ? a + 8 * j : b + 8 * (j - 4);
                uint4 u4;
                __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u4);
#pragma unroll
                for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(src[2 * i], src[2 * i + 1]);
                const uint32_t addr = buf + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(u4.x), "r"(u4.y),
                             "r"(u4.z), "r"(u4.w)
                             : "memory");
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d(m, buf, x, y);
                ptx::bulk_commit();
            }
            ++nstore;
        };
        uint32_t tc = 0;
        for (int w = unit0; w < total; w += nunits, ++tc) {
            const Tile t = decode_tile<BN, DUAL, SCHED, PAIR>(d, w, num_m, num_n, rank);
            const int a = tc & 1;
            const uint32_t aph = (tc >> 1) & 1u;
            if (!wait_uniform(accf_bar(a), aph, 5)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN);
            float v0[32], v1[32];
            if (SCHED == SCHED_WGRAD) {
                // 64-column units through shared memory and TMA stores
#pragma unroll 1
                for (int u = 0; u < BN / 64; ++u) {
                    if (t.kblocks > 0) {
                        tmem_load64f(taddr + u * 64, v0, v1);
                    } else {
                        zero32(v0);
                        zero32(v1);
                    }
                    const bool hi = (DUAL == DUAL_N) && u >= NW / 64;
                    const int col = t.n * NW + (u % (NW / 64)) * 64;
                    stage_store(hi ? &mO1 : &mO0, v0, v1, col, t.e * d.M_out + t.m * TBM + q * 32);
                }
            } else {
                const int row = t.row0 + r_in;
                const bool valid = row < t.valid_end;
                const bool warp_in = t.row0 + q * 32 < t.alloc_end;
                if (EPI == EPI_SWIGLU_FWD) {
                    // 64-column units of a (gate half), u (up half) and h = silu(a) u
                    // (g h with the routing weight folded in)
                    const float grow = (d.gates && valid) ? d.gates[d.slot_of[row]] : 1.f;
#pragma unroll 1
                    for (int u = 0; u < NW / 64; ++u) {
                        float g0[32], g1[32], u0[32], u1[32], h0[32], h1[32];
                        tmem_load64f(taddr + u * 64, g0, g1);
                        tmem_load64f(taddr + NW + u * 64, u0, u1);
                        if (warp_in) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                if (valid) {
                                    SwigluFwd r0(g0[i], u0[i]);
                                    SwigluFwd r1(g1[i], u1[i]);
                                    h0[i] = r0.h * grow;
                                    h1[i] = r1.h * grow;
                                } else {
                                    g0[i] = g1[i] = u0[i] = u1[i] = h0[i] = h1[i] = 0.f;
                                }
                            }
                            const int col = t.n * NW + u * 64, y = t.row0 + q * 32;
                            stage_store(&mO0, g0, g1, col, y);
                            stage_store(&mO1, u0, u1, col, y);
                            stage_store(&mO2, h0, h1, col, y);
                        }
                    }
                } else if (EPI == EPI_SWIGLU_BWD) {
                    const bool fold = d.gates != nullptr;
                    const float grow = (fold && valid) ? d.gates[d.slot_of[row]] : 1.f;
#pragma unroll 1
                    for (int u = 0; u < NW / 64; ++u) {
                        float d0[32], d1[32], e0[32], e1[32];
                        tmem_load64f(taddr + u * 64, d0, d1);
                        if (warp_in) {
                            const size_t o = (size_t)row * d.ldo + t.n * NW + u * 64;
                            const __nv_bfloat16* X0 = static_cast<const __nv_bfloat16*>(d.X0) + o;
                            const __nv_bfloat16* X1 = static_cast<const __nv_bfloat16*>(d.X1) + o;
                            float dgp = 0.f;
                            // folded gates: g h of these columns (the fc2 weight-gradient
                            // operand) is written by this thread straight from registers
                            __nv_bfloat16* Hp = fold && d.O2 ? static_cast<__nv_bfloat16*>(d.O2) + o : nullptr;
                            if (valid) {
                                // all 64 columns of a and u in flight at once (one
                                // load round trip per 64-column unit)
                                uint4 ra[8], ru[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    ra[i] = reinterpret_cast<const uint4*>(X0)[i];
                                    ru[i] = reinterpret_cast<const uint4*>(X1)[i];
                                }
                                float av[32], uv[32];
#pragma unroll
                                for (int hf = 0; hf < 2; ++hf) {
                                    float (&dd)[32] = hf ? d1 : d0;
                                    float (&ee)[32] = hf ? e1 : e0;
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&ra[4 * hf + i]);
                                        const __nv_bfloat162* hu = reinterpret_cast<const __nv_bfloat162*>(&ru[4 * hf + i]);
#pragma unroll
                                        for (int jj = 0; jj < 4; ++jj) {
                                            const float2 fa = __bfloat1622float2(ha[jj]);
                                            const float2 fu = __bfloat1622float2(hu[jj]);
                                            av[8 * i + 2 * jj] = fa.x; av[8 * i + 2 * jj + 1] = fa.y;
                                            uv[8 * i + 2 * jj] = fu.x; uv[8 * i + 2 * jj + 1] = fu.y;
                                        }
                                    }
                                    if (fold) {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) {
                                            const SwigluBwdFold r(dd[i], grow, av[i], uv[i]);
                                            dgp = fmaf(dd[i], r.h, dgp);
                                            dd[i] = r.dA; ee[i] = r.dU;
                                            av[i] = r.h * grow;
                                        }
                                        if (Hp) store32_bf16(Hp + 32 * hf, av);
                                    } else {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) {
                                            const SwigluBwd r(dd[i], av[i], uv[i]);
                                            dd[i] = r.dA; ee[i] = r.dU;
                                        }
                                    }
                                }
                            } else {
                                zero32(d0); zero32(d1); zero32(e0); zero32(e1);
                                if (Hp) {
                                    store32_bf16(Hp, d0);
                                    store32_bf16(Hp + 32, d0);
                                }
                            }
                            const int col = t.n * NW + u * 64, y = t.row0 + q * 32;
                            stage_store(&mO0, d0, d1, col, y);
                            stage_store(&mO1, e0, e1, col, y);
                            // every row of the segment (0 past the computed rows), so
                            // that dropped assignments read dg = 0
                            if (fold) d.dg_part[(size_t)row * d.dg_ld + col / 64] = dgp;
                        }
                    }
                } else {
                    // segments are 128-row aligned, so a warp's 32 rows are all
                    // inside the tile's expert or (a pair's ghost half) all past it
#pragma unroll 1
                    for (int u = 0; u < NW / 64; ++u) {
                        tmem_load64f(taddr + u * 64, v0, v1);
                        if (warp_in) {
                            if (!valid) {
                                zero32(v0);
                                zero32(v1);
                            }
                            stage_store(&mO0, v0, v1, t.n * NW + u * 64, t.row0 + q * 32);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            // relaxed: the arrive publishes no memory writes (the TMEM reads are
            // complete after tcgen05.wait::ld), and a release arrive would first
            // wait for this thread's outstanding global loads
            if (lane == 0) {
                if (PAIR) ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(acce_bar(a), 0));
                else ptx::mbar_arrive_relaxed(acce_bar(a));
            }
        }
        if (lane == 0) ptx::bulk_wait_all();   // stores complete before the CTA exits
        __syncwarp();
    }

    ptx::tc_fence_before();
    if (PAIR) ptx::cluster_sync();   // both CTAs done with TMEM and with remote signals
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if (PAIR) ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    // The one-tile experts' launch starts while the pair launch before it
    // drains (programmatic dependent launch) and completes only after it, so
    // the stream's next kernel sees both.
    if (!PAIR && d.row_set == ROWSET_TAILS) ptx::griddep_wait();
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
    if (!ptr) {   // unused output map: any valid map will do
        static __nv_bfloat16 dummy[64] __attribute__((aligned(16)));
        ptr = dummy;
        rows = 1;
        cols = 64;
        ld = 64;
        box_rows = 1;
    }
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

template <int BN, bool B_MN, int DUAL, int EPI, int SCHED, bool PAIR>
cudaError_t set_attr()
{
    return cudaFuncSetAttribute(gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED, PAIR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN, PAIR>::SMEM);
}

// Co-resident clusters of two for a pair kernel (0 if it cannot launch).
template <int BN, bool B_MN, int DUAL, int EPI, int SCHED>
int pair_slots()
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
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = TcCfg<BN, true>::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED, true>, &cfg) !=
            cudaSuccess)
            n = 0;
        cudaGetLastError();
        return n;
    }();
    return slots;
}

template <int BN, bool B_MN, int DUAL, int EPI, int SCHED, bool PAIR>
cudaError_t run(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    constexpr int NW = (DUAL == DUAL_N) ? BN / 2 : BN;
    constexpr int BROWS = TcCfg<BN, PAIR>::B_COLS;   // K-major B box rows
    CUtensorMap mA0, mA1, mB0, mB1, mO0, mO1, mO2;
    bool ok = true;
    long long units;
    // every output is written by TMA stores of 32-row x 64-column boxes
    if (SCHED == SCHED_ROWS) {
        ok &= make_map(&mO0, d.O0, d.a_rows, d.N, d.ldo, 32);
        ok &= make_map(&mO1, d.O1, d.a_rows, d.N, d.ldo, 32);
        ok &= make_map(&mO2, d.O2, d.a_rows, d.N, d.ldo, 32);
    } else {
        ok &= make_map(&mO0, d.O0, (long long)d.E * d.M_out, d.N, d.ldo, 32);
        ok &= make_map(&mO1, (DUAL == DUAL_N) ? d.O1 : d.O0, (long long)d.E * d.M_out, d.N, d.ldo, 32);
        mO2 = mO0;
    }
    if (SCHED == SCHED_ROWS) {
        // A: [a_rows][K] read as 128-row boxes. B: per-expert blocks stacked.
        ok &= make_map(&mA0, d.A0, d.a_rows, d.K, d.lda, TBM);
        ok &= make_map(&mA1, d.A1 ? d.A1 : d.A0, d.a_rows, d.K, d.lda, TBM);
        if (B_MN) {   // B[e*K + k][n]
            ok &= make_map(&mB0, d.B0, d.b_rows, d.N, d.ldb, 64);
            ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, 64);
        } else {      // B[e*N + n][k]
            ok &= make_map(&mB0, d.B0, d.b_rows, d.K, d.ldb, BROWS);
            ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.K, d.ldb, BROWS);
        }
        long long m_tiles = d.dense_rows > 0 ? (d.dense_rows + TBM - 1) / TBM : max_m_tiles;
        if (PAIR) m_tiles = (m_tiles + 1) / 2;
        else if (d.dense_rows == 0 && d.row_set == ROWSET_TAILS) m_tiles = d.E < m_tiles ? d.E : m_tiles;
        units = m_tiles * (d.N / NW);
    } else {
        // A: [rows][M_out], B: [rows][N], read as 64-row boxes of 64 columns.
        ok &= make_map(&mA0, d.A0, d.a_rows, d.M_out, d.lda, 64);
        mA1 = mA0;
        ok &= make_map(&mB0, d.B0, d.b_rows, d.N, d.ldb, 64);
        ok &= make_map(&mB1, d.B1 ? d.B1 : d.B0, d.b_rows, d.N, d.ldb, 64);
        units = (long long)d.E * (d.M_out / (PAIR ? 2 * TBM : TBM)) * (d.N / NW);
    }
    if (!ok) return cudaErrorInvalidValue;
    if (units <= 0) return cudaSuccess;
    if (!PAIR) {
        const int grid = (int)(units < num_sms ? units : num_sms);
        if (d.row_set == ROWSET_TAILS) {
            // after a pair launch: programmatic dependent launch (see the kernel's end)
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.gridDim = dim3((unsigned)grid, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = TcCfg<BN, false>::SMEM;
            cfg.stream = s;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            count_launches();
            return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED, false>, mA0, mA1,
                                      mB0, mB1, mO0, mO1, mO2, d);
        }
        gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED, false>
            <<<grid, kThreads, TcCfg<BN, false>::SMEM, s>>>(mA0, mA1, mB0, mB1, mO0, mO1, mO2, d);
        count_launches();
        return cudaGetLastError();
    }
    const int slots = pair_slots<BN, B_MN, DUAL, EPI, SCHED>();
    if (slots <= 0) return cudaErrorLaunchOutOfResources;
    const long long clusters = units < slots ? units : slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TcCfg<BN, true>::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches();
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, B_MN, DUAL, EPI, SCHED, true>, mA0, mA1, mB0,
                              mB1, mO0, mO1, mO2, d);
}

// Single-CTA or CTA-pair instance: pairs when the row units come in
// (mostly) complete pairs. Routed rows with split tables take two launches:
// CTA pairs over the experts of two or more tiles, then single CTAs over the
// one-tile experts (which a pair would compute beside an empty "ghost" tile;
// an odd last tile of a larger expert keeps its ghost, since a second launch
// would read that expert's weights again).
template <int BN, bool B_MN, int DUAL, int EPI, int SCHED>
cudaError_t run_any(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    bool pair;
    if (SCHED == SCHED_WGRAD) pair = d.M_out % (2 * TBM) == 0;
    else if (d.dense_rows > 0) pair = d.dense_rows > TBM;
    else pair = d.pair_tab != nullptr && d.prefer_pair;
    if (pair && SCHED == SCHED_ROWS && d.dense_rows == 0 && d.full_tab && d.full_off && d.tail_tab) {
        GemmDesc dp = d;
        dp.row_set = ROWSET_FULL_PAIRS;
        dp.pair_tab = d.full_tab;
        dp.pair_off = d.full_off;
        const cudaError_t e = run<BN, B_MN, DUAL, EPI, SCHED, true>(dp, max_m_tiles, num_sms, s);
        if (e != cudaSuccess) return e;
        GemmDesc dt = d;
        dt.row_set = ROWSET_TAILS;
        return run<BN, B_MN, DUAL, EPI, SCHED, false>(dt, max_m_tiles, num_sms, s);
    }
    if (pair) return run<BN, B_MN, DUAL, EPI, SCHED, true>(d, max_m_tiles, num_sms, s);
    return run<BN, B_MN, DUAL, EPI, SCHED, false>(d, max_m_tiles, num_sms, s);
}

}  // namespace

cudaError_t gemm_tc_prepare(int device)
{
    (void)device;
    if (!get_encode()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
#define MOE_ATTR(BN, BMN, DUAL, EPI, SCHED)                       \
    acc(set_attr<BN, BMN, DUAL, EPI, SCHED, false>());             \
    acc(set_attr<BN, BMN, DUAL, EPI, SCHED, true>());
    MOE_ATTR(256, true, DUAL_N, EPI_SWIGLU_FWD, SCHED_ROWS)
    MOE_ATTR(256, true, DUAL_NONE, EPI_STORE, SCHED_ROWS)
    MOE_ATTR(128, true, DUAL_NONE, EPI_STORE, SCHED_ROWS)
    MOE_ATTR(256, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS)
    MOE_ATTR(128, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS)
    MOE_ATTR(256, false, DUAL_K, EPI_STORE, SCHED_ROWS)
    MOE_ATTR(128, false, DUAL_K, EPI_STORE, SCHED_ROWS)
    MOE_ATTR(256, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD)
    MOE_ATTR(128, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD)
    MOE_ATTR(256, true, DUAL_N, EPI_WGRAD, SCHED_WGRAD)
#undef MOE_ATTR
    return e;
}

cudaError_t launch_gemm_tc_bf16(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    if (!get_encode()) return cudaErrorNotSupported;
    const bool n256 = (d.N % 256) == 0;
    if (d.sched == SCHED_ROWS) {
        switch (d.epi) {
        case EPI_SWIGLU_FWD:
            return run_any<256, true, DUAL_N, EPI_SWIGLU_FWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            if (d.dual == DUAL_K)
                return n256 ? run_any<256, false, DUAL_K, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                            : run_any<128, false, DUAL_K, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
            return n256 ? run_any<256, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                        : run_any<128, true, DUAL_NONE, EPI_STORE, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD:
            return n256 ? run_any<256, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s)
                        : run_any<128, false, DUAL_NONE, EPI_SWIGLU_BWD, SCHED_ROWS>(d, max_m_tiles, num_sms, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (d.dual == DUAL_N) return run_any<256, true, DUAL_N, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s);
    return n256 ? run_any<256, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s)
                : run_any<128, true, DUAL_NONE, EPI_WGRAD, SCHED_WGRAD>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
