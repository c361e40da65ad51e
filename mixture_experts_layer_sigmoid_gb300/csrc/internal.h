// internal.h -- declarations shared by the CUDA translation units of the
// MoE layer library (not part of the public ABI; see include/moe.h).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>
#include <stdint.h>
#include <stddef.h>

#include "moe.h"

struct moe_plan_s;

namespace moe {

// Rows of one grouped-GEMM M tile; every expert segment of the permuted
// buffers is padded with zero rows to a multiple of this.
constexpr int kTileM = 128;
// Tokens per router block (one per-block expert histogram each).
constexpr int kRouterTokens = 32;
// Largest number of routed experts / top-k the kernels accept.
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
constexpr int kRouterSplitMax = 8;   // H splits of the tiled router (partial logits in the workspace)
// Device-side wait limit of the pipelined kernels, in nanoseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Status word at the start of the workspace.
struct DeviceStatus {
    int code;   // moe_status_t
    int where;  // kernel-specific location of the first error
};

// ----------------------------------------------------------- grouped GEMM
// Scheduling of output tiles.
enum Sched : int {
    SCHED_ROWS = 0,   // M = permuted rows (one expert per 128-row tile), fixed K
    SCHED_WGRAD = 1,  // per expert: M_out x N output, K = the expert's rows
};
// Which routed row tiles one launch covers.
enum RowSet : int {
    ROWSET_ALL = 0,         // every tile (pairs: a lone last tile runs beside a ghost)
    ROWSET_FULL_PAIRS = 1,  // CTA pairs over full_tab / full_off (multi-tile experts)
    ROWSET_TAILS = 2,       // single CTAs over tail_tab (one-tile experts)
};
// What the epilogue does with the fp32 accumulator(s).
enum Epi : int {
    EPI_SWIGLU_FWD = 0,  // acc0 = a, acc1 = u -> O0 = a, O1 = u, O2 = silu(a) u
    EPI_STORE = 1,       // acc0 -> O0
    EPI_SWIGLU_BWD = 2,  // acc0 = dh; X0 = a, X1 = u -> O0 = dA, O1 = dU
    EPI_WGRAD = 3,       // acc0 -> O0[e], acc1 -> O1[e] (dual)
};
// Two operand sources.
enum Dual : int {
    DUAL_NONE = 0,
    DUAL_N = 1,  // two B operands, two accumulators over the same A
    DUAL_K = 2,  // A0 B0 + A1 B1 into one accumulator (K = 2 x K0)
};

struct GemmDesc {
    int sched, epi, dual;
    int N;          // columns of each accumulator (whole output width)
    int K;          // SCHED_ROWS: contraction length of each source
    int M_out;      // SCHED_WGRAD: output rows per expert
    int E;          // expert groups (SCHED_WGRAD) -- 1 for a dense group
    int dense_rows; // > 0: a single dense group of rows [0, dense_rows)
    // row tables (routed groups)
    const int* tile_tab;  // expert of each 128-row tile
    const int* meta;      // meta[0] = number of 128-row tiles, meta[1] = padded rows,
                          // meta[2] = number of tile pairs, meta[3] = number of
                          // pairs of multi-tile experts, meta[4] = number of
                          // one-tile experts
    const int* pair_tab;  // first tile of each pair of one expert's tiles (or null)
    const int* pair_off;  // E+1: first pair of each expert (with pair_tab)
    int prefer_pair;      // routed rows per expert are large enough for CTA pairs
    // Split row sets (bf16 tensor-core path): the pairs of the experts with
    // two or more tiles, and the tile of each one-tile expert, so that CTA
    // pairs never compute a ghost tile for an expert of 128 rows or fewer.
    const int* full_tab;  // first tile of each pair of a multi-tile expert
    const int* full_off;  // E+1: first such pair of each expert
    const int* tail_tab;  // the tiles of the one-tile experts
    int row_set;          // ROWSET_* (set by the launcher)
    const int* expert_order;  // weight gradients: experts in this order (null: 0..E-1)
    const int* poff;      // E+1 padded segment offsets
    const int* counts;    // E rows computed per expert (token counts, or the
                          // kept counts under capacity-limited dropping)
    // operands (element pointers; the tensor-core path builds TMA maps from them)
    const void* A0; const void* A1; int lda;      // ROWS: A[row][k]; WGRAD: A[row][m]
    const void* B0; const void* B1; int ldb;
    int b_kmajor;              // ROWS: 1 -> B(k,n) = B[e*bstride + n*ldb + k]
                               //       0 -> B(k,n) = B[e*bstride + k*ldb + n]
    long long b_estride;       // elements between experts' B blocks
    int a_rows, b_rows;        // rows of the A / B tensors (TMA bounds)
    // epilogue
    void* O0; void* O1; void* O2; int ldo;
    long long o_estride;       // WGRAD: elements between experts' outputs
    const void* X0; const void* X1;  // SWIGLU_BWD: saved a, u (ld = ldo)
    DeviceStatus* status;
    // blockwise FP8 only: fp32 block scales of the E4M3 operands
    const float* SA0; const float* SA1; int lds_a;   // A: 1x128 blocks along K
    const float* SB0; const float* SB1; int lds_b;   // B: 128x128 blocks
    int rows_cap;   // SCHED_WGRAD: row capacity of the transposed operands
    // MXFP8 only: UE8M0 scale atoms of the operands (see launch_mx_quant)
    const uint8_t* XA0; const uint8_t* XA1; const uint8_t* XB0; const uint8_t* XB1;
    // MXFP8 SWIGLU_FWD: also the MX row codes [rows][N] of h (O2) and their atoms
    uint8_t* Qrows; uint8_t* Qatoms;
    // NVFP4 operands (nv != 0; the same atoms fields, 64-value K chunks): the
    // largest magnitude of each expert's A and B tensors (index 0 for a
    // dense group), whose tensor scales the epilogue divides out
    int nv;
    const float* gA; const float* gB;
    // NVFP4 SwiGLU epilogues: the largest magnitude of the bf16 values they
    // store, per expert (atomicMax; zeroed by the caller): SWIGLU_FWD h into
    // amaxO; SWIGLU_BWD [dA | dU] into amaxO and, with folded gates, g h into
    // amaxO2 (null: not computed)
    float* amaxO; float* amaxO2;
    // memory-efficient permutation (gates != null): g of permuted row r is
    // gates[slot_of[r]]. SWIGLU_FWD stores O2 = g h; SWIGLU_BWD treats the
    // accumulator as dh', writes dA, dU of dh = g dh', O2 = g h (if O2 is
    // set) and dg_part[r][c / 64] = sum over the 64 columns from c of dh' h
    // (row stride dg_ld floats).
    const int* slot_of;
    const float* gates;
    float* dg_part;
    int dg_ld;
};

// Launchers (return cudaGetLastError()).
cudaError_t launch_gemm_simt_f32(const GemmDesc& d, int max_m_tiles, cudaStream_t s);
cudaError_t launch_gemm_tc_bf16(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s);
cudaError_t gemm_tc_prepare(int device);
cudaError_t launch_gemm_fp8(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s);
cudaError_t gemm_fp8_prepare(int device);

// Kernels enqueued by this host thread: every launcher adds the launches it
// made, so a timed stage can report how many kernels it ran.
extern thread_local unsigned long long t_kernel_launches;
inline void count_launches(int n = 1) { t_kernel_launches += (unsigned long long)n; }

// ------------------------------------------------------------- routing etc.
template <typename T>
cudaError_t launch_router(const T* x, const float* Wr, const float* b, int T_, int H, int E, int k,
                          int score, int* topk, float* gates, float* selsc, int* hist,
                          cudaStream_t s,
                          const int* replay = nullptr, DeviceStatus* status = nullptr,
                          float* zpart = nullptr, size_t zpart_floats = 0);
// fp32 entries of the partial-logit buffer launch_router needs for T tokens
// (0 when the router for this H and E runs unsplit).
size_t router_zpart_floats(int T, int H, int E);
cudaError_t launch_scan(const int* hist, int nblk, int E, int* counts, int* poff, int* blkbase,
                        int* tile_tab, int* meta, int* slot_of, cudaStream_t s,
                        int* pair_tab = nullptr, int* pair_off = nullptr, int cap = -1,
                        int* kept = nullptr, int* eorder = nullptr, int* full_tab = nullptr,
                        int* full_off = nullptr, int* tail_tab = nullptr);
// slot_live (optional, capacity-limited dropping): slot_live[r] = slot_of[r]
// for the rows an expert computes (r < poff[e] + kept[e]); the caller sets
// the array to -1 first, so dropped and pad rows read -1.
cudaError_t launch_index(const int* topk, const int* blkbase, int T_, int E, int k, int* row_of,
                         int* slot_of, cudaStream_t s, const int* poff = nullptr,
                         const int* kept = nullptr, int* slot_live = nullptr);
// slot_live (optional): rows it marks -1 (dropped assignments) are written as zeros.
template <typename T>
cudaError_t launch_permute(const T* x, const int* row_of, const int* poff, const int* counts,
                           int T_, int H, int E, int k, T* Xp, cudaStream_t s,
                           const int* slot_live = nullptr);
template <typename T>
cudaError_t launch_combine(const T* Yp, const T* Ys, const int* row_of, const float* gates,
                           int T_, int H, int k, T* y, cudaStream_t s);
// slot_live (optional): the rows of dropped assignments get dYp = 0.
template <typename T>
cudaError_t launch_gate_grad(const T* dY, const T* Yp, const int* row_of, const int* topk,
                             const float* gates, const float* selsc, const int* poff,
                             const int* counts, int T_, int H, int E, int k, int score, T* dYp,
                             float* dz, cudaStream_t s, const int* slot_live = nullptr);
// Folded routing weights: dz from the fc2-dgrad partial dot products.
cudaError_t launch_gate_dz(const float* dg_part, int nslots, const int* row_of, const float* gates,
                           const float* selsc, int T_, int k, int score, float* dz, cudaStream_t s);
// x: the layer input (row r of the permuted buffer is token slot_of[r] / k);
// part: MT_max x H fp32 scratch (per-tile partial sums).
template <typename T>
cudaError_t launch_router_wgrad(const T* x, const int* slot_of, const int* poff, const int* meta,
                                int MT_max, const float* dz, int H, int E, int k, float* part,
                                float* dWr, cudaStream_t s);
cudaError_t launch_transpose_f32(const float* in, int rows, int cols, float* out, cudaStream_t s);
template <typename T>
cudaError_t launch_unpermute_reduce(const T* dXp, const T* dXs, const int* row_of,
                                    const int* topk, const float* dz, const float* WrT, int T_,
                                    int H, int k, T* dX, cudaStream_t s);

// blockwise FP8 quantisers (quant.cu)
// Xp may be null (codes only).
cudaError_t launch_permute_quant(const __nv_bfloat16* x, const int* row_of, const int* poff,
                                 const int* counts, int T_, int H, int E, int k, __nv_bfloat16* Xp,
                                 uint8_t* Xq, float* sX, cudaStream_t s);
// One pass of the tile quantiser over in[rows][C] (bf16, rows = *rows_dev or
// rows_max, both multiples of 128, as is C). q != null: codes [rows][C] with
// 1x128 row-block scales s[rows][C/128] (q_tiles 0) or one scale per 128x128
// tile s[rows/128][C/128] (q_tiles 1). qT != null: transposed codes
// [C][rows_cap] with per-column scales over 128 rows sT[C][rows_cap/128]
// (t_tiles 0) or per-tile scales sT[C/128][rows_cap/128] (t_tiles 1).
// gather_slot != null: row r of the input is row gather_slot[r] / gather_k of
// `in` (the token of a permuted row), or zeros where gather_slot[r] < 0.
struct QuantJob {
    const __nv_bfloat16* in;
    const int* rows_dev;
    int rows_max, C, rows_cap;
    uint8_t* q; float* s; int q_tiles;
    uint8_t* qT; float* sT; int t_tiles;
    const int* gather_slot = nullptr;
    int gather_k = 1;
};
cudaError_t launch_quant(const QuantJob& j, cudaStream_t s);

// MXFP8 quantisers (quant_mx.cu). Scale atoms: for an operand read as
// [rows][K], one 512-byte atom per (128-row tile rt, 128-deep K block kb) at
// (rt * K/128 + kb) * 512, byte 16 (m % 32) + 4 (m / 32) + j = UE8M0 scale of
// tile row m and 32-deep sub-block j.
cudaError_t launch_mx_permute(const __nv_bfloat16* x, const int* row_of, const int* poff, const int* counts,
                              int T_, int H, int E, int k, uint8_t* Xq, uint8_t* sfX, cudaStream_t s);
// One pass over in[rows][C] (bf16; rows = *rows_dev or rows_max, multiples
// of 128, as is C). q != null: row codes q[rows][C] (blocks along rows) with
// atoms sf. qc != null: column codes (blocks of 32 down each column), either
// transposed qc[C][rows_cap] with atoms sfc of the [C][rows_cap] operand
// (col_mode 1), or in place qc[rows][C] for expert-stacked weights
// [rows / grp][grp][C] read MN-major with K = grp (col_mode 2).
struct MxQuantJob {
    const __nv_bfloat16* in;
    const int* rows_dev;
    int rows_max, C, rows_cap;
    uint8_t* q; uint8_t* sf;
    uint8_t* qc; uint8_t* sfc; int col_mode;
    int grp = 0;
    const int* gather_slot = nullptr;
    int gather_k = 1;
    int rows_valid = 0;   // > 0: rows from here on (up to rows_max) read as zeros
};
cudaError_t launch_mx_quant(const MxQuantJob& j, cudaStream_t s);

// NVFP4 quantisation (quant_nv.cu, encoding in nv.cuh): [rows][C] bf16 in
// 128 x 128 tiles -> row codes q[rows][C/2] (16-value blocks along rows)
// and/or transposed codes qc (16-row blocks down columns, per group of grp
// rows: column c of group g at qc[((g C + c) grp + r) / 2]), each with 512-byte
// scale atoms per 128-row tile and 64-value K chunk. The tensor of a
// 128-row tile (for its fp32 scale 2688 / amax[tensor]): the padded segment
// of seg_off (nseg + 1 offsets) holding it, else row / seg_rows (seg_rows 0:
// one tensor). Gather and rows_valid as in MxQuantJob.
struct NvQuantJob {
    const __nv_bfloat16* in;
    const int* rows_dev;     // rows to visit (device), or null: rows_max
    int rows_max, C, rows_cap;
    uint8_t* q; uint8_t* sf;
    uint8_t* qc; uint8_t* sfc;
    int grp;
    const int* seg_off; int nseg;
    int seg_rows;
    const float* amax;       // quantisation: per-tensor largest magnitudes
    const int* gather_slot; int gather_k;
    int rows_valid;
};
// atomicMax of each tile's largest magnitude into amax[tensor] (amax zeroed
// by the caller)
cudaError_t launch_nv_amax(const NvQuantJob& j, float* amax, cudaStream_t s);
cudaError_t launch_nv_quant(const NvQuantJob& j, cudaStream_t s);
// The permuted rows' NVFP4 row codes (K = H) from x: each expert's maximum
// over the rows it keeps (amax zeroed by the caller), then each token's k
// rows in their experts' tensor scales; pad rows get zero codes.
cudaError_t launch_nv_permute(const __nv_bfloat16* x, const int* topk, const int* row_of, const int* poff,
                              const int* counts, const int* kept, int T_, int H, int E, int k, float* amax,
                              uint8_t* Xq, uint8_t* sfX, cudaStream_t s);
cudaError_t launch_gemm_mx(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s);
cudaError_t gemm_mx_prepare(int device);
// NVFP4 operands (d.nv, d.gA, d.gB set; every B K-major)
cudaError_t launch_gemm_nv(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s);
cudaError_t gemm_nv_prepare(int device);

// Configuration and device of a plan; false for a null plan.
bool plan_info(const moe_plan_s* plan, moe_config_t* cfg, int* device);

}  // namespace moe
