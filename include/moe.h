/*
 * moe.h -- C ABI of a single-GPU Mixture-of-Experts layer for GB300 (sm_103a),
 * forward and backward.
 *
 * The layer is the one described in "Scalable Training of Mixture-of-Experts
 * Models with Megatron Core", §2 (Megatron-Core MoE Architecture): Route
 * (router logits -> probabilities -> top-k experts, routing weights and a
 * token-expert assignment), Dispatch (permute tokens by destination expert),
 * Expert Computation (all experts' FFNs as grouped GEMMs) and Combine
 * (restore token order, weight by the gates, add a shared expert's output).
 * §5 (Selective precision) keeps the router in FP32; §5 (Kernel and shape
 * optimization) pads expert segments with zero rows to aligned sizes; §7
 * (Load Balancing) lists dropless dispatch, which is the only mode here.
 *
 * Formulas (the pages print none; these are the plain readings):
 *   z = x Wr + b                     (fp32; b optional, per expert)
 *   softmax: p = softmax(z);  sigmoid: s = 1 / (1 + exp(-z))
 *   S_t = the k experts with the largest score, slots in descending score
 *   g_tj = score_{e_tj} / sum_{i in S_t} score_i
 *   expert e (SwiGLU): a = x Wg_e, u = x Wu_e, h = silu(a) u, y_e = h Wd_e
 *   y_t = sum_j g_tj y_{e_tj}(x_t) + shared(x_t)
 * The backward returns the gradient of sum(dY * y) with the routing held
 * fixed; no gradient flows to b.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the plan's device, row-major,
 *     16-byte aligned, owned by the caller. The library never allocates,
 *     frees or keeps device memory; the plan holds host state only.
 *   - Work is enqueued on `stream` (a cudaStream_t) and returns without
 *     synchronising. No call copies device data to the host, so forward and
 *     backward can be captured in a CUDA graph.
 *   - Arguments are validated before anything is enqueued; on any error
 *     nothing is launched and the status says why.
 *   - Errors detected on the device (a pipeline wait that timed out) are
 *     written to a status word at the start of the workspace; read them
 *     with moe_read_status.
 *   - Calls on different streams must use different workspaces.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,          /* null pointer, bad size or enum     */
    MOE_ERR_UNSUPPORTED = 2,          /* valid request the library cannot run */
    MOE_ERR_MISALIGNED = 3,           /* a pointer is not 16-byte aligned    */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4,  /* saved or workspace buffer too small */
    MOE_ERR_CUDA = 5,                 /* a CUDA runtime call failed          */
    MOE_ERR_DEVICE_TIMEOUT = 6        /* a device-side wait ran out          */
} moe_status_t;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;

/* Storage and arithmetic type of activations and expert weights.
 *   MOE_FP32: fp32 storage, fp32 FMA arithmetic throughout.
 *   MOE_BF16: bf16 storage, tensor-core GEMMs with fp32 accumulation.
 *   MOE_FP8_BLOCK: bf16 activations, weights and gradients; every expert
 *     GEMM runs on E4M3 operands with fp32 block scales (1x128 blocks along
 *     K for the operand indexing output rows, 128x128 for the other), fp32
 *     accumulation ("Scalable Training of Mixture-of-Experts Models with
 *     Megatron Core", §5, blockwise FP8). The router stays fp32. Layers with
 *     a shared expert are not supported in this mode (MOE_ERR_UNSUPPORTED).
 *   MOE_MXFP8: bf16 activations, weights and gradients; every expert GEMM
 *     runs on E4M3 operands in the MXFP8 recipe ("Scalable Training of
 *     Mixture-of-Experts Models with Megatron Core", §5 Platform-specific
 *     recipes: the default FP8 recipe on Blackwell, 1x32 granularity): each
 *     32 consecutive values along the GEMM's contraction dimension share one
 *     power-of-two scale 2^e (an UE8M0 byte), e the smallest integer with
 *     amax <= 448 2^e; the tensor cores apply the scales. Both operands of
 *     every GEMM are blocked along K, so weights (and the activations and
 *     gradients that feed two GEMMs) are quantised once per orientation.
 *     The router stays fp32. A shared expert runs through the same engine
 *     as a dense group of the T rows; its weights are quantised by every
 *     forward (the weight cache holds the routed experts' weights).
 *   MOE_NVFP4: as MOE_MXFP8, with every expert GEMM on NVFP4 operands
 *     ("Scalable Training of Mixture-of-Experts Models with Megatron Core",
 *     §5 Platform-specific recipes: NVFP4 for Blackwell): E2M1 values, one
 *     unsigned E4M3 scale per 16 values along K and one fp32 scale
 *     S = 2688 / amax per tensor -- one expert's part of a grouped operand
 *     (or a dense operand), with the gate and up projections [W_gate | W_up]
 *     and their output gradients one tensor each; the tensor cores apply the
 *     block scales (tcgen05.mma.kind::mxf4nvf4, .scale_vec::4X) and the GEMM
 *     epilogue divides out the two tensor scales. Requires H, F and Fs to be
 *     multiples of 256. */
typedef enum { MOE_FP32 = 0, MOE_BF16 = 1, MOE_FP8_BLOCK = 2, MOE_MXFP8 = 3, MOE_NVFP4 = 4 } moe_dtype_t;

typedef struct {
    int H;       /* hidden size; multiple of 128                          */
    int E;       /* routed experts, 1..256                                  */
    int F;       /* routed expert FFN width; multiple of 128                */
    int Fs;      /* shared expert FFN width; 0 = no shared expert, else a
                    multiple of 128                                         */
    int top_k;   /* experts per token, 1..min(E, 8)                         */
    int T_max;   /* largest token count a call may pass, >= 1               */
    int score;   /* moe_score_t                                             */
    int dtype;   /* moe_dtype_t                                             */
    unsigned flags; /* 0, or MOE_FLAG_STAGE_TIMING | MOE_FLAG_FOLD_GATES    */
    float capacity_factor; /* 0 = dropless. > 0: capacity-limited dropping
                    ("Scalable Training of Mixture-of-Experts Models with
                    Megatron Core", §7 Load Balancing): expert e computes at
                    most C = ceil(capacity_factor * T * top_k / E) of the
                    (token, slot) assignments it received, the earliest tokens
                    first; a dropped assignment adds nothing to y, gets no
                    expert gradient and has dg = 0 (its routing gradient still
                    flows through the other slots' renormalised gates).
                    In the FP8 recipes a dropped assignment never reaches its
                    expert: its rows are zeros in every quantisation block
                    along the tokens (the weight-gradient operands). */
} moe_config_t;

/* Plan flag: bracket every kernel launch of moe_forward / moe_backward with
 * CUDA events on the call's stream, for moe_stage_times. A plan with this
 * flag must not be used by two host threads at once. */
#define MOE_FLAG_STAGE_TIMING 1u

/* Plan flag: memory-efficient permutation ("Scalable Training of
 * Mixture-of-Experts Models with Megatron Core", §4, Memory-Efficient
 * Permutation: an algebraic rearrangement that drops intermediate tensors).
 * The routing weight g of each routed row is folded into its activation
 * before fc2 (h' = g silu(a) u), so fc2 yields g y_e directly and Combine is
 * a plain sum; the backward pass forms dg = <dh', h> in the fc2-dgrad
 * epilogue and recomputes h' = g h from the saved a, u for the fc2 weight
 * gradient. Results equal the unfolded layer up to rounding; the saved
 * buffer no longer holds h or the permuted expert outputs (R_pad x (F + H)
 * elements less, R_pad = routed rows padded to 128 per expert), which move
 * to the workspace. */
#define MOE_FLAG_FOLD_GATES 2u

/* Per-stage device time accumulated since the previous moe_stage_times. */
typedef struct {
    char  name[24];   /* stage, e.g. "fc1_swiglu", "fc1_wgrad", "combine"  */
    int   launches;   /* kernel launches of this stage                      */
    float total_ms;   /* summed event-timed duration of those launches      */
} moe_stage_time_t;

typedef struct moe_plan_s* moe_plan_t;

/* Opaque CUDA stream handle; pass a cudaStream_t (0 = legacy default). */
typedef struct CUstream_st* moe_stream_t;

/* Forward arguments. Element type "act" = fp32 for MOE_FP32, bf16 for
 * MOE_BF16. Optional outputs may be NULL. */
typedef struct {
    const void*  x;        /* T×H act: token hidden states                */
    const float* Wr;       /* H×E fp32: router weight                      */
    const float* b;        /* E fp32 router logit bias, or NULL            */
    const void*  W_gate;   /* E×H×F act                                    */
    const void*  W_up;     /* E×H×F act                                    */
    const void*  W_down;   /* E×F×H act                                    */
    const void*  Ws_gate;  /* H×Fs act (NULL iff Fs == 0)                   */
    const void*  Ws_up;    /* H×Fs act                                      */
    const void*  Ws_down;  /* Fs×H act                                      */
    void*        y;        /* out, T×H act                                  */
    int32_t*     topk_idx; /* optional out, T×k: chosen experts, slot order */
    float*       gates;    /* optional out, T×k: renormalised gates         */
    int32_t*     counts;   /* optional out, E: tokens per expert            */
    int32_t*     offsets;  /* optional out, E+1: first padded row of each
                              expert's segment (segments padded to 128 rows) */
    int32_t*     row_of;   /* optional out, T×k: padded row of (t, j)        */
    const int32_t* replay_topk; /* optional in, T×k: router replay (§10, RL
                              post-training) — expert of each (t, j) taken
                              from here instead of the top-k selection; the
                              logits, scores and gates are computed as usual
                              over the given experts (gates = their scores
                              over the sum of their scores). Indices outside
                              [0, E) are clamped and reported as
                              MOE_ERR_INVALID_ARG in the status word. */
    const void*  weight_cache; /* optional in (quantised-expert plans:
                              FP8_BLOCK, MXFP8, NVFP4): expert weights
                              quantised by moe_quantize_weights. When given,
                              W_gate, W_up and W_down are not read (they may
                              be NULL) and the call quantises none of the
                              routed experts' weights (an MXFP8 or NVFP4
                              layer's shared expert weights are still read and
                              quantised);
                              the matching moe_backward must be given the same
                              cache. Other dtypes: must be NULL. */
} moe_fwd_args_t;

/* Backward arguments. Gradients are overwritten (not accumulated); experts
 * that received no token get zero weight gradients. */
typedef struct {
    const void*  dY;       /* T×H act: gradient of the layer output         */
    const void*  x;        /* the forward's x                                */
    const float* Wr;       /* the forward's router weight                     */
    const void*  W_gate;   /* the forward's expert weights                    */
    const void*  W_up;
    const void*  W_down;
    const void*  Ws_gate;  /* the forward's shared-expert weights (or NULL)   */
    const void*  Ws_up;
    const void*  Ws_down;
    void*        dX;       /* out, T×H act                                   */
    float*       dWr;      /* out, H×E fp32                                  */
    void*        dW_gate;  /* out, E×H×F act                                 */
    void*        dW_up;    /* out, E×H×F act                                 */
    void*        dW_down;  /* out, E×F×H act                                 */
    void*        dWs_gate; /* out, H×Fs act (NULL iff Fs == 0)                */
    void*        dWs_up;
    void*        dWs_down;
    const void*  weight_cache; /* quantised recipes: the cache given to the
                              forward (W_gate, W_up, W_down then unread), or
                              NULL when the forward quantised the bf16
                              weights itself. Other dtypes: NULL. */
} moe_bwd_args_t;

/* Validate `cfg` for `device` and build a plan (host memory only).
 * Errors: INVALID_ARG (null, sizes out of range, unknown flags,
 *         capacity_factor negative or not finite),
 *         UNSUPPORTED (dtype not built, device not sm_103, MOE_FP8_BLOCK
 *         with a shared expert, MOE_NVFP4 with H, F or Fs not a multiple of
 *         256), CUDA. */
moe_status_t moe_plan_create(const moe_config_t* cfg, int device, moe_plan_t* out);

/* Free a plan. NULL is accepted. */
moe_status_t moe_plan_destroy(moe_plan_t plan);

/* Bytes of the two caller-owned buffers for a call with T tokens:
 *   saved: written by moe_forward, read by moe_backward (routing, permuted
 *          activations and FFN intermediates of that forward);
 *   ws:    scratch for either call; its first 256 bytes hold the status word.
 * Errors: INVALID_ARG (null, T < 1 or T > T_max). */
moe_status_t moe_workspace_size(moe_plan_t plan, int T, size_t* saved_bytes, size_t* ws_bytes);

/* Enqueue the forward pass for T tokens: Route, Dispatch, Expert
 * Computation, Combine. Writes args->y, the optional outputs and `saved`.
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA. */
moe_status_t moe_forward(moe_plan_t plan, int T, const moe_fwd_args_t* args,
                         void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* Enqueue the backward pass for T tokens, using the `saved` buffer of the
 * forward with the same T, inputs and weights (it is only read).
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA. */
moe_status_t moe_backward(moe_plan_t plan, int T, const moe_bwd_args_t* args,
                          const void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* Synchronise `stream`, then return the device status word kept in `ws`
 * (MOE_OK or MOE_ERR_DEVICE_TIMEOUT); CUDA errors give MOE_ERR_CUDA. */
moe_status_t moe_read_status(moe_plan_t plan, const void* ws, moe_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* moe_status_string(moe_status_t status);

/* Device time per stage of every moe_forward / moe_backward enqueued since
 * the previous call (plans created with MOE_FLAG_STAGE_TIMING only; the
 * measurement covers eagerly launched calls, not graph replays). Waits for
 * the recorded events, writes up to `capacity` entries in first-launch
 * order, sets *count to the number of stages and clears the record.
 * Errors: INVALID_ARG (null, or a plan without the flag), CUDA. */
moe_status_t moe_stage_times(moe_plan_t plan, moe_stage_time_t* out, int capacity, int* count);

/* Routing without a caller-provided workspace. The paper has no
 * counterpart: this entry exists for callers that cannot allocate device
 * memory -- their memory is owned by a framework pool or a budget fixed at
 * start-up, or they run in loops that must not call cudaMalloc (it can
 * synchronise the device) -- and so cannot pass the `ws` buffer that
 * moe_forward needs.
 * Computes, for T tokens, the same routing outputs as moe_forward's optional
 * outputs: topk_idx (T×k), gates (T×k), counts (E), offsets (E+1, padded
 * segment starts) and row_of (T×k), from x (T×H act), Wr (H×E fp32) and the
 * optional bias b (E fp32). All pointers are caller-owned device pointers,
 * 16-byte aligned; nothing is allocated or freed.
 * Scratch: a 64 MiB array inside the library's device image, held on every GPU
 * that loads the library until the process exits. A call needs about
 * 8·T·k + 8·ceil(T/32)·E + 508·min(E, T·k) bytes of it, plus up to 32·T·E
 * for E > 32 (the router's partial logits over at most 8 splits of H); larger
 * T returns MOE_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any
 * stream capture. The address is kept for the life of the process: after a
 * cudaDeviceReset (or any other teardown of the device's primary context)
 * it is stale, and neither this entry point nor a plan created before the
 * reset may be used again on that device. All calls share the array and it keeps the last call's
 * contents (every entry a call reads is written earlier in the same call);
 * calls whose work overlaps on the GPU -- from different streams or host
 * threads -- race on it and must be serialised by the caller.
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA. */
moe_status_t moe_route_static(moe_plan_t plan, int T, const void* x, const float* Wr,
                              const float* b, int32_t* topk_idx, float* gates, int32_t* counts,
                              int32_t* offsets, int32_t* row_of, moe_stream_t stream);

/* Blockwise E4M3 quantiser used by the MOE_FP8_BLOCK layer, on a row-major
 * rows x cols bf16 device matrix (both multiples of 128). Scale of a block =
 * amax / 448 in fp32 (1 for an all-zero block); codes are E4M3 of
 * value / scale, rounded to nearest even and saturated ("Scalable Training of
 * Mixture-of-Experts Models with Megatron Core", §5, blockwise FP8).
 *   MOE_Q_ROWS:    1x128 blocks along rows: codes rows x cols,
 *                  scales rows x cols/128.
 *   MOE_Q_TILES:   128x128 blocks: codes rows x cols, scales (rows/128) x
 *                  (cols/128).
 *   With MOE_Q_ROWS or MOE_Q_TILES, when codes_t and scales_t are both
 *   given, the same pass also writes the 128x128-block codes of the
 *   transpose, codes_t cols x rows with scales_t (cols/128) x (rows/128)
 *   (the layer quantises its gradients this way, reading them once).
 *   MOE_Q_COLS_T:  per column over 128-row blocks, transposed output:
 *                  codes_t cols x rows, scales_t cols x rows/128.
 *   MOE_Q_TILES_T: 128x128 blocks, transposed output: codes_t cols x rows,
 *                  scales_t (cols/128) x (rows/128).
 * Unused outputs may be NULL. Enqueued on `stream`.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
enum { MOE_Q_ROWS = 0, MOE_Q_TILES = 1, MOE_Q_COLS_T = 2, MOE_Q_TILES_T = 3 };
moe_status_t moe_fp8_quantize(int rows, int cols, int mode, const void* in, uint8_t* codes,
                              float* scales, uint8_t* codes_t, float* scales_t, moe_stream_t stream);

/* Quantised expert weights for MOE_FP8_BLOCK, MOE_MXFP8 and MOE_NVFP4 plans ("Scalable Training of
 * Mixture-of-Experts Models with Megatron Core", §5 Kernel and shape
 * optimization: grouped quantization of the experts' weights, done once
 * and kept). A caller that keeps E4M3 weights between steps -- they change
 * once per optimizer step, while a step may run several forward/backward
 * passes -- quantises them once into a caller-owned device buffer, the
 * weight cache, and passes it as weight_cache to moe_forward and
 * moe_backward, which then skip their own weight quantisation.
 *
 * moe_weight_cache_size: bytes of the cache for this plan (0 for plans
 * without quantised experts). Errors: INVALID_ARG.
 *
 * moe_quantize_weights: quantise W_gate, W_up (E x H x F bf16) and W_down
 * (E x F x H bf16) into `cache` (cache_bytes >= the size above), enqueued
 * on `stream`. The cache holds each matrix's E4M3 codes in its own layout
 * with the plan's scales (MOE_FP8_BLOCK: one fp32 scale per 128x128 block,
 * amax / 448, 1 for an all-zero block; MOE_MXFP8: the codes of both
 * orientations, each with its UE8M0 scale per 32 values; MOE_NVFP4: the
 * E2M1 codes of both orientations with their E4M3 scales per 16 values, and
 * each expert's tensor maxima of [W_gate | W_up] and W_down), exactly the codes
 * the layer would produce inside moe_forward; its internal layout is
 * private to the library version. 16-byte aligned device pointers, owned by
 * the caller.
 * Errors: INVALID_ARG (null), UNSUPPORTED (plan has no quantised experts),
 * MISALIGNED, WORKSPACE_TOO_SMALL (cache_bytes), CUDA. */
moe_status_t moe_weight_cache_size(moe_plan_t plan, size_t* bytes);
moe_status_t moe_quantize_weights(moe_plan_t plan, const void* W_gate, const void* W_up,
                                  const void* W_down, void* cache, size_t cache_bytes,
                                  moe_stream_t stream);

/* MXFP8 quantiser used by the MOE_MXFP8 layer, on a row-major rows x cols
 * bf16 device matrix (both multiples of 128). Blocks of 32 values share the
 * scale 2^e, e the smallest integer with amax <= 448 2^e, clamped to
 * [-127, 127] (-127 for an all-zero block), stored as the UE8M0 byte
 * e + 127; a value is stored as the E4M3 code of v 2^-e (round to nearest
 * even). Scales are written as "scale atoms", the layout the GEMMs copy into
 * tensor memory: for an operand read as [n][K], one 512-byte atom per
 * 128-row tile t and 128-deep K block b at (t * K/128 + b) * 512, whose byte
 * 16 (m % 32) + 4 (m / 32) + j holds the scale of tile row m and 32-deep
 * sub-block j.
 *   codes, scales (optional): blocks along the rows; codes rows x cols,
 *     atoms of the [rows][K = cols] operand (rows * cols / 32 bytes).
 *   codes_c, scales_c (optional): blocks down the columns (32 rows each);
 *     col_transposed 1: codes cols x rows (the transpose), col_transposed 0:
 *     codes rows x cols in place; atoms of the [cols][K = rows] operand.
 * At least one pair must be given. Enqueued on `stream`.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
moe_status_t moe_mx_quantize(int rows, int cols, const void* in, uint8_t* codes, uint8_t* scales,
                             uint8_t* codes_c, uint8_t* scales_c, int col_transposed, moe_stream_t stream);

/* NVFP4 quantiser used by the MOE_NVFP4 layer, on a row-major rows x cols
 * bf16 device matrix (both multiples of 128) taken as one tensor: its
 * largest magnitude goes to *amax (a device float, overwritten), the tensor
 * scale is S = 2688 / amax (1 for an all-zero matrix), and each block of
 * 16 values gets the E4M3 scale sb = E4M3(a S / 6) (a the block's largest
 * magnitude; s its value) and the E2M1 codes of v (S / s) (nearest, ties to
 * the even code, saturating at 6; zero codes when s = 0), every step an
 * fp32 operation rounded to nearest even. Codes are packed two per byte,
 * the lower-index value in the low 4 bits. Scale atoms: for an operand read
 * as [n][K], one 512-byte atom per 128-row tile t and 64-value K chunk b at
 * (t * K/64 + b) * 512, whose byte 16 (m % 32) + 4 (m / 32) + j holds the
 * scale of tile row m and 16-value sub-block j.
 *   codes, scales (optional): blocks along the rows; codes rows x cols/2
 *     bytes, atoms of the [rows][K = cols] operand (rows * cols / 16 bytes).
 *   codes_t, scales_t (optional): blocks down the columns (16 rows each),
 *     codes of the transpose, cols x rows/2 bytes; atoms of the
 *     [cols][K = rows] operand.
 * At least one pair must be given. Enqueued on `stream`.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
moe_status_t moe_nv_quantize(int rows, int cols, const void* in, float* amax, uint8_t* codes, uint8_t* scales,
                             uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream);

/* Failure-detection check. Every pipelined kernel of the library waits on
 * its shared-memory mbarriers with a bounded wait (2 s); when a wait runs out
 * the kernel records MOE_ERR_DEVICE_TIMEOUT in the status word and returns,
 * so a stalled pipeline ends with an error instead of hanging the GPU. This
 * entry point runs that wait on an mbarrier that is never signalled: after
 * the call, moe_read_status(plan, ws, stream) returns MOE_ERR_DEVICE_TIMEOUT
 * and the device stays usable. `ws` is any workspace (its status word is
 * overwritten). Errors: INVALID_ARG, CUDA. */
moe_status_t moe_diag_wait_timeout(void* ws, moe_stream_t stream);

/* Auxiliary-loss-free load balancing: one update of the per-expert router
 * logit bias ("Scalable Training of Mixture-of-Experts Models with Megatron
 * Core", §7 Load Balancing, "auxiliary-loss-free biasing"; the pages give no
 * rule): with c_e the tokens expert e received in the last forward (the
 * `counts` output) and c_mean their mean over the E experts,
 *   b_e <- b_e + rate * sign(c_mean - c_e),   sign(0) = 0,
 * so under-loaded experts become more likely to be selected and over-loaded
 * ones less. The comparison is exact (integers: E*c_e against sum of c).
 * counts: E int32, b: E fp32 (updated in place), device pointers, enqueued
 * on `stream`. Errors: INVALID_ARG (null, E outside 1..256, rate not
 * finite), CUDA. */
moe_status_t moe_update_bias(int E, const int32_t* counts, float rate, float* b, moe_stream_t stream);

/* MOE_ABI_VERSION of the loaded library. */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
