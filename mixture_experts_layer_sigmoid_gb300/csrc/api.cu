// api.cu -- the C ABI of include/moe.h: argument validation, the layout of
// the caller-owned `saved` and workspace buffers, and the launch sequence of
// the forward and backward passes.
//
// Stage order follows "Scalable Training of Mixture-of-Experts Models with
// Megatron Core", §2: Route -> Dispatch (permute) -> Expert Computation
// (grouped GEMMs) -> Combine; the backward runs the same stages in reverse.
// Nothing here reads device data on the host, so a call is a pure sequence of
// kernel launches (and one status-word memset) on the caller's stream.
#include "internal.h"

#include <cmath>

#include <new>
#include <vector>
#include <string.h>

namespace moe {
namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    int T, R, Rp_max, MT_max, NB;
    // saved
    size_t topk, gates, selsc, counts, kept, poff, meta, tiletab, pairtab, rowof, slotof, eorder, slotlive;
    size_t Xp, A, U, Hh, Yp, As, Us, Hs, saved_bytes;
    // workspace
    size_t status, hist, blkbase, zpart, Ys, dYp, dA, dU, dXp, dz, WrT, wrpart, dAs, dUs, dXs, dgpart, ws_bytes;
    bool fold;   // Hh and Yp live in the workspace (MOE_FLAG_FOLD_GATES)
    bool slotlive_on;   // FP8 recipe with capacity-limited dropping
    // FP8 recipes (saved: permuted activations and, unless the caller passes a
    // weight cache, the weight codes; ws: the rest)
    size_t Xq, sX, wcache;
    size_t hq, sh, dYq, sdY, dAq, sdA, dUq, sdU, hTq, shT, dYpTq, sdYpT, XpTq, sXpT, dATq, sdAT,
        dUTq, sdUT;
    // MXFP8 with a shared expert: its weight codes (saved) and the codes of its
    // dense operands, rows padded to Tp = T rounded up to 128 (workspace)
    int Tp;
    size_t wcache_s, xsq, sxs, hsq, shs, dYsq, sdYs, dYsTq, sdYsT, hsTq, shsT, dAsq, sdAs, dUsq, sdUs,
        dAsTq, sdAsT, dUsTq, sdUsT, xTq, sxT;
    size_t amax;   // NVFP4 tensor maxima (workspace)
    size_t amax_x; // NVFP4 (saved): the maxima of x's tensors (each expert's rows, then the shared
                   // expert's), then those of h, for the backward
};
// NVFP4 tensor maxima in the workspace: h (the backward's g h recomputed
// with folded gates), dY, [dA | dU] per expert, then the shared expert's
// three (the forward's x and h maxima are kept in the saved buffer)
enum { AMAX_H = 0, AMAX_DY = 1, AMAX_DAU = 2, kAmaxKinds = 3 };

// the quantised-expert recipes; the block-scaled ones (MXFP8, NVFP4) share
// the MX layer's stages
bool fp8_recipe(const moe_config_t& c)
{
    return c.dtype == MOE_FP8_BLOCK || c.dtype == MOE_MXFP8 || c.dtype == MOE_NVFP4;
}
bool bs_recipe(const moe_config_t& c) { return c.dtype == MOE_MXFP8 || c.dtype == MOE_NVFP4; }

// The split row tables inside the pair-table block (see make_layout).
struct SplitTabs {
    int* full_tab;
    int* full_off;
    int* tail_tab;
};
SplitTabs split_tabs(const Layout& L, int E, const uint8_t* sv)
{
    int* pairtab = reinterpret_cast<int*>(const_cast<uint8_t*>(sv) + L.pairtab);
    int* full_tab = pairtab + L.MT_max + E + 1;
    int* full_off = full_tab + L.MT_max;
    return {full_tab, full_off, full_off + E + 1};
}

// Quantised expert weights of an FP8 plan (the caller's weight cache, or the
// copy a forward makes in `saved`): for W_gate, W_up (E x H x F) and W_down
// (E x F x H), in this order, q[i] E4M3 codes in the matrix's natural layout
// and s[i] its scales.
//   MOE_FP8_BLOCK: fp32 scales of 128x128 blocks [E][rows/128][cols/128]; the
//     same codes serve the forward GEMMs (read MN-major) and the data-gradient
//     GEMMs (K-major), so q[3..5] = q[0..2].
//   MOE_MXFP8: q[0..2] are the forward orientation (32-element blocks along
//     the matrix's first dimension, the forward GEMM's K, read MN-major) and
//     q[3..5] the data-gradient orientation (blocks along the second
//     dimension, read K-major), each with its UE8M0 scale atoms.
//   MOE_NVFP4: q[0..2] the forward orientation as each expert's transpose
//     (W_gate^T, W_up^T: E x F x H; W_down^T: E x H x F; read K-major), q[3..5]
//     the data-gradient orientation in the natural layout, E2M1 codes two per
//     byte with E4M3 scale atoms; amax: each expert's largest magnitude of
//     [W_gate | W_up] (E floats), then of W_down (E floats).
struct WeightCache {
    size_t q[6], s[6], amax, bytes;
};

// The shared expert as a one-expert layer of width Fs (its weight codes use
// the routed weights' cache layout).
moe_config_t shared_config(const moe_config_t& c)
{
    moe_config_t s = c;
    s.E = 1;
    s.F = c.Fs;
    s.Fs = 0;
    s.top_k = 1;
    return s;
}

WeightCache cache_layout(const moe_config_t& c)
{
    WeightCache W;
    memset(&W, 0, sizeof W);
    if (!fp8_recipe(c)) return W;
    const size_t EHF = (size_t)c.E * c.H * c.F;
    const bool mx = c.dtype == MOE_MXFP8, nv = c.dtype == MOE_NVFP4;
    const size_t sc = nv ? EHF / 16 : mx ? EHF / 32 : 4 * (size_t)(c.H / 128) * (c.F / 128) * c.E;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    for (int i = 0; i < (mx || nv ? 6 : 3); ++i) {
        W.q[i] = take(nv ? EHF / 2 : EHF);
        W.s[i] = take(sc);
    }
    if (!mx && !nv)
        for (int i = 3; i < 6; ++i) { W.q[i] = W.q[i - 3]; W.s[i] = W.s[i - 3]; }
    W.amax = take(nv ? sizeof(float) * 2 * (size_t)c.E : 0);
    W.bytes = o;
    return W;
}

Layout make_layout(const moe_config_t& c, int T)
{
    Layout L;
    const size_t es = (c.dtype == MOE_FP32) ? 4 : 2;   // activations (bf16 for FP8 too)
    L.T = T;
    L.R = T * c.top_k;
    const int nonempty = L.R < c.E ? L.R : c.E;
    L.Rp_max = (int)align_up((size_t)L.R + (size_t)nonempty * (kTileM - 1), kTileM);
    L.MT_max = L.Rp_max / kTileM;
    L.NB = (T + kRouterTokens - 1) / kRouterTokens;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    L.topk = take(sizeof(int) * L.R);
    L.gates = take(sizeof(float) * L.R);
    L.selsc = take(sizeof(float) * L.R);
    L.counts = take(sizeof(int) * c.E);
    L.kept = take(sizeof(int) * c.E);
    L.eorder = take(sizeof(int) * c.E);   // experts, longest padded segment first
    L.poff = take(sizeof(int) * (c.E + 1));
    L.meta = take(sizeof(int) * 8);
    L.tiletab = take(sizeof(int) * L.MT_max);
    // pairs and their E+1 offsets; the pairs of multi-tile experts and their
    // E+1 offsets; the tiles of one-tile experts
    L.pairtab = take(sizeof(int) * (2 * ((size_t)L.MT_max + c.E + 1) + c.E));
    L.rowof = take(sizeof(int) * L.R);
    L.slotof = take(sizeof(int) * L.Rp_max);
    // FP8 recipes with capacity-limited dropping: the slot map of the rows an
    // expert computes (-1 for dropped and pad rows), for the quantisers of the
    // weight-gradient operands
    L.slotlive_on = fp8_recipe(c) && c.capacity_factor > 0.f;
    L.slotlive = take(L.slotlive_on ? sizeof(int) * L.Rp_max : 0);
    // (the FP8 layers keep only the codes of the permuted rows)
    L.Xp = take(fp8_recipe(c) ? 0 : es * L.Rp_max * c.H);
    L.A = take(es * L.Rp_max * c.F);
    L.U = take(es * L.Rp_max * c.F);
    L.fold = (c.flags & MOE_FLAG_FOLD_GATES) != 0;
    L.Hh = take(L.fold ? 0 : es * L.Rp_max * c.F);
    L.Yp = take(L.fold ? 0 : es * L.Rp_max * c.H);
    L.As = take(es * (size_t)T * c.Fs);
    L.Us = take(es * (size_t)T * c.Fs);
    L.Hs = take(es * (size_t)T * c.Fs);
    const bool q8 = c.dtype == MOE_FP8_BLOCK, mx = c.dtype == MOE_MXFP8, nv = c.dtype == MOE_NVFP4;
    const bool bs = mx || nv, anyq = q8 || bs;
    const size_t Rp = L.Rp_max;
    // scale bytes of a codes array: blockwise per 128 values (fp32), MX per
    // 32 (one byte), NVFP4 per 16 (one byte); code bytes: NVFP4 two values a byte
    auto scb = [&](size_t n128) { return q8 ? 4 * n128 : mx ? 4 * n128 : nv ? 8 * n128 : 0; };
    auto cbt = [&](size_t n) { return anyq ? (nv ? n / 2 : n) : 0; };
    L.Xq = take(cbt(Rp * c.H));
    L.sX = take(scb(Rp * (c.H / 128)));
    L.wcache = take(cache_layout(c).bytes);
    const bool mxs = bs && c.Fs > 0;
    L.Tp = (int)align_up((size_t)T, 128);
    L.wcache_s = take(mxs ? cache_layout(shared_config(c)).bytes : 0);
    L.amax_x = take(nv ? sizeof(float) * 2 * ((size_t)c.E + 1) : 0);
    L.saved_bytes = o;
    o = 0;
    L.status = take(256);
    L.hist = take(sizeof(int) * (size_t)L.NB * c.E);
    L.blkbase = take(sizeof(int) * (size_t)L.NB * c.E);
    // partial logits of the H-split router
    L.zpart = take(sizeof(float) * router_zpart_floats(T, c.H, c.E));
    L.Ys = take(c.Fs ? es * (size_t)T * c.H : 0);
    L.dYp = take(es * L.Rp_max * c.H);
    L.dA = take(es * L.Rp_max * c.F);
    L.dU = take(es * L.Rp_max * c.F);
    L.dXp = take(es * L.Rp_max * c.H);
    L.dz = take(sizeof(float) * L.R);
    L.WrT = take(sizeof(float) * (size_t)c.E * c.H);
    L.wrpart = take(sizeof(float) * (size_t)L.MT_max * c.H);
    L.dAs = take(es * (size_t)T * c.Fs);
    L.dUs = take(es * (size_t)T * c.Fs);
    L.dXs = take(c.Fs ? es * (size_t)T * c.H : 0);
    // blockwise: 1x128 row scales, per-column or per-tile transposed scales;
    // MX (NVFP4): one byte per 32 (16) values whatever the orientation
    const size_t RF32 = Rp * c.F / (nv ? 16 : 32), RH32 = Rp * c.H / (nv ? 16 : 32);
    L.hq = take(cbt(Rp * c.F));     L.sh = take(bs ? RF32 : scb(Rp * (c.F / 128)));
    L.dYq = take(cbt(Rp * c.H));    L.sdY = take(bs ? RH32 : scb(Rp * (c.H / 128)));
    L.dAq = take(cbt(Rp * c.F));    L.sdA = take(bs ? RF32 : scb(Rp * (c.F / 128)));
    L.dUq = take(cbt(Rp * c.F));    L.sdU = take(bs ? RF32 : scb(Rp * (c.F / 128)));
    L.hTq = take(cbt(Rp * c.F));    L.shT = take(bs ? RF32 : scb((Rp / 128) * c.F));
    L.dYpTq = take(cbt(Rp * c.H));  L.sdYpT = take(bs ? RH32 : scb((Rp / 128) * (c.H / 128)));
    L.XpTq = take(cbt(Rp * c.H));   L.sXpT = take(bs ? RH32 : scb((Rp / 128) * c.H));
    L.dATq = take(cbt(Rp * c.F));   L.sdAT = take(bs ? RF32 : scb((Rp / 128) * (c.F / 128)));
    L.dgpart = take(L.fold ? sizeof(float) * L.Rp_max * (c.F / 64) : 0);
    if (L.fold) {
        L.Hh = take(es * L.Rp_max * c.F);
        L.Yp = take(es * L.Rp_max * c.H);
    }
    L.dUTq = take(cbt(Rp * c.F));   L.sdUT = take(bs ? RF32 : scb((Rp / 128) * (c.F / 128)));
    {
        const size_t TpH = mxs ? (size_t)L.Tp * c.H : 0, TpF = mxs ? (size_t)L.Tp * c.Fs : 0;
        const size_t vb = nv ? 2 : 1, sb = nv ? 16 : 32;   // values per code byte, per scale byte
        L.xsq = take(TpH / vb);   L.sxs = take(TpH / sb);     // x, rows (shared fc1)
        L.hsq = take(TpF / vb);   L.shs = take(TpF / sb);     // h_s, rows (shared fc2)
        L.dYsq = take(TpH / vb);  L.sdYs = take(TpH / sb);    // dY, rows (shared fc2 dgrad)
        L.dYsTq = take(TpH / vb); L.sdYsT = take(TpH / sb);   // dY, columns (shared fc2 wgrad)
        L.hsTq = take(TpF / vb);  L.shsT = take(TpF / sb);    // h_s, columns
        L.dAsq = take(TpF / vb);  L.sdAs = take(TpF / sb);    // dA_s, dU_s: rows and columns
        L.dUsq = take(TpF / vb);  L.sdUs = take(TpF / sb);
        L.dAsTq = take(TpF / vb); L.sdAsT = take(TpF / sb);
        L.dUsTq = take(TpF / vb); L.sdUsT = take(TpF / sb);
        L.xTq = take(TpH / vb);   L.sxT = take(TpH / sb);     // x, columns (shared fc1 wgrad)
    }
    // NVFP4 tensor maxima of the activations and gradients (per expert: h, dY,
    // [dA | dU]; then the shared expert's), recomputed by each call
    L.amax = take(nv ? sizeof(float) * kAmaxKinds * ((size_t)c.E + 1) : 0);
    L.ws_bytes = o;
    return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows each expert computes under capacity-limited dropping:
// ceil(capacity_factor * T * k / E), or -1 (dropless).
int capacity(const moe_config_t& c, int T)
{
    if (!(c.capacity_factor > 0.f)) return -1;
    const double cap = std::ceil((double)c.capacity_factor * T * c.top_k / c.E);
    return cap > 2147483647.0 ? 2147483647 : (int)cap;
}

moe_status_t check_config(const moe_config_t* c)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->H <= 0 || c->H % 128 || c->E < 1 || c->E > kMaxE || c->F <= 0 || c->F % 128 ||
        c->Fs < 0 || c->Fs % 128 || c->top_k < 1 || c->top_k > kMaxK || c->top_k > c->E ||
        c->T_max < 1 || (c->flags & ~(MOE_FLAG_STAGE_TIMING | MOE_FLAG_FOLD_GATES)) != 0 ||
        !(c->capacity_factor >= 0.f) || !std::isfinite(c->capacity_factor))
        return MOE_ERR_INVALID_ARG;
    if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_FP32 && c->dtype != MOE_BF16 && c->dtype != MOE_FP8_BLOCK && c->dtype != MOE_MXFP8 &&
        c->dtype != MOE_NVFP4)
        return MOE_ERR_INVALID_ARG;
    if (c->dtype == MOE_FP8_BLOCK && c->Fs > 0) return MOE_ERR_UNSUPPORTED;
    // NVFP4 data GEMMs take whole 256-value k blocks of H, F and Fs
    if (c->dtype == MOE_NVFP4 && (c->H % 256 || c->F % 256 || c->Fs % 256)) return MOE_ERR_UNSUPPORTED;
    // int32 row indices: R_pad * max(H, F) elements must stay addressable per
    // buffer with 32-bit row numbers
    const long long R = (long long)c->T_max * c->top_k + (long long)c->E * kTileM;
    if (R > (1ll << 30)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Keeps the caller's current device and switches to the plan's for a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur;
        if (ok && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace
}  // namespace moe

namespace moe {

thread_local unsigned long long t_kernel_launches = 0;

namespace {
enum Stage : int {
    ST_ROUTER, ST_SCAN, ST_INDEX, ST_PERMUTE, ST_FC1, ST_FC2, ST_FC1S, ST_FC2S, ST_COMBINE,
    ST_GATEGRAD, ST_FC2_DGRAD, ST_FC2_WGRAD, ST_FC1_DGRAD, ST_FC1_WGRAD, ST_FC2S_DGRAD,
    ST_FC2S_WGRAD, ST_FC1S_DGRAD, ST_FC1S_WGRAD, ST_ROUTER_WGRAD, ST_TRANSPOSE, ST_UNPERMUTE,
    ST_WQUANT, ST_QROWS, ST_QT, ST_GATEDZ, ST_AMAX, ST_COUNT
};
const char* const kStageNames[ST_COUNT] = {
    "router", "scan", "index", "permute", "fc1_swiglu", "fc2", "shared_fc1_swiglu", "shared_fc2",
    "combine", "gate_grad", "fc2_dgrad_swiglu", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad",
    "shared_fc2_dgrad", "shared_fc2_wgrad", "shared_fc1_dgrad", "shared_fc1_wgrad",
    "router_wgrad", "wr_transpose", "unpermute_reduce", "fp8_weight_quant", "fp8_quant_rows",
    "fp8_quant_t", "gate_dz", "nv_amax"
};
struct StageRec {
    int stage;
    cudaEvent_t start, stop;
    int kernels;   // kernels the stage's call launched
};
}  // namespace
}  // namespace moe

struct moe_plan_s {
    moe_config_t cfg;
    int device;
    int num_sms;
    bool timing;
    std::vector<moe::StageRec> recs;    // recorded since the last moe_stage_times
    std::vector<cudaEvent_t> spare;     // events free for reuse
};

using namespace moe;

// The functions below are declared extern "C" in moe.h, which gives them C linkage.

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "saved or workspace buffer too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side pipeline wait timed out";
    }
    return "unknown status";
}

moe_status_t moe_plan_create(const moe_config_t* cfg, int device, moe_plan_t* out)
{
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return MOE_ERR_CUDA;
    if (device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;   // built for sm_103a only
    {
        DeviceGuard g(device);
        if (!g.ok) return MOE_ERR_CUDA;
        if (cfg->dtype == MOE_BF16 && gemm_tc_prepare(device) != cudaSuccess) return MOE_ERR_CUDA;
        if (cfg->dtype == MOE_FP8_BLOCK && gemm_fp8_prepare(device) != cudaSuccess) return MOE_ERR_CUDA;
        if (cfg->dtype == MOE_MXFP8 && gemm_mx_prepare(device) != cudaSuccess) return MOE_ERR_CUDA;
        if (cfg->dtype == MOE_NVFP4 && gemm_nv_prepare(device) != cudaSuccess) return MOE_ERR_CUDA;
    }
    moe_plan_s* p = new (std::nothrow) moe_plan_s;
    if (!p) return MOE_ERR_CUDA;
    p->cfg = *cfg;
    p->device = device;
    p->num_sms = prop.multiProcessorCount;
    p->timing = (cfg->flags & MOE_FLAG_STAGE_TIMING) != 0;
    *out = p;
    return MOE_OK;
}

moe_status_t moe_plan_destroy(moe_plan_t plan)
{
    if (!plan) return MOE_OK;
    {
        DeviceGuard g(plan->device);
        for (auto& r : plan->recs) {
            cudaEventDestroy(r.start);
            cudaEventDestroy(r.stop);
        }
        for (auto e : plan->spare) cudaEventDestroy(e);
    }
    delete plan;
    return MOE_OK;
}

moe_status_t moe_stage_times(moe_plan_t plan, moe_stage_time_t* out, int capacity, int* count)
{
    if (!plan || !count || capacity < 0 || (capacity > 0 && !out) || !plan->timing)
        return MOE_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return MOE_ERR_CUDA;
    int order[ST_COUNT], n = 0;
    int launches[ST_COUNT] = {0};
    bool seen[ST_COUNT] = {false};
    double ms[ST_COUNT] = {0.0};
    moe_status_t st = MOE_OK;
    for (auto& r : plan->recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            st = MOE_ERR_CUDA;
        if (!seen[r.stage]) {
            seen[r.stage] = true;
            order[n++] = r.stage;
        }
        launches[r.stage] += r.kernels;
        ms[r.stage] += t;
        plan->spare.push_back(r.start);
        plan->spare.push_back(r.stop);
    }
    plan->recs.clear();
    *count = n;
    for (int i = 0; i < n && i < capacity; ++i) {
        memset(out[i].name, 0, sizeof out[i].name);
        strncpy(out[i].name, kStageNames[order[i]], sizeof out[i].name - 1);
        out[i].launches = launches[order[i]];
        out[i].total_ms = (float)ms[order[i]];
    }
    return st;
}

moe_status_t moe_workspace_size(moe_plan_t plan, int T, size_t* saved_bytes, size_t* ws_bytes)
{
    if (!plan || !saved_bytes || !ws_bytes || T < 1 || T > plan->cfg.T_max) return MOE_ERR_INVALID_ARG;
    Layout L = make_layout(plan->cfg, T);
    *saved_bytes = L.saved_bytes;
    *ws_bytes = L.ws_bytes;
    return MOE_OK;
}

#define MOE_CUDA(call)                                   \
    do {                                                 \
        if ((call) != cudaSuccess) return MOE_ERR_CUDA;  \
    } while (0)

// Runs one kernel launch; with stage timing on, brackets it with events.
template <typename Fn>
static cudaError_t run_stage(moe_plan_t p, int stage, cudaStream_t s, Fn&& launch)
{
    if (!p->timing) return launch();
    cudaEvent_t ev[2];
    for (int i = 0; i < 2; ++i) {
        if (!p->spare.empty()) {
            ev[i] = p->spare.back();
            p->spare.pop_back();
        } else if (cudaEventCreate(&ev[i]) != cudaSuccess) {
            return cudaErrorMemoryAllocation;
        }
    }
    cudaError_t e = cudaEventRecord(ev[0], s);
    const unsigned long long n0 = t_kernel_launches;
    if (e == cudaSuccess) e = launch();
    const int kernels = (int)(t_kernel_launches - n0);
    if (e == cudaSuccess) e = cudaEventRecord(ev[1], s);
    p->recs.push_back({stage, ev[0], ev[1], kernels});
    return e;
}
#define MOE_STAGE(stage, call) \
    MOE_CUDA(run_stage(p, stage, s, [&]() -> cudaError_t { return (call); }))

template <typename T>
static moe_status_t forward_impl(moe_plan_t p, int T_, const moe_fwd_args_t* a, uint8_t* sv,
                                 uint8_t* ws, cudaStream_t s)
{
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Fs = c.Fs;
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    int* topk = reinterpret_cast<int*>(sv + L.topk);
    float* gates = reinterpret_cast<float*>(sv + L.gates);
    float* selsc = reinterpret_cast<float*>(sv + L.selsc);
    int* counts = reinterpret_cast<int*>(sv + L.counts);
    int* kept = reinterpret_cast<int*>(sv + L.kept);
    int* poff = reinterpret_cast<int*>(sv + L.poff);
    int* meta = reinterpret_cast<int*>(sv + L.meta);
    int* tiletab = reinterpret_cast<int*>(sv + L.tiletab);
    int* pairtab = reinterpret_cast<int*>(sv + L.pairtab);
    int* rowof = reinterpret_cast<int*>(sv + L.rowof);
    int* slotof = reinterpret_cast<int*>(sv + L.slotof);
    T* Xp = reinterpret_cast<T*>(sv + L.Xp);
    T* A = reinterpret_cast<T*>(sv + L.A);
    T* U = reinterpret_cast<T*>(sv + L.U);
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);
    T* Yp = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Yp);
    T* Ys = Fs ? reinterpret_cast<T*>(ws + L.Ys) : nullptr;
    const T* x = static_cast<const T*>(a->x);

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    MOE_STAGE(ST_ROUTER, launch_router<T>(x, a->Wr, a->b, T_, H, E, k, c.score, topk, gates, selsc,
                              reinterpret_cast<int*>(ws + L.hist), s, a->replay_topk, status,
                              reinterpret_cast<float*>(ws + L.zpart), router_zpart_floats(T_, H, E)));
    const SplitTabs st = split_tabs(L, E, sv);
    MOE_STAGE(ST_SCAN, launch_scan(reinterpret_cast<int*>(ws + L.hist), L.NB, E, counts, poff,
                         reinterpret_cast<int*>(ws + L.blkbase), tiletab, meta, slotof, s, pairtab,
                                   pairtab + L.MT_max, capacity(c, T_), kept,
                                   reinterpret_cast<int*>(sv + L.eorder), st.full_tab, st.full_off,
                                   st.tail_tab));
    MOE_STAGE(ST_INDEX, launch_index(topk, reinterpret_cast<int*>(ws + L.blkbase), T_, E, k, rowof, slotof, s));
    MOE_STAGE(ST_PERMUTE, launch_permute<T>(x, rowof, poff, counts, T_, H, E, k, Xp, s));

    auto gemm = [&](const GemmDesc& d) -> cudaError_t {
        if (c.dtype == MOE_FP32) return launch_gemm_simt_f32(d, L.MT_max, s);
        if (c.dtype == MOE_FP8_BLOCK) return launch_gemm_fp8(d, L.MT_max, p->num_sms, s);
        return launch_gemm_tc_bf16(d, L.MT_max, p->num_sms, s);
    };
    GemmDesc d;
    // fc1 + SwiGLU over the routed rows: [A | U] = Xp [Wg | Wu], Hh = silu(A) U
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_FWD; d.dual = DUAL_N;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.full_tab = st.full_tab; d.full_off = st.full_off; d.tail_tab = st.tail_tab;
    // a pair reads each [Wg | Wu] column tile once for two of an expert's
    // 128-row units; that pays from two units per expert on (the other row
    // GEMMs only from four)
    d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = Xp; d.lda = H; d.a_rows = L.Rp_max;
    d.B0 = a->W_gate; d.B1 = a->W_up; d.ldb = F; d.b_kmajor = 0; d.b_estride = (long long)H * F;
    d.b_rows = E * H;
    d.O0 = A; d.O1 = U; d.O2 = Hh; d.ldo = F; d.status = status;
    if (L.fold) { d.gates = gates; d.slot_of = slotof; }   // Hh = g silu(A) U
    MOE_STAGE(ST_FC1, gemm(d));
    // fc2: Yp = Hh Wd
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_NONE;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.full_tab = st.full_tab; d.full_off = st.full_off; d.tail_tab = st.tail_tab;
    d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = Hh; d.lda = F; d.a_rows = L.Rp_max;
    d.B0 = a->W_down; d.ldb = H; d.b_kmajor = 0; d.b_estride = (long long)F * H; d.b_rows = E * F;
    d.O0 = Yp; d.ldo = H; d.status = status;
    MOE_STAGE(ST_FC2, gemm(d));
    if (Fs) {
        T* As = reinterpret_cast<T*>(sv + L.As);
        T* Us = reinterpret_cast<T*>(sv + L.Us);
        T* Hs = reinterpret_cast<T*>(sv + L.Hs);
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_FWD; d.dual = DUAL_N;
        d.N = Fs; d.K = H; d.E = 1; d.dense_rows = T_;
        d.A0 = x; d.lda = H; d.a_rows = T_;
        d.B0 = a->Ws_gate; d.B1 = a->Ws_up; d.ldb = Fs; d.b_kmajor = 0; d.b_rows = H;
        d.O0 = As; d.O1 = Us; d.O2 = Hs; d.ldo = Fs; d.status = status;
        MOE_STAGE(ST_FC1S, gemm(d));
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_NONE;
        d.N = H; d.K = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = Hs; d.lda = Fs; d.a_rows = T_;
        d.B0 = a->Ws_down; d.ldb = H; d.b_kmajor = 0; d.b_rows = Fs;
        d.O0 = Ys; d.ldo = H; d.status = status;
        MOE_STAGE(ST_FC2S, gemm(d));
    }
    MOE_STAGE(ST_COMBINE, launch_combine<T>(Yp, Ys, rowof, L.fold ? nullptr : gates, T_, H, k,
                                            static_cast<T*>(a->y), s));

    if (a->topk_idx) MOE_CUDA(cudaMemcpyAsync(a->topk_idx, topk, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->gates) MOE_CUDA(cudaMemcpyAsync(a->gates, gates, sizeof(float) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->counts) MOE_CUDA(cudaMemcpyAsync(a->counts, counts, sizeof(int) * E, cudaMemcpyDeviceToDevice, s));
    if (a->offsets) MOE_CUDA(cudaMemcpyAsync(a->offsets, poff, sizeof(int) * (E + 1), cudaMemcpyDeviceToDevice, s));
    if (a->row_of) MOE_CUDA(cudaMemcpyAsync(a->row_of, rowof, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

template <typename T>
static moe_status_t backward_impl(moe_plan_t p, int T_, const moe_bwd_args_t* a, const uint8_t* svc,
                                  uint8_t* ws, cudaStream_t s)
{
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Fs = c.Fs;
    uint8_t* sv = const_cast<uint8_t*>(svc);   // only read below
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    const int* topk = reinterpret_cast<const int*>(sv + L.topk);
    const float* gates = reinterpret_cast<const float*>(sv + L.gates);
    const float* selsc = reinterpret_cast<const float*>(sv + L.selsc);
    const int* counts = reinterpret_cast<const int*>(sv + L.counts);
    const int* kept = reinterpret_cast<const int*>(sv + L.kept);
    const int* poff = reinterpret_cast<const int*>(sv + L.poff);
    const int* meta = reinterpret_cast<const int*>(sv + L.meta);
    const int* tiletab = reinterpret_cast<const int*>(sv + L.tiletab);
    const int* pairtab = reinterpret_cast<const int*>(sv + L.pairtab);
    const SplitTabs st = split_tabs(L, E, sv);
    const int* eorder = reinterpret_cast<const int*>(sv + L.eorder);
    const int* rowof = reinterpret_cast<const int*>(sv + L.rowof);
    const int* slotof = reinterpret_cast<const int*>(sv + L.slotof);
    const T* Xp = reinterpret_cast<const T*>(sv + L.Xp);
    const T* A = reinterpret_cast<const T*>(sv + L.A);
    const T* U = reinterpret_cast<const T*>(sv + L.U);
    // folded gates: Hh is recomputed into the workspace, Yp is not needed
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);
    const T* Yp = reinterpret_cast<const T*>(sv + L.Yp);
    T* dYp = reinterpret_cast<T*>(ws + L.dYp);
    T* dA = reinterpret_cast<T*>(ws + L.dA);
    T* dU = reinterpret_cast<T*>(ws + L.dU);
    T* dXp = reinterpret_cast<T*>(ws + L.dXp);
    float* dz = reinterpret_cast<float*>(ws + L.dz);
    float* WrT = reinterpret_cast<float*>(ws + L.WrT);
    float* dgpart = reinterpret_cast<float*>(ws + L.dgpart);
    const T* dY = static_cast<const T*>(a->dY);

    auto gemm = [&](const GemmDesc& d) -> cudaError_t {
        if (c.dtype == MOE_FP32) return launch_gemm_simt_f32(d, L.MT_max, s);
        if (c.dtype == MOE_FP8_BLOCK) return launch_gemm_fp8(d, L.MT_max, p->num_sms, s);
        return launch_gemm_tc_bf16(d, L.MT_max, p->num_sms, s);
    };

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    // Combine backward: gate gradients, gate-scaled output gradients, router
    // dz; with folded gates only the permuted copy of dY (dg and dz follow
    // from the fc2-dgrad epilogue)
    if (L.fold)
        MOE_STAGE(ST_GATEGRAD, launch_permute<T>(dY, rowof, poff, counts, T_, H, E, k, dYp, s));
    else
        MOE_STAGE(ST_GATEGRAD, launch_gate_grad<T>(dY, Yp, rowof, topk, gates, selsc, poff, counts, T_, H,
                                                   E, k, c.score, dYp, dz, s));
    GemmDesc d;
    // fc2 dgrad + SwiGLU backward: dh = dYp Wd^T -> dA, dU
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_BWD; d.dual = DUAL_NONE;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.full_tab = st.full_tab; d.full_off = st.full_off; d.tail_tab = st.tail_tab;
    d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = dYp; d.lda = H; d.a_rows = L.Rp_max;
    d.B0 = a->W_down; d.ldb = H; d.b_kmajor = 1; d.b_estride = (long long)F * H; d.b_rows = E * F;
    d.X0 = A; d.X1 = U; d.O0 = dA; d.O1 = dU; d.ldo = F; d.status = status;
    if (L.fold) {
        d.gates = gates; d.slot_of = slotof; d.dg_part = dgpart; d.dg_ld = F / 64;
        d.O2 = Hh;   // g h, recomputed for the fc2 weight gradient
    }
    MOE_STAGE(ST_FC2_DGRAD, gemm(d));
    if (L.fold)
        MOE_STAGE(ST_GATEDZ, launch_gate_dz(dgpart, F / 64, rowof, gates, selsc, T_, k, c.score, dz, s));
    // fc2 wgrad: dWd[e] = Hh_e^T dYp_e
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_NONE;
    d.N = H; d.M_out = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = Hh; d.lda = F; d.a_rows = L.Rp_max;
    d.B0 = dYp; d.ldb = H; d.b_rows = L.Rp_max;
    d.O0 = a->dW_down; d.ldo = H; d.o_estride = (long long)F * H; d.status = status;
    d.expert_order = eorder;
    MOE_STAGE(ST_FC2_WGRAD, gemm(d));
    // fc1 dgrad: dXp = dA Wg^T + dU Wu^T
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_K;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.full_tab = st.full_tab; d.full_off = st.full_off; d.tail_tab = st.tail_tab;
    d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = dA; d.A1 = dU; d.lda = F; d.a_rows = L.Rp_max;
    d.B0 = a->W_gate; d.B1 = a->W_up; d.ldb = F; d.b_kmajor = 1; d.b_estride = (long long)H * F;
    d.b_rows = E * H;
    d.O0 = dXp; d.ldo = H; d.status = status;
    MOE_STAGE(ST_FC1_DGRAD, gemm(d));
    // fc1 wgrad: dWg[e] = Xp_e^T dA_e, dWu[e] = Xp_e^T dU_e
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_N;
    d.N = F; d.M_out = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept; d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max;
    d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = Xp; d.lda = H; d.a_rows = L.Rp_max;
    d.B0 = dA; d.B1 = dU; d.ldb = F; d.b_rows = L.Rp_max;
    d.O0 = a->dW_gate; d.O1 = a->dW_up; d.ldo = F; d.o_estride = (long long)H * F; d.status = status;
    d.expert_order = eorder;
    MOE_STAGE(ST_FC1_WGRAD, gemm(d));

    T* dXs = nullptr;
    if (Fs) {
        const T* As = reinterpret_cast<const T*>(sv + L.As);
        const T* Us = reinterpret_cast<const T*>(sv + L.Us);
        const T* Hs = reinterpret_cast<const T*>(sv + L.Hs);
        T* dAs = reinterpret_cast<T*>(ws + L.dAs);
        T* dUs = reinterpret_cast<T*>(ws + L.dUs);
        dXs = reinterpret_cast<T*>(ws + L.dXs);
        // shared expert: its output gradient is dY itself (unweighted add)
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_BWD; d.dual = DUAL_NONE;
        d.N = Fs; d.K = H; d.E = 1; d.dense_rows = T_;
        d.A0 = dY; d.lda = H; d.a_rows = T_;
        d.B0 = a->Ws_down; d.ldb = H; d.b_kmajor = 1; d.b_rows = Fs;
        d.X0 = As; d.X1 = Us; d.O0 = dAs; d.O1 = dUs; d.ldo = Fs; d.status = status;
        MOE_STAGE(ST_FC2S_DGRAD, gemm(d));
        memset(&d, 0, sizeof d);
        d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_NONE;
        d.N = H; d.M_out = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = Hs; d.lda = Fs; d.a_rows = T_;
        d.B0 = dY; d.ldb = H; d.b_rows = T_;
        d.O0 = a->dWs_down; d.ldo = H; d.status = status;
        MOE_STAGE(ST_FC2S_WGRAD, gemm(d));
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_K;
        d.N = H; d.K = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = dAs; d.A1 = dUs; d.lda = Fs; d.a_rows = T_;
        d.B0 = a->Ws_gate; d.B1 = a->Ws_up; d.ldb = Fs; d.b_kmajor = 1; d.b_rows = H;
        d.O0 = dXs; d.ldo = H; d.status = status;
        MOE_STAGE(ST_FC1S_DGRAD, gemm(d));
        memset(&d, 0, sizeof d);
        d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_N;
        d.N = Fs; d.M_out = H; d.E = 1; d.dense_rows = T_;
        d.A0 = a->x; d.lda = H; d.a_rows = T_;
        d.B0 = dAs; d.B1 = dUs; d.ldb = Fs; d.b_rows = T_;
        d.O0 = a->dWs_gate; d.O1 = a->dWs_up; d.ldo = Fs; d.status = status;
        MOE_STAGE(ST_FC1S_WGRAD, gemm(d));
    }
    // router backward and the unpermute-reduce of dX
    MOE_STAGE(ST_ROUTER_WGRAD, launch_router_wgrad<T>(static_cast<const T*>(a->x), slotof, poff, meta,
                                   L.MT_max, dz, H, E, k, reinterpret_cast<float*>(ws + L.wrpart), a->dWr, s));
    MOE_STAGE(ST_TRANSPOSE, launch_transpose_f32(a->Wr, H, E, WrT, s));
    MOE_STAGE(ST_UNPERMUTE, launch_unpermute_reduce<T>(dXp, dXs, rowof, topk, dz, WrT, T_, H, k,
                                        static_cast<T*>(a->dX), s));
    return MOE_OK;
}

// ---------------------------------------------------------- blockwise FP8
// E4M3 weight codes and scales a call uses: the caller's cache, or the copy
// the forward quantises into `saved`.
struct WQ {
    uint8_t* q[6];   // gate, up, down: forward orientation, then data-gradient orientation
    void* s[6];
    float* amax;     // NVFP4: per expert, [W_gate | W_up] then W_down
};
static WQ codes_at(const moe_config_t& c, uint8_t* b)
{
    WQ w;
    const WeightCache C = cache_layout(c);
    for (int i = 0; i < 6; ++i) {
        w.q[i] = b + C.q[i];
        w.s[i] = b + C.s[i];
    }
    w.amax = reinterpret_cast<float*>(b + C.amax);
    return w;
}
static WQ weight_codes(const moe_config_t& c, const Layout& L, uint8_t* sv, const void* cache)
{
    return codes_at(c, cache ? static_cast<uint8_t*>(const_cast<void*>(cache)) : sv + L.wcache);
}

// Quantise W_gate, W_up, W_down into the weight codes w (both orientations).
static cudaError_t quantize_weights(const moe_config_t& c, const void* Wg, const void* Wu, const void* Wd,
                                    const WQ& w, cudaStream_t s)
{
    using T = __nv_bfloat16;
    const int E = c.E, H = c.H, F = c.F;
    const void* W[3] = {Wg, Wu, Wd};
    const int R[3] = {H, H, F}, Cc[3] = {F, F, H};
    if (c.dtype == MOE_NVFP4) {
        // each expert's tensor maxima ([W_gate | W_up] into one), then one pass
        // per matrix: row codes (the data-gradient orientation) and each
        // expert's transposed codes (the forward orientation, K-major)
        cudaError_t e = cudaMemsetAsync(w.amax, 0, sizeof(float) * 2 * (size_t)E, s);
        NvQuantJob j[3];
        for (int i = 0; i < 3 && e == cudaSuccess; ++i) {
            memset(&j[i], 0, sizeof j[i]);
            j[i].in = static_cast<const T*>(W[i]);
            j[i].rows_max = E * R[i];
            j[i].C = Cc[i];
            j[i].rows_cap = E * R[i];
            j[i].q = w.q[3 + i];
            j[i].sf = static_cast<uint8_t*>(w.s[3 + i]);
            j[i].qc = w.q[i];
            j[i].sfc = static_cast<uint8_t*>(w.s[i]);
            j[i].grp = R[i];
            j[i].seg_rows = R[i];
            j[i].gather_k = 1;
            j[i].amax = w.amax + (i == 2 ? E : 0);
            e = launch_nv_amax(j[i], w.amax + (i == 2 ? E : 0), s);
        }
        for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = launch_nv_quant(j[i], s);
        return e;
    }
    for (int i = 0; i < 3; ++i) {
        cudaError_t e;
        if (c.dtype == MOE_MXFP8) {
            // one pass: row codes (the data-gradient orientation) and in-place
            // column codes (the forward orientation, K = R[i] per expert)
            MxQuantJob j{static_cast<const T*>(W[i]), nullptr, E * R[i], Cc[i], 128, w.q[3 + i],
                         static_cast<uint8_t*>(w.s[3 + i]), w.q[i], static_cast<uint8_t*>(w.s[i]), 2};
            j.grp = R[i];
            e = launch_mx_quant(j, s);
        } else {
            e = launch_quant(QuantJob{static_cast<const T*>(W[i]), nullptr, E * R[i], Cc[i], 128, w.q[i],
                                      static_cast<float*>(w.s[i]), 1, nullptr, nullptr, 0}, s);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Same stages as the bf16 layer; the expert GEMMs take E4M3 operands with
// fp32 block scales (A: 1x128 along K, B: 128x128), all K-major, produced by
// the quantisers in quant.cu; intermediates and outputs stay bf16.
static moe_status_t forward_fp8_impl(moe_plan_t p, int T_, const moe_fwd_args_t* a, uint8_t* sv,
                                     uint8_t* ws, cudaStream_t s)
{
    using T = __nv_bfloat16;
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Rp = L.Rp_max;
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    int* topk = reinterpret_cast<int*>(sv + L.topk);
    float* gates = reinterpret_cast<float*>(sv + L.gates);
    float* selsc = reinterpret_cast<float*>(sv + L.selsc);
    int* counts = reinterpret_cast<int*>(sv + L.counts);
    int* kept = reinterpret_cast<int*>(sv + L.kept);
    int* poff = reinterpret_cast<int*>(sv + L.poff);
    int* meta = reinterpret_cast<int*>(sv + L.meta);
    int* tiletab = reinterpret_cast<int*>(sv + L.tiletab);
    int* pairtab = reinterpret_cast<int*>(sv + L.pairtab);
    int* rowof = reinterpret_cast<int*>(sv + L.rowof);
    int* slotof = reinterpret_cast<int*>(sv + L.slotof);
    T* A = reinterpret_cast<T*>(sv + L.A);
    T* U = reinterpret_cast<T*>(sv + L.U);
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);
    T* Yp = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Yp);
    auto u8 = [&](uint8_t* base, size_t off) { return base + off; };
    auto f32 = [&](uint8_t* base, size_t off) { return reinterpret_cast<float*>(base + off); };
    const T* x = static_cast<const T*>(a->x);

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    MOE_STAGE(ST_ROUTER, launch_router<T>(x, a->Wr, a->b, T_, H, E, k, c.score, topk, gates, selsc,
                                          reinterpret_cast<int*>(ws + L.hist), s, a->replay_topk, status,
                                          reinterpret_cast<float*>(ws + L.zpart),
                                          router_zpart_floats(T_, H, E)));
    MOE_STAGE(ST_SCAN, launch_scan(reinterpret_cast<int*>(ws + L.hist), L.NB, E, counts, poff,
                                   reinterpret_cast<int*>(ws + L.blkbase), tiletab, meta, slotof, s, pairtab,
                                   pairtab + L.MT_max, capacity(c, T_), kept,
                                   reinterpret_cast<int*>(sv + L.eorder)));
    int* slotlive = L.slotlive_on ? reinterpret_cast<int*>(sv + L.slotlive) : nullptr;
    if (slotlive) MOE_CUDA(cudaMemsetAsync(slotlive, 0xFF, sizeof(int) * (size_t)L.Rp_max, s));
    MOE_STAGE(ST_INDEX, launch_index(topk, reinterpret_cast<int*>(ws + L.blkbase), T_, E, k, rowof, slotof, s,
                                     poff, kept, slotlive));
    MOE_STAGE(ST_PERMUTE, launch_permute_quant(x, rowof, poff, counts, T_, H, E, k, nullptr, u8(sv, L.Xq),
                                               f32(sv, L.sX), s));
    // one orientation of the weight codes: the forward GEMMs read them
    // MN-major, the data-gradient GEMMs K-major. Pre-quantised weights
    // (moe_quantize_weights) are read from the caller's cache; otherwise the
    // bf16 weights are quantised into the saved buffer for this step.
    const WQ wq = weight_codes(c, L, sv, a->weight_cache);
    if (!a->weight_cache)
        MOE_STAGE(ST_WQUANT, quantize_weights(c, a->W_gate, a->W_up, a->W_down, wq, s));
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_FWD; d.dual = DUAL_N;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(sv, L.Xq); d.lda = H; d.a_rows = Rp; d.SA0 = f32(sv, L.sX); d.lds_a = H / 128;
    d.B0 = wq.q[0]; d.B1 = wq.q[1]; d.ldb = F; d.b_rows = E * H; d.b_kmajor = 0;
    d.SB0 = static_cast<float*>(wq.s[0]); d.SB1 = static_cast<float*>(wq.s[1]);
    d.O0 = A; d.O1 = U; d.O2 = Hh; d.ldo = F; d.status = status;
    if (L.fold) { d.gates = gates; d.slot_of = slotof; }   // Hh = g silu(A) U
    MOE_STAGE(ST_FC1, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    MOE_STAGE(ST_QROWS, launch_quant(QuantJob{Hh, meta + 1, Rp, F, Rp, u8(ws, L.hq), f32(ws, L.sh), 0,
                                              nullptr, nullptr, 0}, s));
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_NONE;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(ws, L.hq); d.lda = F; d.a_rows = Rp; d.SA0 = f32(ws, L.sh); d.lds_a = F / 128;
    d.B0 = wq.q[2]; d.ldb = H; d.b_rows = E * F; d.SB0 = static_cast<float*>(wq.s[2]); d.b_kmajor = 0;
    d.O0 = Yp; d.ldo = H; d.status = status;
    MOE_STAGE(ST_FC2, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    MOE_STAGE(ST_COMBINE, launch_combine<T>(Yp, nullptr, rowof, L.fold ? nullptr : gates, T_, H, k,
                                            static_cast<T*>(a->y), s));

    if (a->topk_idx) MOE_CUDA(cudaMemcpyAsync(a->topk_idx, topk, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->gates) MOE_CUDA(cudaMemcpyAsync(a->gates, gates, sizeof(float) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->counts) MOE_CUDA(cudaMemcpyAsync(a->counts, counts, sizeof(int) * E, cudaMemcpyDeviceToDevice, s));
    if (a->offsets) MOE_CUDA(cudaMemcpyAsync(a->offsets, poff, sizeof(int) * (E + 1), cudaMemcpyDeviceToDevice, s));
    if (a->row_of) MOE_CUDA(cudaMemcpyAsync(a->row_of, rowof, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

static moe_status_t backward_fp8_impl(moe_plan_t p, int T_, const moe_bwd_args_t* a,
                                      const uint8_t* svc, uint8_t* ws, cudaStream_t s)
{
    using T = __nv_bfloat16;
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Rp = L.Rp_max;
    uint8_t* sv = const_cast<uint8_t*>(svc);   // only read below
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    const int* topk = reinterpret_cast<const int*>(sv + L.topk);
    const float* gates = reinterpret_cast<const float*>(sv + L.gates);
    const float* selsc = reinterpret_cast<const float*>(sv + L.selsc);
    const int* counts = reinterpret_cast<const int*>(sv + L.counts);
    const int* kept = reinterpret_cast<const int*>(sv + L.kept);
    const int* poff = reinterpret_cast<const int*>(sv + L.poff);
    const int* meta = reinterpret_cast<const int*>(sv + L.meta);
    const int* tiletab = reinterpret_cast<const int*>(sv + L.tiletab);
    const int* pairtab = reinterpret_cast<const int*>(sv + L.pairtab);
    const int* rowof = reinterpret_cast<const int*>(sv + L.rowof);
    const int* slotof = reinterpret_cast<const int*>(sv + L.slotof);
    // rows of dropped assignments: zero output gradients, no part in the quantisation blocks
    const int* slotlive = L.slotlive_on ? reinterpret_cast<const int*>(sv + L.slotlive) : nullptr;
    const T* A = reinterpret_cast<const T*>(sv + L.A);
    const T* U = reinterpret_cast<const T*>(sv + L.U);
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);   // folded: recomputed below
    const T* Yp = reinterpret_cast<const T*>(sv + L.Yp);
    T* dYp = reinterpret_cast<T*>(ws + L.dYp);
    T* dA = reinterpret_cast<T*>(ws + L.dA);
    T* dU = reinterpret_cast<T*>(ws + L.dU);
    T* dXp = reinterpret_cast<T*>(ws + L.dXp);
    float* dz = reinterpret_cast<float*>(ws + L.dz);
    float* WrT = reinterpret_cast<float*>(ws + L.WrT);
    float* dgpart = reinterpret_cast<float*>(ws + L.dgpart);
    auto u8 = [&](uint8_t* base, size_t off) { return base + off; };
    auto f32 = [&](uint8_t* base, size_t off) { return reinterpret_cast<float*>(base + off); };
    const T* dY = static_cast<const T*>(a->dY);
    const WQ wq = weight_codes(c, L, sv, a->weight_cache);

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    if (L.fold)
        MOE_STAGE(ST_GATEGRAD, launch_permute<T>(dY, rowof, poff, counts, T_, H, E, k, dYp, s, slotlive));
    else
        MOE_STAGE(ST_GATEGRAD, launch_gate_grad<T>(dY, Yp, rowof, topk, gates, selsc, poff, counts, T_, H,
                                                   E, k, c.score, dYp, dz, s, slotlive));
    // fc2 dgrad + SwiGLU backward
    // dYp once: 1x128 row codes (fc2 dgrad) and transposed 128x128-tile codes (fc2 wgrad)
    MOE_STAGE(ST_QROWS, launch_quant(QuantJob{dYp, meta + 1, Rp, H, Rp, u8(ws, L.dYq), f32(ws, L.sdY), 0,
                                              u8(ws, L.dYpTq), f32(ws, L.sdYpT), 1}, s));
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_BWD; d.dual = DUAL_NONE;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(ws, L.dYq); d.lda = H; d.a_rows = Rp; d.SA0 = f32(ws, L.sdY); d.lds_a = H / 128;
    d.B0 = wq.q[5]; d.ldb = H; d.b_rows = E * F; d.SB0 = static_cast<float*>(wq.s[5]); d.b_kmajor = 1;
    d.X0 = A; d.X1 = U; d.O0 = dA; d.O1 = dU; d.ldo = F; d.status = status;
    if (L.fold) {
        d.gates = gates; d.slot_of = slotof; d.dg_part = dgpart; d.dg_ld = F / 64;
        d.O2 = Hh;   // g h, recomputed for the fc2 weight gradient
    }
    MOE_STAGE(ST_FC2_DGRAD, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    if (L.fold)
        MOE_STAGE(ST_GATEDZ, launch_gate_dz(dgpart, F / 64, rowof, gates, selsc, T_, k, c.score, dz, s));
    // fc2 wgrad: dWd[e] = h_e^T dYp_e
    MOE_STAGE(ST_QT, launch_quant(QuantJob{Hh, meta + 1, Rp, F, Rp, nullptr, nullptr, 0, u8(ws, L.hTq),
                                           f32(ws, L.shT), 0}, s));
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_NONE;
    d.N = H; d.M_out = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(ws, L.hTq); d.lda = Rp; d.SA0 = f32(ws, L.shT); d.lds_a = Rp / 128;
    d.B0 = u8(ws, L.dYpTq); d.ldb = Rp; d.SB0 = f32(ws, L.sdYpT); d.lds_b = Rp / 128;
    d.rows_cap = Rp;
    d.O0 = a->dW_down; d.ldo = H; d.o_estride = (long long)F * H; d.status = status;
    MOE_STAGE(ST_FC2_WGRAD, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    // fc1 dgrad: dXp = dA Wg^T + dU Wu^T
    // dA, dU once each: row codes (fc1 dgrad) and transposed tile codes (fc1 wgrad)
    MOE_STAGE(ST_QROWS, launch_quant(QuantJob{dA, meta + 1, Rp, F, Rp, u8(ws, L.dAq), f32(ws, L.sdA), 0,
                                              u8(ws, L.dATq), f32(ws, L.sdAT), 1}, s));
    MOE_STAGE(ST_QROWS, launch_quant(QuantJob{dU, meta + 1, Rp, F, Rp, u8(ws, L.dUq), f32(ws, L.sdU), 0,
                                              u8(ws, L.dUTq), f32(ws, L.sdUT), 1}, s));
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_K;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(ws, L.dAq); d.A1 = u8(ws, L.dUq); d.lda = F; d.a_rows = Rp;
    d.SA0 = f32(ws, L.sdA); d.SA1 = f32(ws, L.sdU); d.lds_a = F / 128;
    d.B0 = wq.q[3]; d.B1 = wq.q[4]; d.ldb = F; d.b_rows = E * H; d.b_kmajor = 1;
    d.SB0 = static_cast<float*>(wq.s[3]); d.SB1 = static_cast<float*>(wq.s[4]);
    d.O0 = dXp; d.ldo = H; d.status = status;
    MOE_STAGE(ST_FC1_DGRAD, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    // fc1 wgrad: dWg[e] = Xp_e^T dA_e, dWu[e] = Xp_e^T dU_e
    // the permuted rows are token rows of x (no bf16 copy of them is kept)
    MOE_STAGE(ST_QT, launch_quant(QuantJob{static_cast<const T*>(a->x), meta + 1, Rp, H, Rp, nullptr,
                                           nullptr, 0, u8(ws, L.XpTq), f32(ws, L.sXpT), 0,
                                           slotlive ? slotlive : slotof, k}, s));
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_N;
    d.N = F; d.M_out = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 512ll * E;
    d.A0 = u8(ws, L.XpTq); d.lda = Rp; d.SA0 = f32(ws, L.sXpT); d.lds_a = Rp / 128;
    d.B0 = u8(ws, L.dATq); d.B1 = u8(ws, L.dUTq); d.ldb = Rp;
    d.SB0 = f32(ws, L.sdAT); d.SB1 = f32(ws, L.sdUT); d.lds_b = Rp / 128;
    d.rows_cap = Rp;
    d.O0 = a->dW_gate; d.O1 = a->dW_up; d.ldo = F; d.o_estride = (long long)H * F; d.status = status;
    MOE_STAGE(ST_FC1_WGRAD, launch_gemm_fp8(d, L.MT_max, p->num_sms, s));
    // router backward and the unpermute-reduce of dX
    MOE_STAGE(ST_ROUTER_WGRAD, launch_router_wgrad<T>(static_cast<const T*>(a->x), slotof, poff, meta,
                                   L.MT_max, dz, H, E, k, reinterpret_cast<float*>(ws + L.wrpart), a->dWr, s));
    MOE_STAGE(ST_TRANSPOSE, launch_transpose_f32(a->Wr, H, E, WrT, s));
    MOE_STAGE(ST_UNPERMUTE, launch_unpermute_reduce<T>(dXp, nullptr, rowof, topk, dz, WrT, T_, H, k,
                                                       static_cast<T*>(a->dX), s));
    return MOE_OK;
}

// ------------------------------------------------------- MXFP8 and NVFP4
// The blockwise-FP8 layer's stages with the MXFP8 recipe: every GEMM operand
// is quantised in 32-element blocks along the GEMM's K with power-of-two
// scales (quant_mx.cu), so the activations and gradients that feed a data
// GEMM and a weight-gradient GEMM get one quantisation per orientation, like
// the weights, and the grouped GEMMs apply the scales in the tensor cores.
// NVFP4 takes the same stages with 16-value E2M1 blocks (quant_nv.cu,
// gemm_nv.cu); each tensor first gets its largest magnitude (a maximum pass
// per expert segment, stage nv_amax), for its fp32 tensor scale, and every
// GEMM reads its weights K-major.

// NVFP4 quantisation job over the routed rows (one tensor per expert
// segment) or over a dense group of T rows padded to Tp
static NvQuantJob nv_job(const Layout& L, int T_, const int* meta, const int* poff, int E, bool dense,
                         const __nv_bfloat16* in, int C, uint8_t* q, uint8_t* sf, uint8_t* qc, uint8_t* sfc,
                         const float* amax)
{
    NvQuantJob j;
    memset(&j, 0, sizeof j);
    j.in = in;
    j.C = C;
    j.q = q; j.sf = sf; j.qc = qc; j.sfc = sfc;
    j.gather_k = 1;
    j.amax = amax;
    if (dense) {
        j.rows_max = j.rows_cap = j.grp = L.Tp;
        j.rows_valid = T_;
    } else {
        j.rows_dev = meta + 1;
        j.rows_max = j.rows_cap = j.grp = L.Rp_max;
        j.seg_off = poff;
        j.nseg = E;
    }
    return j;
}

static moe_status_t forward_mx_impl(moe_plan_t p, int T_, const moe_fwd_args_t* a, uint8_t* sv,
                                    uint8_t* ws, cudaStream_t s)
{
    using T = __nv_bfloat16;
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Rp = L.Rp_max;
    const bool nv = c.dtype == MOE_NVFP4;
    auto gemm = [&](const GemmDesc& g) {
        return nv ? launch_gemm_nv(g, L.MT_max, p->num_sms, s) : launch_gemm_mx(g, L.MT_max, p->num_sms, s);
    };
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    int* topk = reinterpret_cast<int*>(sv + L.topk);
    float* gates = reinterpret_cast<float*>(sv + L.gates);
    float* selsc = reinterpret_cast<float*>(sv + L.selsc);
    int* counts = reinterpret_cast<int*>(sv + L.counts);
    int* kept = reinterpret_cast<int*>(sv + L.kept);
    int* poff = reinterpret_cast<int*>(sv + L.poff);
    int* meta = reinterpret_cast<int*>(sv + L.meta);
    int* tiletab = reinterpret_cast<int*>(sv + L.tiletab);
    int* pairtab = reinterpret_cast<int*>(sv + L.pairtab);
    int* rowof = reinterpret_cast<int*>(sv + L.rowof);
    int* slotof = reinterpret_cast<int*>(sv + L.slotof);
    T* A = reinterpret_cast<T*>(sv + L.A);
    T* U = reinterpret_cast<T*>(sv + L.U);
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);
    T* Yp = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Yp);
    const T* x = static_cast<const T*>(a->x);

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    MOE_STAGE(ST_ROUTER, launch_router<T>(x, a->Wr, a->b, T_, H, E, k, c.score, topk, gates, selsc,
                                          reinterpret_cast<int*>(ws + L.hist), s, a->replay_topk, status,
                                          reinterpret_cast<float*>(ws + L.zpart),
                                          router_zpart_floats(T_, H, E)));
    MOE_STAGE(ST_SCAN, launch_scan(reinterpret_cast<int*>(ws + L.hist), L.NB, E, counts, poff,
                                   reinterpret_cast<int*>(ws + L.blkbase), tiletab, meta, slotof, s, pairtab,
                                   pairtab + L.MT_max, capacity(c, T_), kept,
                                   reinterpret_cast<int*>(sv + L.eorder)));
    int* slotlive = L.slotlive_on ? reinterpret_cast<int*>(sv + L.slotlive) : nullptr;
    if (slotlive) MOE_CUDA(cudaMemsetAsync(slotlive, 0xFF, sizeof(int) * (size_t)L.Rp_max, s));
    MOE_STAGE(ST_INDEX, launch_index(topk, reinterpret_cast<int*>(ws + L.blkbase), T_, E, k, rowof, slotof, s,
                                     poff, kept, slotlive));
    // x's and h's maxima, kept for the backward
    float* amx = nv ? reinterpret_cast<float*>(sv + L.amax_x) : nullptr;
    float* amh = nv ? amx + E + 1 : nullptr;
    if (nv) {
        // each expert's maximum over the rows it keeps, then every token's k
        // rows in their experts' tensor scales (x read twice, not gathered)
        MOE_CUDA(cudaMemsetAsync(amx, 0, sizeof(float) * 2 * ((size_t)E + 1), s));
        MOE_STAGE(ST_PERMUTE, launch_nv_permute(x, topk, rowof, poff, counts, kept, T_, H, E, k, amx, sv + L.Xq,
                                                sv + L.sX, s));
    } else {
        MOE_STAGE(ST_PERMUTE, launch_mx_permute(x, rowof, poff, counts, T_, H, E, k, sv + L.Xq, sv + L.sX, s));
    }
    const WQ wq = weight_codes(c, L, sv, a->weight_cache);
    if (!a->weight_cache)
        MOE_STAGE(ST_WQUANT, quantize_weights(c, a->W_gate, a->W_up, a->W_down, wq, s));
    auto xs = [](void* v) { return static_cast<const uint8_t*>(v); };
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_FWD; d.dual = DUAL_N;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = sv + L.Xq; d.lda = H; d.a_rows = Rp; d.XA0 = sv + L.sX;
    d.B0 = wq.q[0]; d.B1 = wq.q[1]; d.ldb = F; d.b_rows = E * H; d.b_kmajor = 0;
    d.XB0 = xs(wq.s[0]); d.XB1 = xs(wq.s[1]);
    d.O0 = A; d.O1 = U; d.O2 = Hh; d.ldo = F; d.status = status;
    if (L.fold) { d.gates = gates; d.slot_of = slotof; }   // Hh = g silu(A) U
    if (nv) {   // [Wg^T | Wu^T] K-major; the epilogue folds each expert's max |h| into amh
        d.nv = 1; d.gA = amx; d.gB = wq.amax; d.amaxO = amh;
        d.ldb = H; d.b_rows = E * F; d.b_kmajor = 1;
    } else {
        d.Qrows = ws + L.hq; d.Qatoms = ws + L.sh;          // fc2's A operand, from the epilogue
    }
    MOE_STAGE(ST_FC1, gemm(d));
    if (nv)
        MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, false, Hh, F, ws + L.hq, ws + L.sh, nullptr,
                                                   nullptr, amh), s));
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_NONE;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = ws + L.hq; d.lda = F; d.a_rows = Rp; d.XA0 = ws + L.sh;
    d.B0 = wq.q[2]; d.ldb = H; d.b_rows = E * F; d.XB0 = xs(wq.s[2]); d.b_kmajor = 0;
    if (nv) {   // Wd^T K-major
        d.nv = 1; d.gA = amh; d.gB = wq.amax + E;
        d.ldb = F; d.b_rows = E * H; d.b_kmajor = 1;
    }
    d.O0 = Yp; d.ldo = H; d.status = status;
    MOE_STAGE(ST_FC2, gemm(d));
    T* Ys = nullptr;
    if (c.Fs) {
        // the shared expert: a dense group of the T token rows (padded to Tp
        // in its codes), its weights quantised like a one-expert layer's
        const moe_config_t cs = shared_config(c);
        const WQ wqs = codes_at(cs, sv + L.wcache_s);
        const int Fs = c.Fs, Tp = L.Tp;
        T* As = reinterpret_cast<T*>(sv + L.As);
        T* Us = reinterpret_cast<T*>(sv + L.Us);
        T* Hs = reinterpret_cast<T*>(sv + L.Hs);
        Ys = reinterpret_cast<T*>(ws + L.Ys);
        MOE_STAGE(ST_WQUANT, quantize_weights(cs, a->Ws_gate, a->Ws_up, a->Ws_down, wqs, s));
        if (nv) {
            NvQuantJob j = nv_job(L, T_, meta, poff, E, true, x, H, ws + L.xsq, ws + L.sxs, nullptr, nullptr,
                                  amx + E);
            MOE_STAGE(ST_AMAX, launch_nv_amax(j, amx + E, s));
            MOE_STAGE(ST_QROWS, launch_nv_quant(j, s));
        } else {
            MxQuantJob j{x, nullptr, Tp, H, Tp, ws + L.xsq, ws + L.sxs, nullptr, nullptr, 0};
            j.rows_valid = T_;
            MOE_STAGE(ST_QROWS, launch_mx_quant(j, s));
        }
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_FWD; d.dual = DUAL_N;
        d.N = Fs; d.K = H; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.xsq; d.lda = H; d.a_rows = Tp; d.XA0 = ws + L.sxs;
        d.B0 = wqs.q[0]; d.B1 = wqs.q[1]; d.ldb = Fs; d.b_rows = H; d.b_kmajor = 0;
        d.XB0 = xs(wqs.s[0]); d.XB1 = xs(wqs.s[1]);
        d.O0 = As; d.O1 = Us; d.O2 = Hs; d.ldo = Fs; d.status = status;
        if (nv) {
            d.nv = 1; d.gA = amx + E; d.gB = wqs.amax; d.amaxO = amh + E;
            d.ldb = H; d.b_rows = Fs; d.b_kmajor = 1;
        } else {
            d.Qrows = ws + L.hsq; d.Qatoms = ws + L.shs;          // shared fc2's A operand
        }
        MOE_STAGE(ST_FC1S, gemm(d));
        if (nv)
            MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, true, Hs, Fs, ws + L.hsq, ws + L.shs,
                                                       nullptr, nullptr, amh + E), s));
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_NONE;
        d.N = H; d.K = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.hsq; d.lda = Fs; d.a_rows = Tp; d.XA0 = ws + L.shs;
        d.B0 = wqs.q[2]; d.ldb = H; d.b_rows = Fs; d.XB0 = xs(wqs.s[2]); d.b_kmajor = 0;
        if (nv) {
            d.nv = 1; d.gA = amh + E; d.gB = wqs.amax + 1;
            d.ldb = Fs; d.b_rows = H; d.b_kmajor = 1;
        }
        d.O0 = Ys; d.ldo = H; d.status = status;
        MOE_STAGE(ST_FC2S, gemm(d));
    }
    MOE_STAGE(ST_COMBINE, launch_combine<T>(Yp, Ys, rowof, L.fold ? nullptr : gates, T_, H, k,
                                            static_cast<T*>(a->y), s));

    if (a->topk_idx) MOE_CUDA(cudaMemcpyAsync(a->topk_idx, topk, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->gates) MOE_CUDA(cudaMemcpyAsync(a->gates, gates, sizeof(float) * L.R, cudaMemcpyDeviceToDevice, s));
    if (a->counts) MOE_CUDA(cudaMemcpyAsync(a->counts, counts, sizeof(int) * E, cudaMemcpyDeviceToDevice, s));
    if (a->offsets) MOE_CUDA(cudaMemcpyAsync(a->offsets, poff, sizeof(int) * (E + 1), cudaMemcpyDeviceToDevice, s));
    if (a->row_of) MOE_CUDA(cudaMemcpyAsync(a->row_of, rowof, sizeof(int) * L.R, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

static moe_status_t backward_mx_impl(moe_plan_t p, int T_, const moe_bwd_args_t* a,
                                     const uint8_t* svc, uint8_t* ws, cudaStream_t s)
{
    using T = __nv_bfloat16;
    const moe_config_t& c = p->cfg;
    const Layout L = make_layout(c, T_);
    const int H = c.H, E = c.E, k = c.top_k, F = c.F, Rp = L.Rp_max;
    uint8_t* sv = const_cast<uint8_t*>(svc);   // only read below
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(ws + L.status);
    const int* topk = reinterpret_cast<const int*>(sv + L.topk);
    const float* gates = reinterpret_cast<const float*>(sv + L.gates);
    const float* selsc = reinterpret_cast<const float*>(sv + L.selsc);
    const int* counts = reinterpret_cast<const int*>(sv + L.counts);
    const int* kept = reinterpret_cast<const int*>(sv + L.kept);
    const int* poff = reinterpret_cast<const int*>(sv + L.poff);
    const int* meta = reinterpret_cast<const int*>(sv + L.meta);
    const int* tiletab = reinterpret_cast<const int*>(sv + L.tiletab);
    const int* pairtab = reinterpret_cast<const int*>(sv + L.pairtab);
    const int* eorder = reinterpret_cast<const int*>(sv + L.eorder);
    const int* rowof = reinterpret_cast<const int*>(sv + L.rowof);
    const int* slotof = reinterpret_cast<const int*>(sv + L.slotof);
    // rows of dropped assignments: zero output gradients, no part in the quantisation blocks
    const int* slotlive = L.slotlive_on ? reinterpret_cast<const int*>(sv + L.slotlive) : nullptr;
    const T* A = reinterpret_cast<const T*>(sv + L.A);
    const T* U = reinterpret_cast<const T*>(sv + L.U);
    T* Hh = reinterpret_cast<T*>((L.fold ? ws : sv) + L.Hh);   // folded: recomputed below
    const T* Yp = reinterpret_cast<const T*>(sv + L.Yp);
    T* dYp = reinterpret_cast<T*>(ws + L.dYp);
    T* dA = reinterpret_cast<T*>(ws + L.dA);
    T* dU = reinterpret_cast<T*>(ws + L.dU);
    T* dXp = reinterpret_cast<T*>(ws + L.dXp);
    float* dz = reinterpret_cast<float*>(ws + L.dz);
    float* WrT = reinterpret_cast<float*>(ws + L.WrT);
    float* dgpart = reinterpret_cast<float*>(ws + L.dgpart);
    const T* dY = static_cast<const T*>(a->dY);
    const WQ wq = weight_codes(c, L, sv, a->weight_cache);
    auto xs = [](void* v) { return static_cast<const uint8_t*>(v); };
    const bool nv = c.dtype == MOE_NVFP4;
    float* am = nv ? reinterpret_cast<float*>(ws + L.amax) : nullptr;   // [3][E], then the shared expert's
    auto gemm = [&](const GemmDesc& g) {
        return nv ? launch_gemm_nv(g, L.MT_max, p->num_sms, s) : launch_gemm_mx(g, L.MT_max, p->num_sms, s);
    };
    // NVFP4: each tensor's maximum (one array for a pair that shares a
    // tensor scale), then its codes
    auto nvq = [&](const NvQuantJob& j, int stage) -> moe_status_t {
        MOE_STAGE(ST_AMAX, launch_nv_amax(j, const_cast<float*>(j.amax), s));
        MOE_STAGE(stage, launch_nv_quant(j, s));
        return MOE_OK;
    };
    if (nv) MOE_CUDA(cudaMemsetAsync(am, 0, sizeof(float) * kAmaxKinds * ((size_t)E + 1), s));
    // the forward's x and h maxima
    const float* amx = nv ? reinterpret_cast<const float*>(sv + L.amax_x) : nullptr;
    const float* amh = nv ? amx + E + 1 : nullptr;
    // h of the fc2 weight gradient: the forward's, or g h recomputed by the
    // fc2-dgrad epilogue (folded gates), which also takes its maxima
    const float* amh_b = nv ? (L.fold ? am + AMAX_H * E : amh) : nullptr;

    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s));
    if (L.fold)
        MOE_STAGE(ST_GATEGRAD, launch_permute<T>(dY, rowof, poff, counts, T_, H, E, k, dYp, s, slotlive));
    else
        MOE_STAGE(ST_GATEGRAD, launch_gate_grad<T>(dY, Yp, rowof, topk, gates, selsc, poff, counts, T_, H,
                                                   E, k, c.score, dYp, dz, s, slotlive));
    // dYp once: row codes (fc2 dgrad, K = H) and transposed column codes (fc2 wgrad, K = tokens)
    if (nv) {
        const moe_status_t r = nvq(nv_job(L, T_, meta, poff, E, false, dYp, H, ws + L.dYq, ws + L.sdY, ws + L.dYpTq,
                                          ws + L.sdYpT, am + AMAX_DY * E), ST_QROWS);
        if (r != MOE_OK) return r;
    } else {
        MxQuantJob j{dYp, meta + 1, Rp, H, Rp, ws + L.dYq, ws + L.sdY, ws + L.dYpTq, ws + L.sdYpT, 1};
        MOE_STAGE(ST_QROWS, launch_mx_quant(j, s));
    }
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_BWD; d.dual = DUAL_NONE;
    d.N = F; d.K = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = ws + L.dYq; d.lda = H; d.a_rows = Rp; d.XA0 = ws + L.sdY;
    d.B0 = wq.q[5]; d.ldb = H; d.b_rows = E * F; d.XB0 = xs(wq.s[5]); d.b_kmajor = 1;
    d.X0 = A; d.X1 = U; d.O0 = dA; d.O1 = dU; d.ldo = F; d.status = status;
    if (L.fold) {
        d.gates = gates; d.slot_of = slotof; d.dg_part = dgpart; d.dg_ld = F / 64;
        d.O2 = Hh;   // g h, recomputed for the fc2 weight gradient
    }
    if (nv) {   // the epilogue folds each expert's max |dA|, |dU| (and |g h|) into the workspace
        d.nv = 1; d.gA = am + AMAX_DY * E; d.gB = wq.amax + E;
        d.amaxO = am + AMAX_DAU * E;
        if (L.fold) d.amaxO2 = am + AMAX_H * E;
    }
    MOE_STAGE(ST_FC2_DGRAD, gemm(d));
    if (L.fold)
        MOE_STAGE(ST_GATEDZ, launch_gate_dz(dgpart, F / 64, rowof, gates, selsc, T_, k, c.score, dz, s));
    // fc2 wgrad: dWd[e] = h_e^T dYp_e
    if (nv) {
        MOE_STAGE(ST_QT, launch_nv_quant(nv_job(L, T_, meta, poff, E, false, Hh, F, nullptr, nullptr, ws + L.hTq,
                                                ws + L.shT, amh_b), s));
    } else {
        MxQuantJob j{Hh, meta + 1, Rp, F, Rp, nullptr, nullptr, ws + L.hTq, ws + L.shT, 1};
        MOE_STAGE(ST_QT, launch_mx_quant(j, s));
    }
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_NONE;
    d.N = H; d.M_out = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = ws + L.hTq; d.lda = Rp; d.XA0 = ws + L.shT;
    d.B0 = ws + L.dYpTq; d.ldb = Rp; d.XB0 = ws + L.sdYpT;
    d.rows_cap = Rp; d.expert_order = eorder;
    d.O0 = a->dW_down; d.ldo = H; d.o_estride = (long long)F * H; d.status = status;
    if (nv) { d.nv = 1; d.gA = amh_b; d.gB = am + AMAX_DY * E; }
    MOE_STAGE(ST_FC2_WGRAD, gemm(d));
    // dA, dU once each: row codes (fc1 dgrad, K = F) and transposed column codes (fc1 wgrad)
    if (nv) {   // one tensor [dA | dU] per expert, its maxima from the fc2-dgrad epilogue
        const float* g = am + AMAX_DAU * E;
        MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, false, dA, F, ws + L.dAq, ws + L.sdA,
                                                   ws + L.dATq, ws + L.sdAT, g), s));
        MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, false, dU, F, ws + L.dUq, ws + L.sdU,
                                                   ws + L.dUTq, ws + L.sdUT, g), s));
    } else {
        MxQuantJob ja{dA, meta + 1, Rp, F, Rp, ws + L.dAq, ws + L.sdA, ws + L.dATq, ws + L.sdAT, 1};
        MOE_STAGE(ST_QROWS, launch_mx_quant(ja, s));
        MxQuantJob ju{dU, meta + 1, Rp, F, Rp, ws + L.dUq, ws + L.sdU, ws + L.dUTq, ws + L.sdUT, 1};
        MOE_STAGE(ST_QROWS, launch_mx_quant(ju, s));
    }
    memset(&d, 0, sizeof d);
    d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_K;
    d.N = H; d.K = F; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = ws + L.dAq; d.A1 = ws + L.dUq; d.lda = F; d.a_rows = Rp;
    d.XA0 = ws + L.sdA; d.XA1 = ws + L.sdU;
    d.B0 = wq.q[3]; d.B1 = wq.q[4]; d.ldb = F; d.b_rows = E * H; d.b_kmajor = 1;
    d.XB0 = xs(wq.s[3]); d.XB1 = xs(wq.s[4]);
    d.O0 = dXp; d.ldo = H; d.status = status;
    if (nv) { d.nv = 1; d.gA = am + AMAX_DAU * E; d.gB = wq.amax; }
    MOE_STAGE(ST_FC1_DGRAD, gemm(d));
    // fc1 wgrad: the permuted rows are token rows of x (no bf16 copy of them is kept)
    if (nv) {
        NvQuantJob j = nv_job(L, T_, meta, poff, E, false, static_cast<const T*>(a->x), H, nullptr, nullptr,
                              ws + L.XpTq, ws + L.sXpT, amx);
        j.gather_slot = slotlive ? slotlive : slotof;
        j.gather_k = k;
        MOE_STAGE(ST_QT, launch_nv_quant(j, s));
    } else {
        MxQuantJob j{static_cast<const T*>(a->x), meta + 1, Rp, H, Rp, nullptr, nullptr, ws + L.XpTq,
                     ws + L.sXpT, 1};
        j.gather_slot = slotlive ? slotlive : slotof;
        j.gather_k = k;
        MOE_STAGE(ST_QT, launch_mx_quant(j, s));
    }
    memset(&d, 0, sizeof d);
    d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_N;
    d.N = F; d.M_out = H; d.E = E;
    d.tile_tab = tiletab; d.meta = meta; d.poff = poff; d.counts = kept;
    d.pair_tab = pairtab; d.pair_off = pairtab + L.MT_max; d.prefer_pair = (long long)T_ * k >= 256ll * E;
    d.A0 = ws + L.XpTq; d.lda = Rp; d.XA0 = ws + L.sXpT;
    d.B0 = ws + L.dATq; d.B1 = ws + L.dUTq; d.ldb = Rp;
    d.XB0 = ws + L.sdAT; d.XB1 = ws + L.sdUT;
    d.rows_cap = Rp; d.expert_order = eorder;
    d.O0 = a->dW_gate; d.O1 = a->dW_up; d.ldo = F; d.o_estride = (long long)H * F; d.status = status;
    if (nv) { d.nv = 1; d.gA = amx; d.gB = am + AMAX_DAU * E; }
    MOE_STAGE(ST_FC1_WGRAD, gemm(d));
    T* dXs = nullptr;
    if (c.Fs) {
        // the shared expert's backward; its output gradient is dY itself
        const moe_config_t cs = shared_config(c);
        const WQ wqs = codes_at(cs, sv + L.wcache_s);
        const int Fs = c.Fs, Tp = L.Tp;
        const T* As = reinterpret_cast<const T*>(sv + L.As);
        const T* Us = reinterpret_cast<const T*>(sv + L.Us);
        const T* Hs = reinterpret_cast<const T*>(sv + L.Hs);
        T* dAs = reinterpret_cast<T*>(ws + L.dAs);
        T* dUs = reinterpret_cast<T*>(ws + L.dUs);
        dXs = reinterpret_cast<T*>(ws + L.dXs);
        float* ams = nv ? am + kAmaxKinds * E : nullptr;   // the shared expert's h, dY, [dA | dU]
        // dY: row codes (shared fc2 dgrad, K = H), column codes (shared fc2 wgrad, K = tokens)
        if (nv) {
            const moe_status_t r = nvq(nv_job(L, T_, meta, poff, E, true, dY, H, ws + L.dYsq, ws + L.sdYs,
                                              ws + L.dYsTq, ws + L.sdYsT, ams + AMAX_DY), ST_QROWS);
            if (r != MOE_OK) return r;
        } else {
            MxQuantJob j{dY, nullptr, Tp, H, Tp, ws + L.dYsq, ws + L.sdYs, ws + L.dYsTq, ws + L.sdYsT, 1};
            j.rows_valid = T_;
            MOE_STAGE(ST_QROWS, launch_mx_quant(j, s));
        }
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_SWIGLU_BWD; d.dual = DUAL_NONE;
        d.N = Fs; d.K = H; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.dYsq; d.lda = H; d.a_rows = Tp; d.XA0 = ws + L.sdYs;
        d.B0 = wqs.q[5]; d.ldb = H; d.b_rows = Fs; d.XB0 = xs(wqs.s[5]); d.b_kmajor = 1;
        d.X0 = As; d.X1 = Us; d.O0 = dAs; d.O1 = dUs; d.ldo = Fs; d.status = status;
        if (nv) { d.nv = 1; d.gA = ams + AMAX_DY; d.gB = wqs.amax + 1; d.amaxO = ams + AMAX_DAU; }
        MOE_STAGE(ST_FC2S_DGRAD, gemm(d));
        if (nv) {
            MOE_STAGE(ST_QT, launch_nv_quant(nv_job(L, T_, meta, poff, E, true, Hs, Fs, nullptr, nullptr,
                                                    ws + L.hsTq, ws + L.shsT, amh + E), s));
        } else {
            MxQuantJob j{Hs, nullptr, Tp, Fs, Tp, nullptr, nullptr, ws + L.hsTq, ws + L.shsT, 1};
            j.rows_valid = T_;
            MOE_STAGE(ST_QT, launch_mx_quant(j, s));
        }
        memset(&d, 0, sizeof d);
        d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_NONE;
        d.N = H; d.M_out = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.hsTq; d.lda = Tp; d.XA0 = ws + L.shsT;
        d.B0 = ws + L.dYsTq; d.ldb = Tp; d.XB0 = ws + L.sdYsT;
        d.rows_cap = Tp;
        d.O0 = a->dWs_down; d.ldo = H; d.o_estride = (long long)Fs * H; d.status = status;
        if (nv) { d.nv = 1; d.gA = amh + E; d.gB = ams + AMAX_DY; }
        MOE_STAGE(ST_FC2S_WGRAD, gemm(d));
        if (nv) {
            const float* g = ams + AMAX_DAU;
            MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, true, dAs, Fs, ws + L.dAsq, ws + L.sdAs,
                                                       ws + L.dAsTq, ws + L.sdAsT, g), s));
            MOE_STAGE(ST_QROWS, launch_nv_quant(nv_job(L, T_, meta, poff, E, true, dUs, Fs, ws + L.dUsq, ws + L.sdUs,
                                                       ws + L.dUsTq, ws + L.sdUsT, g), s));
        } else {
            MxQuantJob ja{dAs, nullptr, Tp, Fs, Tp, ws + L.dAsq, ws + L.sdAs, ws + L.dAsTq, ws + L.sdAsT, 1};
            ja.rows_valid = T_;
            MOE_STAGE(ST_QROWS, launch_mx_quant(ja, s));
            MxQuantJob ju{dUs, nullptr, Tp, Fs, Tp, ws + L.dUsq, ws + L.sdUs, ws + L.dUsTq, ws + L.sdUsT, 1};
            ju.rows_valid = T_;
            MOE_STAGE(ST_QROWS, launch_mx_quant(ju, s));
        }
        memset(&d, 0, sizeof d);
        d.sched = SCHED_ROWS; d.epi = EPI_STORE; d.dual = DUAL_K;
        d.N = H; d.K = Fs; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.dAsq; d.A1 = ws + L.dUsq; d.lda = Fs; d.a_rows = Tp;
        d.XA0 = ws + L.sdAs; d.XA1 = ws + L.sdUs;
        d.B0 = wqs.q[3]; d.B1 = wqs.q[4]; d.ldb = Fs; d.b_rows = H; d.b_kmajor = 1;
        d.XB0 = xs(wqs.s[3]); d.XB1 = xs(wqs.s[4]);
        d.O0 = dXs; d.ldo = H; d.status = status;
        if (nv) { d.nv = 1; d.gA = ams + AMAX_DAU; d.gB = wqs.amax; }
        MOE_STAGE(ST_FC1S_DGRAD, gemm(d));
        if (nv) {
            MOE_STAGE(ST_QT, launch_nv_quant(nv_job(L, T_, meta, poff, E, true, static_cast<const T*>(a->x), H,
                                                    nullptr, nullptr, ws + L.xTq, ws + L.sxT, amx + E), s));
        } else {
            MxQuantJob j{static_cast<const T*>(a->x), nullptr, Tp, H, Tp, nullptr, nullptr, ws + L.xTq,
                         ws + L.sxT, 1};
            j.rows_valid = T_;
            MOE_STAGE(ST_QT, launch_mx_quant(j, s));
        }
        memset(&d, 0, sizeof d);
        d.sched = SCHED_WGRAD; d.epi = EPI_WGRAD; d.dual = DUAL_N;
        d.N = Fs; d.M_out = H; d.E = 1; d.dense_rows = T_;
        d.A0 = ws + L.xTq; d.lda = Tp; d.XA0 = ws + L.sxT;
        d.B0 = ws + L.dAsTq; d.B1 = ws + L.dUsTq; d.ldb = Tp;
        d.XB0 = ws + L.sdAsT; d.XB1 = ws + L.sdUsT;
        d.rows_cap = Tp;
        d.O0 = a->dWs_gate; d.O1 = a->dWs_up; d.ldo = Fs; d.o_estride = (long long)H * Fs; d.status = status;
        if (nv) { d.nv = 1; d.gA = amx + E; d.gB = ams + AMAX_DAU; }
        MOE_STAGE(ST_FC1S_WGRAD, gemm(d));
    }
    MOE_STAGE(ST_ROUTER_WGRAD, launch_router_wgrad<T>(static_cast<const T*>(a->x), slotof, poff, meta,
                                   L.MT_max, dz, H, E, k, reinterpret_cast<float*>(ws + L.wrpart), a->dWr, s));
    MOE_STAGE(ST_TRANSPOSE, launch_transpose_f32(a->Wr, H, E, WrT, s));
    MOE_STAGE(ST_UNPERMUTE, launch_unpermute_reduce<T>(dXp, dXs, rowof, topk, dz, WrT, T_, H, k,
                                                       static_cast<T*>(a->dX), s));
    return MOE_OK;
}

static moe_status_t check_call(moe_plan_t plan, int T, const void* saved, size_t saved_bytes,
                               const void* ws, size_t ws_bytes)
{
    if (!plan || T < 1 || T > plan->cfg.T_max || !saved || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(saved) || !aligned16(ws)) return MOE_ERR_MISALIGNED;
    Layout L = make_layout(plan->cfg, T);
    if (saved_bytes < L.saved_bytes || ws_bytes < L.ws_bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

moe_status_t moe_forward(moe_plan_t plan, int T, const moe_fwd_args_t* a, void* saved,
                         size_t saved_bytes, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!a) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_call(plan, T, saved, saved_bytes, ws, ws_bytes);
    if (st != MOE_OK) return st;
    const bool shared = plan->cfg.Fs > 0;
    // a weight cache (FP8 plans only) replaces the bf16 expert weights
    if (a->weight_cache && !fp8_recipe(plan->cfg)) return MOE_ERR_INVALID_ARG;
    const bool wneed = a->weight_cache == nullptr;
    if (!a->x || !a->Wr || (wneed && (!a->W_gate || !a->W_up || !a->W_down)) || !a->y)
        return MOE_ERR_INVALID_ARG;
    if (shared != (a->Ws_gate != nullptr) || shared != (a->Ws_up != nullptr) ||
        shared != (a->Ws_down != nullptr))
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {a->x, a->Wr, a->b, a->W_gate, a->W_up, a->W_down, a->Ws_gate, a->Ws_up,
                          a->Ws_down, a->y, a->topk_idx, a->gates, a->counts, a->offsets, a->row_of,
                          a->weight_cache};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_MISALIGNED;
    DeviceGuard g(plan->device);
    if (!g.ok) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan->cfg.dtype == MOE_FP32)
        return forward_impl<float>(plan, T, a, static_cast<uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    if (plan->cfg.dtype == MOE_FP8_BLOCK)
        return forward_fp8_impl(plan, T, a, static_cast<uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    if (bs_recipe(plan->cfg))
        return forward_mx_impl(plan, T, a, static_cast<uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    return forward_impl<__nv_bfloat16>(plan, T, a, static_cast<uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
}

moe_status_t moe_backward(moe_plan_t plan, int T, const moe_bwd_args_t* a, const void* saved,
                          size_t saved_bytes, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!a) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_call(plan, T, saved, saved_bytes, ws, ws_bytes);
    if (st != MOE_OK) return st;
    const bool shared = plan->cfg.Fs > 0;
    if (a->weight_cache && !fp8_recipe(plan->cfg)) return MOE_ERR_INVALID_ARG;
    const bool wneed = a->weight_cache == nullptr;
    if (!a->dY || !a->x || !a->Wr || (wneed && (!a->W_gate || !a->W_up || !a->W_down)) || !a->dX ||
        !a->dWr || !a->dW_gate || !a->dW_up || !a->dW_down)
        return MOE_ERR_INVALID_ARG;
    const void* sh[] = {a->Ws_gate, a->Ws_up, a->Ws_down, a->dWs_gate, a->dWs_up, a->dWs_down};
    for (const void* q : sh)
        if (shared != (q != nullptr)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {a->dY, a->x, a->Wr, a->W_gate, a->W_up, a->W_down, a->Ws_gate,
                          a->Ws_up, a->Ws_down, a->dX, a->dWr, a->dW_gate, a->dW_up, a->dW_down,
                          a->dWs_gate, a->dWs_up, a->dWs_down, a->weight_cache};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_MISALIGNED;
    DeviceGuard g(plan->device);
    if (!g.ok) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan->cfg.dtype == MOE_FP32)
        return backward_impl<float>(plan, T, a, static_cast<const uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    if (plan->cfg.dtype == MOE_FP8_BLOCK)
        return backward_fp8_impl(plan, T, a, static_cast<const uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    if (bs_recipe(plan->cfg))
        return backward_mx_impl(plan, T, a, static_cast<const uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
    return backward_impl<__nv_bfloat16>(plan, T, a, static_cast<const uint8_t*>(saved), static_cast<uint8_t*>(ws), s);
}

moe_status_t moe_read_status(moe_plan_t plan, const void* ws, moe_stream_t stream)
{
    if (!plan || !ws) return MOE_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    DeviceStatus h;
    if (cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    return h.code == 0 ? MOE_OK : static_cast<moe_status_t>(h.code);
}

bool moe::plan_info(const moe_plan_s* plan, moe_config_t* cfg, int* device)
{
    if (!plan) return false;
    *cfg = plan->cfg;
    *device = plan->device;
    return true;
}

moe_status_t moe_fp8_quantize(int rows, int cols, int mode, const void* in, uint8_t* codes,
                              float* scales, uint8_t* codes_t, float* scales_t, moe_stream_t stream)
{
    if (rows < 1 || cols < 1 || rows % 128 || cols % 128 || !in) return MOE_ERR_INVALID_ARG;
    if (!aligned16(in) || (codes && !aligned16(codes)) || (codes_t && !aligned16(codes_t)))
        return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(in);
    cudaError_t e;
    switch (mode) {
    case MOE_Q_ROWS:
    case MOE_Q_TILES: {
        if (!codes || !scales) return MOE_ERR_INVALID_ARG;
        const bool t = codes_t && scales_t;   // also the transposed 128x128-tile codes
        e = launch_quant(QuantJob{x, nullptr, rows, cols, rows, codes, scales, mode == MOE_Q_TILES ? 1 : 0,
                                  t ? codes_t : nullptr, t ? scales_t : nullptr, 1}, s);
        break;
    }
    case MOE_Q_COLS_T:
    case MOE_Q_TILES_T:
        if (!codes_t || !scales_t) return MOE_ERR_INVALID_ARG;
        e = launch_quant(QuantJob{x, nullptr, rows, cols, rows, nullptr, nullptr, 0, codes_t, scales_t,
                                  mode == MOE_Q_TILES_T ? 1 : 0}, s);
        break;
    default:
        return MOE_ERR_INVALID_ARG;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_weight_cache_size(moe_plan_t plan, size_t* bytes)
{
    if (!plan || !bytes) return MOE_ERR_INVALID_ARG;
    *bytes = cache_layout(plan->cfg).bytes;
    return MOE_OK;
}

moe_status_t moe_quantize_weights(moe_plan_t plan, const void* W_gate, const void* W_up,
                                  const void* W_down, void* cache, size_t cache_bytes,
                                  moe_stream_t stream)
{
    if (!plan || !W_gate || !W_up || !W_down || !cache) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = plan->cfg;
    if (!fp8_recipe(c)) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(cache))
        return MOE_ERR_MISALIGNED;
    if (cache_bytes < cache_layout(c).bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceGuard g(plan->device);
    if (!g.ok) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Layout L;
    memset(&L, 0, sizeof L);
    const WQ w = weight_codes(c, L, nullptr, cache);
    return quantize_weights(c, W_gate, W_up, W_down, w, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_mx_quantize(int rows, int cols, const void* in, uint8_t* codes, uint8_t* scales,
                             uint8_t* codes_c, uint8_t* scales_c, int col_transposed, moe_stream_t stream)
{
    if (rows < 1 || cols < 1 || rows % 128 || cols % 128 || !in) return MOE_ERR_INVALID_ARG;
    if ((codes == nullptr) != (scales == nullptr) || (codes_c == nullptr) != (scales_c == nullptr) ||
        (!codes && !codes_c) || (col_transposed != 0 && col_transposed != 1))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(in) || (codes && !aligned16(codes)) || (codes_c && !aligned16(codes_c)))
        return MOE_ERR_MISALIGNED;
    MxQuantJob j{static_cast<const __nv_bfloat16*>(in), nullptr, rows, cols, rows, codes, scales, codes_c,
                 scales_c, col_transposed ? 1 : 2};
    j.grp = rows;
    const cudaError_t e = launch_mx_quant(j, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_nv_quantize(int rows, int cols, const void* in, float* amax, uint8_t* codes, uint8_t* scales,
                             uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream)
{
    if (rows < 1 || cols < 1 || rows % 128 || cols % 128 || !in || !amax) return MOE_ERR_INVALID_ARG;
    if ((codes == nullptr) != (scales == nullptr) || (codes_t == nullptr) != (scales_t == nullptr) ||
        (!codes && !codes_t))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(in) || (codes && !aligned16(codes)) || (codes_t && !aligned16(codes_t)) ||
        (reinterpret_cast<uintptr_t>(amax) & 3u))
        return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NvQuantJob j;
    memset(&j, 0, sizeof j);
    j.in = static_cast<const __nv_bfloat16*>(in);
    j.rows_max = j.rows_cap = j.grp = rows;
    j.C = cols;
    j.q = codes; j.sf = scales; j.qc = codes_t; j.sfc = scales_t;
    j.gather_k = 1;
    j.amax = amax;
    if (cudaMemsetAsync(amax, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_nv_amax(j, amax, s) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_nv_quant(j, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
