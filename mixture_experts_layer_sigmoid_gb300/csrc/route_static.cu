// route_static.cu -- moe_route_static: the routing step (router logits,
// top-k, gates, per-expert counts, padded offsets, row_of) for callers that
// cannot hand this library a scratch buffer.
//
// Who needs it: code whose device memory is entirely owned by someone else
// -- a framework's caching pool, or an inference service that reserves a
// fixed memory budget at start-up and forbids growth afterwards -- and code
// in latency-critical loops that must not call cudaMalloc, which can
// synchronise the device. Such callers can still pass their input and
// output tensors, but cannot obtain the extra workspace that moe_forward
// needs for its per-block expert histograms, block bases, tile table and
// row->slot map.
//
// Those scratch arrays live here instead, in one file-scope __device__
// array of kStaticScratchBytes. It belongs to the library's module, so
// every GPU on which the library is loaded keeps that memory until the
// process exits. Its size bounds the token count one call can route (see
// static_bytes); larger calls are rejected before anything is launched.
//
// The host never names the array directly as a pointer: its device address
// is looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call on that device.
#include "internal.h"

#include <mutex>

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_route_scratch on the current device `device`.
cudaError_t scratch_address(int device, void** out)
{
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

struct StaticLayout {
    size_t selsc, hist, blkbase, tiletab, meta, slotof, zpart, bytes;
};

// Offsets of the routing scratch inside the static array for T tokens.
StaticLayout static_layout(const moe_config_t& c, int T)
{
    StaticLayout L;
    const size_t R = (size_t)T * c.top_k;
    const size_t nonempty = R < (size_t)c.E ? R : (size_t)c.E;
    const size_t Rp = (R + nonempty * (kTileM - 1) + kTileM - 1) / kTileM * kTileM;
    const size_t nb = (T + kRouterTokens - 1) / kRouterTokens;
    size_t o = 0;
    L.selsc = o;   o = up256(o + sizeof(float) * R);
    L.hist = o;    o = up256(o + sizeof(int) * nb * c.E);
    L.blkbase = o; o = up256(o + sizeof(int) * nb * c.E);
    L.tiletab = o; o = up256(o + sizeof(int) * (Rp / kTileM));
    L.meta = o;    o = up256(o + sizeof(int) * 4);
    L.slotof = o;  o = up256(o + sizeof(int) * Rp);
    L.zpart = o;   o = up256(o + sizeof(float) * router_zpart_floats(T, c.H, c.E));
    L.bytes = o;
    return L;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

moe_status_t moe_route_static(moe_plan_t plan, int T, const void* x, const float* Wr,
                              const float* b, int32_t* topk_idx, float* gates, int32_t* counts,
                              int32_t* offsets, int32_t* row_of, moe_stream_t stream)
{
    moe_config_t c;
    int device = -1;
    if (!plan_info(plan, &c, &device)) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > c.T_max || !x || !Wr || !topk_idx || !gates || !counts || !offsets || !row_of)
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, Wr, b, topk_idx, gates, counts, offsets, row_of};
    for (const void* p : ptrs)
        if (p && !al16(p)) return MOE_ERR_MISALIGNED;
    const StaticLayout L = static_layout(c, T);
    if (L.bytes > kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status_t st = MOE_OK;
    void* base = nullptr;
    if (scratch_address(device, &base) != cudaSuccess) {
        st = MOE_ERR_CUDA;
    } else {
        // Every scratch entry read below is written earlier in the same call,
        // so nothing has to be cleared first.
        uint8_t* s8 = static_cast<uint8_t*>(base);
        float* selsc = reinterpret_cast<float*>(s8 + L.selsc);
        int* hist = reinterpret_cast<int*>(s8 + L.hist);
        int* blkbase = reinterpret_cast<int*>(s8 + L.blkbase);
        int* tiletab = reinterpret_cast<int*>(s8 + L.tiletab);
        int* meta = reinterpret_cast<int*>(s8 + L.meta);
        int* slotof = reinterpret_cast<int*>(s8 + L.slotof);
        float* zpart = reinterpret_cast<float*>(s8 + L.zpart);
        const size_t nz = router_zpart_floats(T, c.H, c.E);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        const int nb = (T + kRouterTokens - 1) / kRouterTokens;
        cudaError_t e;
        if (c.dtype == MOE_FP32)
            e = launch_router<float>(static_cast<const float*>(x), Wr, b, T, c.H, c.E, c.top_k,
                                     c.score, topk_idx, gates, selsc, hist, s, nullptr, nullptr, zpart, nz);
        else
            e = launch_router<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(x), Wr, b, T, c.H,
                                             c.E, c.top_k, c.score, topk_idx, gates, selsc, hist, s,
                                             nullptr, nullptr, zpart, nz);
        if (e == cudaSuccess)
            e = launch_scan(hist, nb, c.E, counts, offsets, blkbase, tiletab, meta, slotof, s);
        if (e == cudaSuccess) e = launch_index(topk_idx, blkbase, T, c.E, c.top_k, row_of, slotof, s);
        if (e != cudaSuccess) st = MOE_ERR_CUDA;
    }
    if (prev != device) cudaSetDevice(prev);
    return st;
}
