// diag.cu -- small entry points outside the layer's forward and backward.
//
// moe_update_bias: the auxiliary-loss-free bias update ("Scalable Training of
// Mixture-of-Experts Models with Megatron Core", §7 Load Balancing):
// b_e += rate * sign(mean load - load of e), compared exactly in integers.
//
// moe_diag_wait_timeout: exercises the device-side bounded wait
// (ptx::wait_bounded) that every pipelined kernel of the library uses, on an
// mbarrier that nothing ever signals. The wait gives up after its limit and
// records MOE_ERR_DEVICE_TIMEOUT in the status word, so a test can check
// that a stalled pipeline ends with an error instead of hanging the GPU.
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(DeviceStatus* status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        ptx::wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, status, 99);
    __syncthreads();
}

__global__ void __launch_bounds__(kMaxE)
update_bias_kernel(int E, const int* __restrict__ counts, float rate, float* __restrict__ b)
{
    __shared__ long long total;
    if (threadIdx.x == 0) {
        long long s = 0;
        for (int e = 0; e < E; ++e) s += counts[e];   // fixed order
        total = s;
    }
    __syncthreads();
    const int e = threadIdx.x;
    if (e < E) {
        const long long d = total - (long long)E * counts[e];   // E * (mean - c_e)
        const float sg = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
        b[e] = b[e] + rate * sg;
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

moe_status_t moe_update_bias(int E, const int32_t* counts, float rate, float* b, moe_stream_t stream)
{
    if (!counts || !b || E < 1 || E > kMaxE || !(rate == rate) || rate - rate != 0.f)
        return MOE_ERR_INVALID_ARG;
    update_bias_kernel<<<1, kMaxE, 0, reinterpret_cast<cudaStream_t>(stream)>>>(E, counts, rate, b);
    count_launches();
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_diag_wait_timeout(void* ws, moe_stream_t stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceStatus* st = static_cast<DeviceStatus*>(ws);
    if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, s>>>(st);
    count_launches();
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
