// gemm_nv.cu -- the NVFP4 instances of the block-scaled grouped GEMM
// (gemm_bs.cuh) for the MOE_NVFP4 layer: every operand K-major, K (and the
// data GEMMs' K = H or F) a multiple of 256 values.
#include "gemm_bs.cuh"

namespace moe {

cudaError_t gemm_nv_prepare(int device)
{
    (void)device;
    if (!encx()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    acc(xattr<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, false, true>());
    acc(xattr<EPI_STORE, SCHED_ROWS, DUAL_NONE, false, true>());
    acc(xattr<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE, false, true>());
    acc(xattr<EPI_STORE, SCHED_ROWS, DUAL_K, false, true>());
    acc(xattr<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE, false, true>());
    acc(xattr<EPI_WGRAD, SCHED_WGRAD, DUAL_N, false, true>());
    return e;
}

cudaError_t launch_gemm_nv(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    if (!encx()) return cudaErrorNotSupported;
    if (!d.nv || !d.gA || !d.gB) return cudaErrorInvalidValue;
    if (d.sched == SCHED_ROWS) {
        if (!d.b_kmajor || d.K % 256) return cudaErrorInvalidValue;
        switch (d.epi) {
        case EPI_SWIGLU_FWD:
            return xrun_any<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, false, true>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD:
            return xrun_any<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE, false, true>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            return d.dual == DUAL_K ? xrun_any<EPI_STORE, SCHED_ROWS, DUAL_K, false, true>(d, max_m_tiles, num_sms, s)
                                    : xrun_any<EPI_STORE, SCHED_ROWS, DUAL_NONE, false, true>(d, max_m_tiles, num_sms, s);
        default: return cudaErrorInvalidValue;
        }
    }
    return d.dual == DUAL_N ? xrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_N, false, true>(d, max_m_tiles, num_sms, s)
                            : xrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE, false, true>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
