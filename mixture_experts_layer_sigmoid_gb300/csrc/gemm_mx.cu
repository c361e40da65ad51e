// gemm_mx.cu -- the MXFP8 instances of the block-scaled grouped GEMM
// (gemm_bs.cuh) for the MOE_MXFP8 layer.
#include "gemm_bs.cuh"

namespace moe {

cudaError_t gemm_mx_prepare(int device)
{
    (void)device;
    if (!encx()) return cudaErrorNotSupported;
    cudaError_t e = cudaSuccess;
    auto acc = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    acc(xattr<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, true, false>());
    acc(xattr<EPI_STORE, SCHED_ROWS, DUAL_NONE, true, false>());
    acc(xattr<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE, false, false>());
    acc(xattr<EPI_STORE, SCHED_ROWS, DUAL_K, false, false>());
    acc(xattr<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE, false, false>());
    acc(xattr<EPI_WGRAD, SCHED_WGRAD, DUAL_N, false, false>());
    return e;
}

cudaError_t launch_gemm_mx(const GemmDesc& d, int max_m_tiles, int num_sms, cudaStream_t s)
{
    if (!encx()) return cudaErrorNotSupported;
    if (d.nv) return cudaErrorInvalidValue;
    if (d.sched == SCHED_ROWS) {
        switch (d.epi) {
        // forward GEMMs read the weights' codes MN-major (b_kmajor 0), the
        // data-gradient GEMMs K-major (b_kmajor 1)
        case EPI_SWIGLU_FWD:
            if (d.b_kmajor) return cudaErrorInvalidValue;
            return xrun_any<EPI_SWIGLU_FWD, SCHED_ROWS, DUAL_N, true, false>(d, max_m_tiles, num_sms, s);
        case EPI_SWIGLU_BWD:
            if (!d.b_kmajor) return cudaErrorInvalidValue;
            return xrun_any<EPI_SWIGLU_BWD, SCHED_ROWS, DUAL_NONE, false, false>(d, max_m_tiles, num_sms, s);
        case EPI_STORE:
            if (d.dual == DUAL_K)
                return d.b_kmajor ? xrun_any<EPI_STORE, SCHED_ROWS, DUAL_K, false, false>(d, max_m_tiles, num_sms, s)
                                  : cudaErrorInvalidValue;
            return d.b_kmajor ? cudaErrorInvalidValue
                              : xrun_any<EPI_STORE, SCHED_ROWS, DUAL_NONE, true, false>(d, max_m_tiles, num_sms, s);
        default: return cudaErrorInvalidValue;
        }
    }
    return d.dual == DUAL_N ? xrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_N, false, false>(d, max_m_tiles, num_sms, s)
                            : xrun_any<EPI_WGRAD, SCHED_WGRAD, DUAL_NONE, false, false>(d, max_m_tiles, num_sms, s);
}

}  // namespace moe
