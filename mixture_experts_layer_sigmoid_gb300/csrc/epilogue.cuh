// epilogue.cuh -- per-element epilogues of the grouped GEMMs (SwiGLU forward
// and backward, plain store), shared by the fp32 SIMT and the bf16 tensor-core
// engines.
//
// SwiGLU expert FFN (the pages name the expert FFN and its activation
// recomputation, "moe_act", in "Scalable Training of Mixture-of-Experts Models
// with Megatron Core", §4 and App. B.2; the form is the plain SwiGLU):
//   h = silu(a) u,  silu(a) = a sigma(a),  sigma(a) = 1 / (1 + exp(-a))
//   dA = dh u silu'(a),  silu'(a) = sigma(a) (1 + a (1 - sigma(a))),  dU = dh silu(a)
#pragma once
#include <cuda_bf16.h>

namespace moe {

__device__ __forceinline__ float sigmoid_f(float a) { return 1.f / (1.f + expf(-a)); }

struct SwigluFwd {
    float a, u, h;
    __device__ __forceinline__ SwigluFwd(float a_, float u_) : a(a_), u(u_) {
        h = a_ * sigmoid_f(a_) * u_;
    }
};

struct SwigluBwd {
    float dA, dU;
    __device__ __forceinline__ SwigluBwd(float dh, float a, float u) {
        const float s = sigmoid_f(a);
        dU = dh * a * s;
        dA = dh * u * s * (1.f + a * (1.f - s));
    }
};

// Memory-efficient permutation ("Scalable Training of Mixture-of-Experts
// Models with Megatron Core", §4, Memory-Efficient Permutation): the routing
// weight g of a permuted row is folded into its activation before fc2,
// h' = g h, so fc2 directly yields g y_e and Combine is a plain sum. In the
// backward pass fc2 dgrad yields dh' = dY Wd^T for the row, and
//   dg = <dh', h>,  dh = g dh',  then dA, dU as above;
// h is recomputed from the saved a, u (and h' = g h for the fc2 weight
// gradient), so neither h nor the expert outputs are kept between passes.
struct SwigluBwdFold {
    float dA, dU, h;
    __device__ __forceinline__ SwigluBwdFold(float dhp, float g, float a, float u) {
        const float s = sigmoid_f(a);
        const float as = a * s;
        h = as * u;
        const float dh = g * dhp;
        dU = dh * as;
        dA = dh * u * s * (1.f + a * (1.f - s));
    }
};

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
__device__ __forceinline__ float as_f32(float v) { return v; }
__device__ __forceinline__ float as_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

}  // namespace moe
