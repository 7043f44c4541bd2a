// Device helpers shared by the CUDA-core kernels: activation loads and the
// Taylor feature map.
//
// Feature map (BASED reading notes, "Simple linear attention language models
// balance the recall-throughput tradeoff", sec. 2.3):
//   phi(x) = [1, xbar, vec(xbar xbar^T)/sqrt(2)],  xbar = x / 16^(1/4) = x / 2.
// Index f: 0 constant, 1 + a linear, 17 + 16 a + b quadratic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

template <typename T> struct Act;
template <> struct Act<float> {
    static __device__ __forceinline__ float load(const float *p, int64_t i) { return p[i]; }
    static __device__ __forceinline__ void store(float *p, int64_t i, float x) { p[i] = x; }
};
template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p, int64_t i) {
        return __bfloat162float(p[i]);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, int64_t i, float x) {
        p[i] = __float2bfloat16_rn(x);
    }
};

// Programmatic dependent launch (a launch with the programmatic stream
// serialization attribute): pdl_wait blocks until the previous kernel in the
// stream has completed and its memory is visible (a no-op without the
// attribute); pdl_trigger lets the next kernel be scheduled once every CTA of
// this grid has triggered or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 1/sqrt(2) rounded to fp32.
constexpr float kInvSqrt2 = 0.70710678118654752440f;

// phi_f(xbar) for one feature index, xbar already scaled (x/2).
__device__ __forceinline__ float phi_feature(const float *xbar, int f) {
    if (f == 0) return 1.0f;
    if (f <= 16) return xbar[f - 1];
    const int a = (f - 17) >> 4, b = (f - 17) & 15;
    return xbar[a] * xbar[b] * kInvSqrt2;
}

}  // namespace la
