// la_device.cuh -- small device helpers shared by the SIMT kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace la {

// phi(x) = elu(x) + 1, written as x + 1 (x > 0), e^x (x <= 0): the simplified
// piecewise form given on the "Linear Transformer" page ("La función ELU + 1").
// e^x uses CUDA's fast exponential intrinsic; phi > 0 except where e^x
// underflows for x below about -87.
__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// The feature map of a call: elu(x) + 1 (kind 0) or the identity (kind 1),
// the two element-wise maps of "Mapas de características".
__device__ __forceinline__ float feature_f(float x, int kind) { return kind ? x : phi_f(x); }

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace la
