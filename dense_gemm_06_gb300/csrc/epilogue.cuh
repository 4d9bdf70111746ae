// epilogue.cuh -- the fused epilogue applied to each accumulator before it is
// stored: D = act(alpha * acc + beta * C_old + bias[col or row]), in fp32,
// then rounded to C's type. It is the CuTe DSL Ampere SGEMM example's
// `epilogue_op` hook (applied to the accumulator fragment before the store)
// with the usual GEMM scaling, a bias vector and an activation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "internal.h"

namespace libgemm {

template <typename T>
__device__ __forceinline__ float to_f32(T v) {
    if constexpr (std::is_same<T, float>::value) return v;
    else if constexpr (std::is_same<T, __nv_bfloat16>::value) return __bfloat162float(v);
    else return __half2float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v) {
    if constexpr (std::is_same<T, float>::value) return v;
    else if constexpr (std::is_same<T, __nv_bfloat16>::value) return __float2bfloat16_rn(v);
    else return __float2half_rn(v);
}

__device__ __forceinline__ float activate(float x, int act) {
    if (act == 1) return fmaxf(x, 0.f);
    if (act == 2) return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));  // x * Phi(x)
    return x;
}

// One output value. `c_old` is the incoming C element (read only if beta != 0).
template <typename OutT>
__device__ __forceinline__ float epilogue_value(const EpiParams& e, float acc, float c_old,
                                                int row, int col) {
    float x = e.alpha * acc;
    if (e.beta != 0.f) x = fmaf(e.beta, c_old, x);
    if (e.bias) x += to_f32(static_cast<const OutT*>(e.bias)[e.bias_rows ? row : col]);
    return activate(x, e.act);
}

}  // namespace libgemm
