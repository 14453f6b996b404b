// epilogue.cuh -- the output epilogue shared by the GEMM kernels: bias,
// activation, output type (see Epi in internal.h).  Device code only.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {

// act(v + b): ReLU; SiLU v * sigmoid(v); GELU in its erf form
// 0.5 v (1 + erf(v / sqrt(2))).  fp32, with the CUDA math library's expf/erff.
__device__ __forceinline__ float epi_value(float v, float b, int act) {
    v += b;
    switch (act) {
        case ACT_RELU:
            return fmaxf(v, 0.0f);
        case ACT_SILU:
            return v / (1.0f + expf(-v));
        case ACT_GELU:
            return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
        default:
            return v;
    }
}

// Store element idx of y in the output type.
__device__ __forceinline__ void epi_store(void* y, int64_t idx, float v, int out) {
    if (out == OUT_F16)
        static_cast<__half*>(y)[idx] = __float2half_rn(v);
    else if (out == OUT_BF16)
        static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<float*>(y)[idx] = v;
}

// The epilogue over a thread's C accumulators (one output column n, C
// consecutive rows m0 .. m0+C-1 with row stride ldy), with each decision taken
// once outside an unrolled loop: a per-element switch, unrolled C times with
// the inlined expf / erff, made the kernel's code several times larger (and
// the GEMM twice as slow, measured on GB300).
// bn: bias[n] (0 without a bias), loaded by the caller ahead of time.
// SiLU uses the fast exponential and divide (__expf, __fdividef: relative
// error a few 1e-6 for |v| < 20, far below an fp16 output's rounding); GELU
// the library erff.
template <int C>
__device__ __forceinline__ void epi_tile(float (&acc)[C], const Epi& epi, float bn, void* y, int64_t ldy, int n,
                                         int m0, int m_end) {
    if (epi.bias) {
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] += bn;
    }
    if (epi.act == ACT_RELU) {
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] = fmaxf(acc[j], 0.0f);
    } else if (epi.act == ACT_SILU) {
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] = __fdividef(acc[j], 1.0f + __expf(-acc[j]));
    } else if (epi.act == ACT_GELU) {
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] = 0.5f * acc[j] * (1.0f + erff(acc[j] * 0.70710678118654752f));
    }
    if (epi.out == OUT_F16) {
        __half* yh = static_cast<__half*>(y);
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (m0 + j < m_end) yh[static_cast<int64_t>(m0 + j) * ldy + n] = __float2half_rn(acc[j]);
    } else if (epi.out == OUT_BF16) {
        __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (m0 + j < m_end) yb[static_cast<int64_t>(m0 + j) * ldy + n] = __float2bfloat16_rn(acc[j]);
    } else {
        float* yf = static_cast<float*>(y);
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (m0 + j < m_end) yf[static_cast<int64_t>(m0 + j) * ldy + n] = acc[j];
    }
}

}  // namespace qg
