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

}  // namespace qg
