// Device side of the fused epilogue C = act(alpha * op(A) op(B) + beta * C +
// bias), shared by every kernel that writes C. The activations are written
// from their definitions (sgemm.h, enum sgemm_activation) on top of CUDA's
// erff, expf and __fdividef.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sgemm.h"

namespace sgemm {

__device__ __forceinline__ float activate(float x, int act) {
    switch (act) {
        case SGEMM_ACT_RELU: return x < 0.0f ? 0.0f : x;  // NaN compares false: stays NaN
        case SGEMM_ACT_GELU: return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));  // x * Phi(x)
        // The fast division (about 2 ulp) keeps the IEEE division's slow path
        // and its register spills out of the kernels; a denominator of +inf
        // (x below about -88) gives -0, the limit of the function.
        case SGEMM_ACT_SILU: return __fdividef(x, 1.0f + expf(-x));
        default: return x;
    }
}

// act(x + bias) for the element (row, col) of a product; col < N and row < M.
__device__ __forceinline__ float epilogue_value(float x, const float *bias, int bias_kind, int act, int64_t row,
                                                int64_t col) {
    if (bias_kind == SGEMM_BIAS_PER_COL)
        x += __ldg(bias + col);
    else if (bias_kind == SGEMM_BIAS_PER_ROW)
        x += __ldg(bias + row);
    return activate(x, act);
}

}  // namespace sgemm
