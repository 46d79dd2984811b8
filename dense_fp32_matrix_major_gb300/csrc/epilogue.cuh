// Device side of the fused epilogue C = act(alpha * op(A) op(B) + beta * C +
// bias), shared by every kernel that writes C. The activations are written
// from their definitions (sgemm.h, enum sgemm_activation): GELU through the
// normal distribution function below, SiLU on top of CUDA's expf and
// __fdividef.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sgemm.h"

namespace sgemm {

// Phi(x), the standard normal distribution function, by the rational
// approximation of Zelen and Severo (Abramowitz and Stegun, Handbook of
// Mathematical Functions, 26.2.17): with t = 1 / (1 + p |x|),
// 1 - Phi(|x|) = phi(|x|) (b1 t + b2 t^2 + b3 t^3 + b4 t^4 + b5 t^5), whose
// error is below 7.5e-8 for every x; phi is the normal density. Branch-free
// and about half the instructions of erff, which kept the GELU epilogue
// latency-bound in the four epilogue warps. Phi(-|x|) = 1 - Phi(|x|).
__device__ __forceinline__ float normal_cdf(float x) {
    const float z = fabsf(x);
    const float t = __fdividef(1.0f, fmaf(0.2316419f, z, 1.0f));
    float poly = fmaf(t, 1.330274429f, -1.821255978f);
    poly = fmaf(t, poly, 1.781477937f);
    poly = fmaf(t, poly, -0.356563782f);
    poly = fmaf(t, poly, 0.319381530f);
    const float tail = 0.3989422804014327f * __expf(-0.5f * z * z) * (poly * t);  // 1 - Phi(z)
    return x >= 0.0f ? 1.0f - tail : tail;
}

__device__ __forceinline__ float activate(float x, int act) {
    switch (act) {
        case SGEMM_ACT_RELU: return x < 0.0f ? 0.0f : x;  // NaN compares false: stays NaN
        case SGEMM_ACT_GELU: return x * normal_cdf(x);   // x * Phi(x); NaN stays NaN
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
