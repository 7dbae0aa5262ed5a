// epilogue_ops.cuh -- element operations of the fused epilogue,
//     r = act(alpha * acc + beta * C + bias[n]),
// the CATLASS page's fusion by a replaced epilogue after an unchanged mainloop
// (section 5.2), in its usual linear-layer form: a per-output-column bias and one of
// ReLU, GELU (erf form) or SiLU, evaluated in FP32 before the output cast.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gemm103 {

enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2, kActSilu = 3 };

// erf(x) by the rational approximation of Abramowitz and Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (after Hastings):
//     erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//     t = 1 / (1 + p x),  x >= 0,  |error| <= 1.5e-7,
// extended to x < 0 by oddness; t uses the approximate reciprocal (a couple of
// ulps, scaled by the polynomial and exp(-x^2) <= 1 in erf).  About a dozen
// instructions against the
// several dozen of a fully accurate erf: the GELU epilogue runs once per output
// element and must hide under the MMA of the next tile.  The error is far
// inside the GEMM's own tolerance (1e-5 of the operand scale).
__device__ __forceinline__ float erf_as7126(float x) {
    const float ax = fabsf(x);
    const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));   // approximate reciprocal
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    poly *= t;
    const float y = fmaf(-poly, __expf(-ax * ax), 1.0f);
    return copysignf(y, x);
}

__device__ __forceinline__ float activate(int act, float x) {
    switch (act) {
        case kActRelu: return x > 0.0f ? x : (x != x ? x : 0.0f);     // NaN stays NaN
        case kActGelu: return 0.5f * x * (1.0f + erf_as7126(x * 0.70710678118654752f));
        case kActSilu: return __fdividef(x, 1.0f + __expf(-x));
        default: return x;
    }
}

// Element idx of a bias vector of type 0 = F16, 1 = BF16, 2 = F32.
__device__ __forceinline__ float load_bias_elem(const void* bias, int32_t dtype, int64_t idx) {
    if (dtype == 2) return reinterpret_cast<const float*>(bias)[idx];
    if (dtype == 1) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(bias)[idx]);
    return __half2float(reinterpret_cast<const __half*>(bias)[idx]);
}

}  // namespace gemm103
