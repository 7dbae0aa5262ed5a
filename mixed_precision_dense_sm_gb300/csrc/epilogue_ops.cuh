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

// erfc(u), u >= 0, with a small *relative* error everywhere: the Chebyshev
// fit of Press, Teukolsky, Vetterling and Flannery, Numerical Recipes in C
// (2nd ed.), section 6.2, routine erfcc:
//     erfc(u) = t exp(-u^2 + P(t)),  t = 1 / (1 + u / 2),
// P a degree-9 polynomial, fractional error < 1.2e-7 for every u >= 0.
// Here t uses the approximate reciprocal (2 ulp) and exp the fast
// exponential, whose error grows like |argument| 2^-23; in all
// |relative error| <= (u^2 + 2) 2^-22 + 3e-7.
__device__ __forceinline__ float erfc_nr(float u) {
    const float t = __fdividef(1.0f, fmaf(0.5f, u, 1.0f));
    float p = fmaf(t, 0.17087277f, -0.82215223f);
    p = fmaf(t, p, 1.48851587f);
    p = fmaf(t, p, -1.13520398f);
    p = fmaf(t, p, 0.27886807f);
    p = fmaf(t, p, -0.18628806f);
    p = fmaf(t, p, 0.09678418f);
    p = fmaf(t, p, 0.37409196f);
    p = fmaf(t, p, 1.00002368f);
    p = fmaf(t, p, -1.26551223f);
    return t * __expf(fmaf(-u, u, p));
}

// GELU(x) = x Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2: for x >= 0
// x (1 - erfc(x / sqrt 2) / 2), for x < 0 x erfc(|x| / sqrt 2) / 2 -- no
// cancellation on either side, so the relative error stays near that of
// erfc_nr even where Phi(x) is tiny (a 16-bit output of a very negative x is
// then still correctly rounded or one ulp off).  About twenty instructions,
// run once per output element; the epilogue evaluates 32 of them at a time
// (act32 below) so their chains interleave and hide under the next tile's
// MMA.  NaN stays NaN; GELU(+inf) = inf, GELU(-inf) = NaN (-inf * 0), as
// x Phi(x) evaluates in IEEE arithmetic.
__device__ __forceinline__ float gelu(float x) {
    const float e = erfc_nr(fabsf(x) * 0.70710678118654752f);
    return x >= 0.0f ? x * fmaf(-0.5f, e, 1.0f) : 0.5f * x * e;
}

__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ float relu(float x) {
    return x > 0.0f ? x : (x != x ? x : 0.0f);     // NaN stays NaN
}

__device__ __forceinline__ float activate(int act, float x) {
    switch (act) {
        case kActRelu: return relu(x);
        case kActGelu: return gelu(x);
        case kActSilu: return silu(x);
        default: return x;
    }
}

// The activation on 32 values, the choice made once outside the element loop
// so that the 32 independent evaluations interleave.
__device__ __forceinline__ void act32(int act, float (&v)[32]) {
    if (act == kActGelu) {
        #pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu(v[j]);
    } else if (act == kActSilu) {
        #pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = silu(v[j]);
    } else if (act == kActRelu) {
        #pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = relu(v[j]);
    }
}

// Element idx of a bias vector of type 0 = F16, 1 = BF16, 2 = F32.
__device__ __forceinline__ float load_bias_elem(const void* bias, int32_t dtype, int64_t idx) {
    if (dtype == 2) return reinterpret_cast<const float*>(bias)[idx];
    if (dtype == 1) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(bias)[idx]);
    return __half2float(reinterpret_cast<const __half*>(bias)[idx]);
}

}  // namespace gemm103
