// aux_kernels.cuh -- the small memory-bound kernels around the GEMM mainloop.
//
//  * pack_rows_kernel: copy a 16-bit matrix whose row pitch (or base address)
//    is not a multiple of 16 bytes into a workspace whose pitch is, zero-filling
//    the new padding columns.  TMA can only describe 16-byte-aligned rows; this
//    is the GB300 form of the pages' "pad to the tile and zero-fill" edge
//    handling (DeepGEMM page, section 3.4) for operands the caller laid out
//    with an odd leading dimension.
//  * scale_c_kernel: C = act(beta * C + bias) for the quick-return cases
//    (K == 0 or alpha == 0); beta == 0 never reads C.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue_ops.cuh"

namespace gemm103 {

// dst[r][c] = src[r][c] for c < cols, 0 for cols <= c < dst_ld.
// One thread per 8 destination elements (one 16-byte store); source reads are
// 2-byte loads because the source rows are not 16-byte aligned.
__global__ void __launch_bounds__(256)
    pack_rows_kernel(const uint16_t* __restrict__ src, int64_t src_ld, int64_t rows, int64_t cols,
                     uint16_t* __restrict__ dst, int64_t dst_ld) {
    const int64_t vec_per_row = dst_ld / 8;
    const int64_t total = rows * vec_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / vec_per_row;
        const int64_t c0 = (i - r * vec_per_row) * 8;
        const uint16_t* s = src + r * src_ld;
        uint16_t v[8];
        #pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (c0 + e < cols) ? s[c0 + e] : static_cast<uint16_t>(0);
        uint4 out;
        out.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
        out.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
        out.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
        out.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
        *reinterpret_cast<uint4*>(dst + r * dst_ld + c0) = out;
    }
}

template <typename OutT>
__device__ __forceinline__ float scale_load(const OutT* p);
template <>
__device__ __forceinline__ float scale_load<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float scale_load<__half>(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float scale_load<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename OutT>
__device__ __forceinline__ OutT scale_store(float v);
template <>
__device__ __forceinline__ float scale_store<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half scale_store<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 scale_store<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

template <typename OutT>
__global__ void __launch_bounds__(256)
    scale_c_kernel(OutT* __restrict__ C, int64_t M, int64_t N, int64_t ldc, float beta,
                   const void* bias, int32_t bias_dtype, int32_t act) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        OutT* p = C + r * ldc + c;
        float x = beta == 0.0f ? 0.0f : beta * scale_load<OutT>(p);
        if (bias != nullptr) x += load_bias_elem(bias, bias_dtype, c);
        *p = scale_store<OutT>(activate(act, x));
    }
}

}  // namespace gemm103
