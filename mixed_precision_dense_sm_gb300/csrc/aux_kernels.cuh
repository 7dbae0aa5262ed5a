// aux_kernels.cuh -- the small memory-bound kernels around the GEMM mainloop.
//
//  * pack_rows_kernel: copy a matrix of 16- or 32-bit elements whose row
//    pitch (or base address) is not a multiple of 16 bytes into a workspace
//    whose pitch is, zero-filling the new padding columns.  TMA can only
//    describe 16-byte-aligned rows; this is the GB300 form of the pages' "pad
//    to the tile and zero-fill" edge handling (DeepGEMM page, section 3.4) for
//    operands the caller laid out with an odd leading dimension.
//  * transpose_rows_kernel: rewrite an FP32 operand stored with its M/N index
//    contiguous (K rows x MN columns) as MN rows x K columns, for the TF32
//    path: tcgen05 kind::tf32 reads K-major operands only.
//  * scale_c_kernel: C = act(beta * C + bias) for the quick-return cases
//    (K == 0 or alpha == 0); beta == 0 never reads C.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue_ops.cuh"

namespace gemm103 {

// dst[r][c] = src[r][c] for c < cols, 0 for cols <= c < dst_ld (T = uint16_t
// or uint32_t; dst_ld a multiple of 16 / sizeof(T)).  One thread per 16-byte
// destination store; source reads are element-sized because the source rows
// are not 16-byte aligned.
template <typename T>
__global__ void __launch_bounds__(256)
    pack_rows_kernel(const T* __restrict__ src, int64_t src_ld, int64_t rows, int64_t cols,
                     T* __restrict__ dst, int64_t dst_ld) {
    constexpr int kVec = 16 / sizeof(T);
    const int64_t vec_per_row = dst_ld / kVec;
    const int64_t total = rows * vec_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / vec_per_row;
        const int64_t c0 = (i - r * vec_per_row) * kVec;
        const T* s = src + r * src_ld;
        union {
            T e[kVec];
            uint4 u;
        } v;
        #pragma unroll
        for (int e = 0; e < kVec; ++e) v.e[e] = (c0 + e < cols) ? s[c0 + e] : static_cast<T>(0);
        *reinterpret_cast<uint4*>(dst + r * dst_ld + c0) = v.u;
    }
}

// dst[n][k] = src[k][n] for k < K, n < MN; dst's columns K..dst_ld-1 are
// written as zeros (dst_ld <= K rounded up to 32).  One 32 x 32 tile per
// iteration through shared memory (padded against bank conflicts), so the
// reads run along n and the writes along k, both coalesced.  Blocks are
// 256 threads (32 x 8) and loop over the tiles.
__global__ void __launch_bounds__(256)
    transpose_rows_kernel(const uint32_t* __restrict__ src, int64_t src_ld, int64_t K, int64_t MN,
                          uint32_t* __restrict__ dst, int64_t dst_ld) {
    __shared__ uint32_t tile[32][33];
    const int64_t tiles_n = (MN + 31) / 32;
    const int64_t tiles = tiles_n * ((K + 31) / 32);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t k0 = (t / tiles_n) * 32, n0 = (t % tiles_n) * 32;
        for (int r = ty; r < 32; r += 8) {
            const int64_t k = k0 + r, n = n0 + tx;
            tile[r][tx] = (k < K && n < MN) ? src[k * src_ld + n] : 0u;
        }
        __syncthreads();
        for (int r = ty; r < 32; r += 8) {
            const int64_t n = n0 + r, k = k0 + tx;
            if (n < MN && k < dst_ld) dst[n * dst_ld + k] = tile[tx][r];
        }
        __syncthreads();
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
