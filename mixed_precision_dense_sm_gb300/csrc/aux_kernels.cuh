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
//  * ln_rows_stats_kernel: the row pass of LayerNorm after the linear layer
//    for rows wider than one GEMM tile (merges the tiles' statistics);
//    ln_rows_kernel: the same from scratch for the quick-return cases.
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

// Sum over the CTA's 256 threads, the same order on every run; `red` holds 8
// floats.  Every thread gets the total.
__device__ __forceinline__ float block_sum256(float v, float* red) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.0f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    __syncthreads();                       // red is reused by the next call
    return t;
}

// KV consecutive elements j0.. of a per-column vector (gamma, shift) of type
// 0 = F16, 1 = BF16, 2 = F32.  `aligned`: the vector's base is 16-byte
// aligned (j0 is a multiple of KV), so the loads are 8-, 16- or 32-byte wide.
template <int KV>
__device__ __forceinline__ void load_vec_kv(const void* vec, int32_t dtype, int64_t j0,
                                            bool aligned, float (&o)[KV]) {
    static_assert(KV == 4 || KV == 8, "KV");
    if (!aligned) {
        #pragma unroll
        for (int e = 0; e < KV; ++e) o[e] = load_bias_elem(vec, dtype, j0 + e);
        return;
    }
    if (dtype == 2) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(vec) + j0);
        #pragma unroll
        for (int q = 0; q < KV / 4; ++q) {
            const uint4 t = __ldg(src + q);
            o[4 * q] = __uint_as_float(t.x);
            o[4 * q + 1] = __uint_as_float(t.y);
            o[4 * q + 2] = __uint_as_float(t.z);
            o[4 * q + 3] = __uint_as_float(t.w);
        }
        return;
    }
    uint32_t w[KV / 2];
    const uint16_t* src = static_cast<const uint16_t*>(vec) + j0;
    if constexpr (KV == 8) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(src));
        w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
    } else {
        const uint2 t = __ldg(reinterpret_cast<const uint2*>(src));
        w[0] = t.x; w[1] = t.y;
    }
    #pragma unroll
    for (int e = 0; e < KV / 2; ++e) {
        const uint16_t lo = static_cast<uint16_t>(w[e] & 0xFFFFu);
        const uint16_t hi = static_cast<uint16_t>(w[e] >> 16);
        if (dtype == 1) {
            o[2 * e] = __bfloat162float(__ushort_as_bfloat16(lo));
            o[2 * e + 1] = __bfloat162float(__ushort_as_bfloat16(hi));
        } else {
            o[2 * e] = __half2float(__ushort_as_half(lo));
            o[2 * e + 1] = __half2float(__ushort_as_half(hi));
        }
    }
}

// y = (h - mean) * rstd * gamma + shift for KV elements held in one 16-byte
// vector of C's type, in place.
template <typename OutT, int KV>
__device__ __forceinline__ uint4 ln_apply_vec(uint4 hv, int64_t j0, float mean, float rstd,
                                              const void* gamma, bool g_al, const void* shift,
                                              bool s_al, int32_t ln_dtype) {
    union {
        uint4 u;
        OutT e[KV];
    } h;
    h.u = hv;
    float y[KV];
    #pragma unroll
    for (int e = 0; e < KV; ++e) y[e] = (scale_load<OutT>(&h.e[e]) - mean) * rstd;
    if (gamma != nullptr) {
        float g[KV];
        load_vec_kv<KV>(gamma, ln_dtype, j0, g_al, g);
        #pragma unroll
        for (int e = 0; e < KV; ++e) y[e] *= g[e];
    }
    if (shift != nullptr) {
        float t[KV];
        load_vec_kv<KV>(shift, ln_dtype, j0, s_al, t);
        #pragma unroll
        for (int e = 0; e < KV; ++e) y[e] += t[e];
    }
    #pragma unroll
    for (int e = 0; e < KV; ++e) h.e[e] = scale_store<OutT>(y[e]);
    return h.u;
}

// Elements j_from.. of one row of C (scalar, a CTA of kT threads):
// y = (h - mean) * rstd * gamma + shift.
template <typename OutT, int kT>
__device__ __forceinline__ void ln_apply_scalar(OutT* c, int64_t j_from, int64_t N, float mean,
                                                float rstd, const void* gamma, const void* shift,
                                                int32_t ln_dtype) {
    for (int64_t j = j_from + threadIdx.x; j < N; j += kT) {
        float y = (scale_load<OutT>(c + j) - mean) * rstd;
        if (gamma != nullptr) y *= load_bias_elem(gamma, ln_dtype, j);
        if (shift != nullptr) y += load_bias_elem(shift, ln_dtype, j);
        c[j] = scale_store<OutT>(y);
    }
}

// Sum over a warp by a butterfly of shuffles: every lane ends with the same
// value (each level adds the same two operands in every lane, and FP32
// addition is commutative).
__device__ __forceinline__ float warp_sum_all(float v) {
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kLnRowThreads = 128;

// The row pass of LayerNorm after the linear layer, from per-tile statistics:
// stats[row * tiles_n + t] = (sum, M2) of h over the tile's n_t columns
// t * block_n .. (M2 about the tile's own mean).  The row's statistics follow
// from the decomposition of the sum of squares over a partition:
//     mean = sum_t sum_t / N,   M2 = sum_t M2_t + sum_t n_t (sum_t / n_t - mean)^2,
// each total a fixed-order per-lane sum over the lane's tiles followed by a
// butterfly over warp 0 (the same bits on every run).  One CTA of 128 threads
// per row, rows strided over the grid; each thread issues the loads of its
// first kPre 16-byte vectors of the row before the statistics are ready, so
// both latencies overlap.  The row is read once and written once; rows whose
// start is not 16-byte aligned go element by element.  FP32 throughout.
template <typename OutT>
__global__ void __launch_bounds__(kLnRowThreads, 8)
    ln_rows_stats_kernel(OutT* __restrict__ C, int64_t ldc, int64_t M, int64_t N,
                         const float2* __restrict__ stats, int32_t tiles_n, int32_t block_n,
                         const void* gamma, const void* shift, int32_t ln_dtype, float eps) {
    constexpr int KV = 16 / static_cast<int>(sizeof(OutT));
    constexpr int kPre = 4;
    constexpr int kT = kLnRowThreads;
    __shared__ float row_stat[2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool g_al = (reinterpret_cast<uintptr_t>(gamma) & 15u) == 0;
    const bool s_al = (reinterpret_cast<uintptr_t>(shift) & 15u) == 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        OutT* c = C + row * ldc;
        const bool vec = (reinterpret_cast<uintptr_t>(c) & 15u) == 0;
        const int64_t nvec = vec ? N / KV : 0;
        const uint4* c4 = reinterpret_cast<const uint4*>(c);
        uint4 h[kPre];
        #pragma unroll
        for (int r = 0; r < kPre; ++r) {
            const int64_t iv = threadIdx.x + static_cast<int64_t>(r) * kT;
            h[r] = iv < nvec ? __ldcs(c4 + iv) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (warp == 0) {
            const float2* st = stats + row * tiles_n;
            float s = 0.0f;
            for (int32_t t = lane; t < tiles_n; t += 32) s += st[t].x;
            const float mean = warp_sum_all(s) / static_cast<float>(N);
            float q = 0.0f;
            for (int32_t t = lane; t < tiles_n; t += 32) {
                const float2 v = st[t];
                const int64_t left = N - static_cast<int64_t>(t) * block_n;
                const float nt = static_cast<float>(left < block_n ? left : block_n);
                const float d = v.x / nt - mean;
                q += v.y + nt * d * d;
            }
            const float m2 = warp_sum_all(q);
            if (lane == 0) {
                row_stat[0] = mean;
                row_stat[1] = 1.0f / sqrtf(m2 / static_cast<float>(N) + eps);
            }
        }
        __syncthreads();
        const float mean = row_stat[0], rstd = row_stat[1];
        uint4* o4 = reinterpret_cast<uint4*>(c);
        #pragma unroll
        for (int r = 0; r < kPre; ++r) {
            const int64_t iv = threadIdx.x + static_cast<int64_t>(r) * kT;
            if (iv < nvec)
                __stcs(o4 + iv, ln_apply_vec<OutT, KV>(h[r], iv * KV, mean, rstd, gamma, g_al,
                                                       shift, s_al, ln_dtype));
        }
        #pragma unroll 2
        for (int64_t iv = threadIdx.x + kPre * kT; iv < nvec; iv += kT)
            __stcs(o4 + iv, ln_apply_vec<OutT, KV>(__ldcs(c4 + iv), iv * KV, mean, rstd, gamma,
                                                   g_al, shift, s_al, ln_dtype));
        ln_apply_scalar<OutT, kT>(c, nvec * KV, N, mean, rstd, gamma, shift, ln_dtype);
        __syncthreads();                   // row_stat is rewritten for the next row
    }
}

// LayerNorm of whole rows of C in place when no statistics exist (the quick
// returns K == 0 or alpha == 0, where h = round_C(beta * C + bias) was just
// written): one CTA (256 threads) per row computes the mean and then the sum
// of squared deviations (two passes, no cancellation) and then applies
// y = (h - mean) / sqrt(M2 / N + eps) * gamma + shift.  FP32 throughout.
template <typename OutT>
__global__ void __launch_bounds__(256)
    ln_rows_kernel(OutT* __restrict__ C, int64_t ldc, int64_t M, int64_t N, const void* gamma,
                   const void* shift, int32_t ln_dtype, float eps) {
    __shared__ float red[8];
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        OutT* c = C + row * ldc;
        float s = 0.0f;
        for (int64_t j = threadIdx.x; j < N; j += 256) s += scale_load<OutT>(c + j);
        const float mean = block_sum256(s, red) / static_cast<float>(N);
        float q = 0.0f;
        for (int64_t j = threadIdx.x; j < N; j += 256) {
            const float d = scale_load<OutT>(c + j) - mean;
            q = fmaf(d, d, q);
        }
        const float m2 = block_sum256(q, red);
        const float rstd = 1.0f / sqrtf(m2 / static_cast<float>(N) + eps);
        ln_apply_scalar<OutT, 256>(c, 0, N, mean, rstd, gamma, shift, ln_dtype);
        __syncthreads();                   // every read of the row precedes the next row's
    }
}

}  // namespace gemm103
