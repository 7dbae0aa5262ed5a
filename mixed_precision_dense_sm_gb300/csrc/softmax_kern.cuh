// softmax_kern.cuh -- the row-softmax kernel (include/softmax_sm103.h) and its
// launcher, instantiated per input type in softmax_{f32,f16,bf16}.cu.
//
// For each row: m = max x, s = sum exp(x - m), y = exp(x - m) / s (SGEMM
// tutorial page, sections 2.1-2.2), in FP32 for every storage type.
//
// Work split.  A "row group" owns one row at a time and loops over rows
// (persistent grid):
//   * WARP_ROWS: a warp per row (rows of at most 32 x kE = 1024 elements);
//     reductions by shuffles only.
//   * otherwise a CTA per row, or a thread-block cluster of `cluster` CTAs
//     each holding a `slice` of the row; the CTAs' (m, s) pairs are merged
//     through distributed shared memory.
// Each thread keeps up to kE elements in registers per chunk.  When a CTA's
// slice fits one chunk (resident) the row is read once and written from
// registers; otherwise a first pass folds the chunks into a running (m, s)
// with the online rule and a second pass re-reads the slice to write y.
//
// Pairs (m, s) combine by m' = max(m1, m2), s' = s1 e^(m1 - m') +
// s2 e^(m2 - m') (SGEMM tutorial page, section 2.2), where a side with
// m = -inf (no finite entries) contributes 0.  The maximum propagates NaN, so
// NaN anywhere makes the row NaN; +inf makes s NaN (inf - inf); a fully
// masked row keeps m = -inf and its y = exp(-inf - (-inf)) / 0 is NaN.
#pragma once
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace smx {

constexpr int kE = 32;                 // elements per thread per chunk
constexpr int kWarpCtaThreads = 256;   // warp mode: 8 rows in flight per CTA
constexpr int kMaxCluster = 8;

struct SoftmaxParams {
    const void* X;
    void* Y;
    int64_t ldx, ldy;
    int64_t rows;
    int32_t cols;
    int32_t slice;      // elements of a row per CTA (multiple of 8)
    int32_t cluster;    // CTAs per row
    int32_t vec;        // rows are 16-byte aligned: 16-byte loads and stores
    int32_t resident;   // slice <= threads * kE
};

template <typename T> struct VecOf;
template <> struct VecOf<float> { static constexpr int V = 4; };
template <> struct VecOf<__half> { static constexpr int V = 8; };
template <> struct VecOf<__nv_bfloat16> { static constexpr int V = 8; };

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// max that returns NaN when either operand is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// (m, s) <- (m, s) combined with (m2, s2)
__device__ __forceinline__ void merge(float& m, float& s, float m2, float s2) {
    const float mm = fmax_nan(m, m2);
    const float a = (m == -INFINITY) ? 0.0f : s * __expf(m - mm);
    const float b = (m2 == -INFINITY) ? 0.0f : s2 * __expf(m2 - mm);
    m = mm;
    s = a + b;
}

__device__ __forceinline__ void warp_merge(float& m, float& s) {
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        merge(m, s, m2, s2);
    }
}

// Element e (0 <= e < kE) of thread t in a chunk of T * kE elements starting
// at `base`: the vector path gives each thread whole 16-byte vectors (V
// elements: vector k of thread t is vector k * T + t of the chunk), the
// scalar path interleaves single elements across the threads (element e of
// thread t is element e * T + t).  Both cover the chunk once and keep each
// warp's accesses contiguous.  Offsets are 32-bit: a row has < 2^31 elements.
// KEEP: the chunk will be read again soon (the first of two passes over a
// slice), so its lines stay in L2 (ld.global.cg); otherwise this is the last
// read and they go first (ld.global.cs).
template <typename InT, bool KEEP = false>
__device__ __forceinline__ void load_chunk(const InT* __restrict__ x, int32_t base, int32_t end,
                                           bool vec, int t, int T, float (&v)[kE]) {
    constexpr int V = VecOf<InT>::V;
    if (vec) {
        #pragma unroll
        for (int k = 0; k < kE / V; ++k) {
            const int32_t e0 = base + (k * T + t) * V;
            if (e0 + V <= end) {
                const uint4 u = KEEP ? __ldcg(reinterpret_cast<const uint4*>(x + e0))
                                     : __ldcs(reinterpret_cast<const uint4*>(x + e0));
                const InT* q = reinterpret_cast<const InT*>(&u);
                #pragma unroll
                for (int i = 0; i < V; ++i) v[k * V + i] = to_f(q[i]);
            } else {
                #pragma unroll
                for (int i = 0; i < V; ++i) v[k * V + i] = (e0 + i < end) ? to_f(x[e0 + i]) : -INFINITY;
            }
        }
    } else {
        #pragma unroll
        for (int e = 0; e < kE; ++e) {
            const int32_t i = base + e * T + t;
            v[e] = (i < end) ? to_f(x[i]) : -INFINITY;
        }
    }
}

template <typename InT, typename OutT>
__device__ __forceinline__ void store_chunk(OutT* __restrict__ y, int32_t base, int32_t end,
                                            bool vec, int t, int T, const float (&v)[kE],
                                            float m, float inv_s) {
    // the register layout follows the input's vector width
    constexpr int V = VecOf<InT>::V;
    constexpr int VO = VecOf<OutT>::V;
    if (vec) {
        #pragma unroll
        for (int k = 0; k < kE / V; ++k) {
            const int32_t e0 = base + (k * T + t) * V;
            float o[V];
            #pragma unroll
            for (int i = 0; i < V; ++i) o[i] = __expf(v[k * V + i] - m) * inv_s;
            if (e0 + V <= end) {
                // V input elements are V * sizeof(OutT) output bytes: one or
                // two 16-byte stores, or one 8-byte store
                if constexpr (V == VO) {
                    uint4 u;
                    OutT* q = reinterpret_cast<OutT*>(&u);
                    #pragma unroll
                    for (int i = 0; i < V; ++i) q[i] = from_f<OutT>(o[i]);
                    __stcs(reinterpret_cast<uint4*>(y + e0), u);
                } else if constexpr (V > VO) {      // 8 16-bit inputs -> 8 FP32 outputs
                    #pragma unroll
                    for (int h = 0; h < V / VO; ++h) {
                        uint4 u;
                        OutT* q = reinterpret_cast<OutT*>(&u);
                        #pragma unroll
                        for (int i = 0; i < VO; ++i) q[i] = from_f<OutT>(o[h * VO + i]);
                        __stcs(reinterpret_cast<uint4*>(y + e0 + h * VO), u);
                    }
                } else {                            // 4 FP32 inputs -> 4 16-bit outputs
                    uint2 u;
                    OutT* q = reinterpret_cast<OutT*>(&u);
                    #pragma unroll
                    for (int i = 0; i < V; ++i) q[i] = from_f<OutT>(o[i]);
                    __stcs(reinterpret_cast<uint2*>(y + e0), u);
                }
            } else {
                #pragma unroll
                for (int i = 0; i < V; ++i)
                    if (e0 + i < end) y[e0 + i] = from_f<OutT>(o[i]);
            }
        }
    } else {
        #pragma unroll
        for (int e = 0; e < kE; ++e) {
            const int32_t i = base + e * T + t;
            if (i < end) y[i] = from_f<OutT>(__expf(v[e] - m) * inv_s);
        }
    }
}

// per-thread (m, s) of a chunk held in registers
__device__ __forceinline__ void chunk_stats(const float (&v)[kE], float& m, float& s) {
    m = -INFINITY;
    #pragma unroll
    for (int e = 0; e < kE; ++e) m = fmax_nan(m, v[e]);
    s = 0.0f;
    if (m != -INFINITY) {
        #pragma unroll
        for (int e = 0; e < kE; ++e) s += __expf(v[e] - m);
    }
}

template <typename InT, typename OutT, bool WARP_ROWS>
__global__ void __launch_bounds__(512)
    softmax_kernel(const __grid_constant__ SoftmaxParams p) {
    const InT* __restrict__ X = static_cast<const InT*>(p.X);
    OutT* __restrict__ Y = static_cast<OutT*>(p.Y);
    const bool vec = p.vec != 0;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;

    // Nothing global is touched before the previous kernel on the stream
    // has completed (programmatic dependent launch).
    gemm103::grid_dependency_wait();

    if constexpr (WARP_ROWS) {
        const int64_t group = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
        const int64_t groups = static_cast<int64_t>(gridDim.x) * nwarps;
        for (int64_t r = group; r < p.rows; r += groups) {
            const InT* x = X + r * p.ldx;
            OutT* y = Y + r * p.ldy;
            float v[kE];
            load_chunk<InT>(x, 0, p.cols, vec, lane, 32, v);
            float m, s;
            chunk_stats(v, m, s);
            warp_merge(m, s);
            store_chunk<InT, OutT>(y, 0, p.cols, vec, lane, 32, v, m, 1.0f / s);
        }
        return;
    } else {
        __shared__ float red_m[2][16], red_s[2][16];
        __shared__ float part_m[2], part_s[2];      // this CTA's pair, per row parity
        const int T = blockDim.x;
        const int CL = p.cluster;
        const uint32_t rank = CL > 1 ? gemm103::cluster_ctarank() : 0u;
        const int64_t group = blockIdx.x / CL;
        const int64_t groups = gridDim.x / CL;
        const int32_t s0 = static_cast<int32_t>(rank) * p.slice;
        const int32_t s1 = p.cols - s0 > p.slice ? s0 + p.slice : p.cols;
        const int32_t chunk = T * kE;
        int parity = 0;
        for (int64_t r = group; r < p.rows; r += groups, parity ^= 1) {
            const InT* x = X + r * p.ldx;
            OutT* y = Y + r * p.ldy;
            float v[kE];
            float m = -INFINITY, s = 0.0f;
            for (int32_t c = s0; c < s1; c += chunk) {
                const int32_t ce = s1 - c > chunk ? c + chunk : s1;
                // a slice of several chunks is read again by the second pass
                // while it is still in L2 (the slices of all resident CTAs,
                // 152 x 512 KB for the longest rows, fit in it)
                if (p.resident) load_chunk<InT, false>(x, c, ce, vec, threadIdx.x, T, v);
                else load_chunk<InT, true>(x, c, ce, vec, threadIdx.x, T, v);
                float mc, sc;
                chunk_stats(v, mc, sc);
                merge(m, s, mc, sc);                 // the online rule, chunk by chunk
                if (p.resident) break;               // one chunk: v keeps the slice
            }
            // CTA: warps -> shared memory -> every thread merges in warp order
            warp_merge(m, s);
            if (lane == 0) {
                red_m[parity][warp] = m;
                red_s[parity][warp] = s;
            }
            __syncthreads();
            m = red_m[parity][0];
            s = red_s[parity][0];
            for (int w = 1; w < nwarps; ++w) merge(m, s, red_m[parity][w], red_s[parity][w]);
            if (CL > 1) {
                // cluster: every CTA publishes its pair, then merges all of
                // them in rank order (the same order in every CTA)
                if (threadIdx.x == 0) {
                    part_m[parity] = m;
                    part_s[parity] = s;
                }
                gemm103::cluster_sync_all();
                const uint32_t am = gemm103::smem_addr(&part_m[parity]);
                const uint32_t as = gemm103::smem_addr(&part_s[parity]);
                for (int q = 0; q < CL; ++q) {
                    float mq, sq;
                    asm volatile("ld.shared::cluster.f32 %0, [%1];"
                                 : "=f"(mq) : "r"(gemm103::map_to_rank(am, q)) : "memory");
                    asm volatile("ld.shared::cluster.f32 %0, [%1];"
                                 : "=f"(sq) : "r"(gemm103::map_to_rank(as, q)) : "memory");
                    if (q == 0) {
                        m = mq;
                        s = sq;
                    } else {
                        merge(m, s, mq, sq);
                    }
                }
            }
            const float inv_s = 1.0f / s;
            if (p.resident) {
                if (s0 < s1) store_chunk<InT, OutT>(y, s0, s1, vec, threadIdx.x, T, v, m, inv_s);
            } else {
                for (int32_t c = s0; c < s1; c += chunk) {
                    const int32_t ce = s1 - c > chunk ? c + chunk : s1;
                    load_chunk<InT>(x, c, ce, vec, threadIdx.x, T, v);
                    store_chunk<InT, OutT>(y, c, ce, vec, threadIdx.x, T, v, m, inv_s);
                }
            }
        }
        // no CTA may leave while a peer can still read its shared memory
        if (CL > 1) gemm103::cluster_sync_all();
    }
}

// Launch one kernel of the plan.  `warp_rows` selects the kernel; threads,
// cluster and grid come from the host planner.
template <typename InT, typename OutT>
cudaError_t launch_softmax(const SoftmaxParams& p, bool warp_rows, int threads, int grid,
                           cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (warp_rows) return cudaLaunchKernelEx(&cfg, softmax_kernel<InT, OutT, true>, p);
    if (p.cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, softmax_kernel<InT, OutT, false>, p);
}

// Resident row groups for a launch shape: CTAs per SM for a single-CTA
// group, or clusters on the whole GPU (cached per shape).
template <typename InT, typename OutT>
int resident_groups(bool warp_rows, int threads, int cluster, int num_sms) {
    static std::mutex mu;
    static int cache[2][2][kMaxCluster + 1] = {};
    const int ti = threads > 256 ? 1 : 0;
    std::lock_guard<std::mutex> g(mu);
    int& c = cache[warp_rows ? 1 : 0][ti][cluster];
    if (c > 0) return c;
    int n = 0;
    if (cluster <= 1) {
        int per_sm = 0;
        cudaError_t e = warp_rows
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_kernel<InT, OutT, true>, threads, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_kernel<InT, OutT, false>, threads, 0);
        if (e != cudaSuccess) cudaGetLastError();
        n = (per_sm > 0 ? per_sm : 1) * num_sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cluster * num_sms, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, softmax_kernel<InT, OutT, false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
        n = clusters > 0 ? clusters : num_sms / cluster;
    }
    c = n > 0 ? n : 1;
    return c;
}

}  // namespace smx
