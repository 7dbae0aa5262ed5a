// softmax_tma.cuh -- the row softmax with rows staged in shared memory by
// bulk copies (TMA), for rows of 256 bytes to 64 KB whose starts are 16-byte
// aligned.
//
// One CTA of 16 warps per SM, split into groups of `group_warps` warps (1 to
// 16, sized so that a row fits in the group's registers at <= 32 elements
// per thread).  Every group is an independent pipeline over its own
// rows with `depth` row slots: its first thread keeps the bulk copies of the
// next depth - 1 rows in flight while the group works on one, so an SM has
// ~130-190 KB of loads outstanding without registers holding them, and up to
// 16 rows are worked on at once.  A row is moved from its slot into registers
// once, as FP32; the maximum (NaN-propagating), e = exp(x - m) with its sum,
// and the output e / s then run on the registers -- the three steps of the
// SGEMM tutorial page, section 2.1, with HBM and shared memory each read once
// and one exponential per element.  The
// last (cols * size) % 16 bytes of a row, which a bulk copy cannot move, are
// read from global memory directly.
//
// Every wait is bounded; a wait that runs out sets the error word, waits
// (bounded) for the group's other copies to land and leaves.
#pragma once
#include <cstdint>
#include <mutex>

#include "softmax_kern.cuh"

namespace smx {

constexpr int kTmaThreads = 512;         // 16 warps
constexpr int kTmaMaxDepth = 8;
constexpr int kTmaMaxElems = 32;         // row elements per thread (held as FP32)
constexpr uint32_t kSmxDebugSkipFirstLoad = 1u;

struct TmaSoftmaxParams {
    const void* X;
    void* Y;
    int64_t ldx, ldy;
    int64_t rows;
    int32_t cols;
    int32_t bulk_elems;     // elements moved by the bulk copy: (cols * size) rounded down to 16 B
    int32_t slot_bytes;     // one row slot (row bytes rounded up to 128)
    int32_t depth;          // slots per group
    int32_t group_warps;    // warps per group (power of two, 1..16)
    int32_t unit_rows;      // rows per slot: 1 (the group shares the row) or a multiple of
                            // group_warps (each warp of the group takes its own rows)
    int32_t row_stride;     // bytes from one row to the next inside a slot
    int32_t contiguous;     // 1: a slot's rows are adjacent in X, one copy moves them all
    int32_t kv;             // 16-byte vectors per thread: 1, 2, 4 (or 8 for FP32 input)
    int* err;               // device error word (1: a wait ran out)
    uint64_t wait_limit_ns;
    uint32_t debug_flags;
};

__device__ __forceinline__ float warp_max(float m) {
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, off));
    return m;
}

__device__ __forceinline__ float warp_sum(float s) {
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// Barrier of the group's threads (named barrier 1 + group); a single-warp
// group needs only __syncwarp.
__device__ __forceinline__ void group_sync(int gw, int group) {
    if (gw == 1) {
        __syncwarp();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(gw * 32) : "memory");
    }
}

// true on every thread of the group iff `pred` is true on all of them
__device__ __forceinline__ bool group_all(int gw, int group, bool pred) {
    if (gw == 1) return __all_sync(0xffffffffu, pred) != 0;
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(1 + group), "r"(gw * 32)
        : "memory");
    return r != 0;
}

template <typename InT, typename OutT>
__device__ __forceinline__ void store_vec16(OutT* dst, const float (&o)[VecOf<InT>::V]) {
    constexpr int V = VecOf<InT>::V;
    constexpr int VO = VecOf<OutT>::V;
    if constexpr (V == VO) {
        uint4 w;
        OutT* r = reinterpret_cast<OutT*>(&w);
        #pragma unroll
        for (int i = 0; i < V; ++i) r[i] = from_f<OutT>(o[i]);
        __stcs(reinterpret_cast<uint4*>(dst), w);
    } else if constexpr (V > VO) {               // 8 16-bit inputs -> 8 FP32 outputs
        #pragma unroll
        for (int h = 0; h < V / VO; ++h) {
            uint4 w;
            OutT* r = reinterpret_cast<OutT*>(&w);
            #pragma unroll
            for (int i = 0; i < VO; ++i) r[i] = from_f<OutT>(o[h * VO + i]);
            __stcs(reinterpret_cast<uint4*>(dst + h * VO), w);
        }
    } else {                                     // 4 FP32 inputs -> 4 16-bit outputs
        uint2 w;
        OutT* r = reinterpret_cast<OutT*>(&w);
        #pragma unroll
        for (int i = 0; i < V; ++i) r[i] = from_f<OutT>(o[i]);
        __stcs(reinterpret_cast<uint2*>(dst), w);
    }
}

// Arm `bar` for the rows of unit u and issue their copies: one copy when the
// rows are adjacent in X, else one per row (unless the test hook says not to).
// bulk_elems: the elements of a row moved by the copy.
template <typename InT>
__device__ __forceinline__ void issue_unit(const TmaSoftmaxParams& p, const InT* X,
                                           int32_t bulk_elems, uint8_t* slot, int64_t u,
                                           uint64_t* bar, uint64_t policy, bool skip) {
    const int64_t first = u * p.unit_rows;
    const int64_t left = p.rows - first;
    const uint32_t nr = static_cast<uint32_t>(left < p.unit_rows ? left : p.unit_rows);
    const uint32_t bytes = static_cast<uint32_t>(bulk_elems) * sizeof(InT);
    gemm103::mbar_arrive_expect_tx(bar, nr * bytes);
    if (skip) return;
    if (p.contiguous) {
        gemm103::bulk_load_1d(slot, X + first * p.ldx, nr * bytes, bar, policy);
    } else {
        for (uint32_t j = 0; j < nr; ++j)
            gemm103::bulk_load_1d(slot + static_cast<size_t>(j) * p.row_stride,
                                  X + (first + j) * p.ldx, bytes, bar, policy);
    }
}

// One row from its slot: KV 16-byte vectors per thread (vector k of thread t
// is vector t + k * T) into registers as FP32 -- each element converted once
// -- then the maximum, e = exp(x - m) kept in place of x, s = sum e, and the
// output e / s.  One exponential per element.  The T threads are one warp
// (gw = 1) or the group's gw warps, which combine their partial results
// through red_m / red_s and the group barrier.
template <typename InT, typename OutT, int KV>
__device__ __forceinline__ void process_row(const uint8_t* srow, const InT* __restrict__ grow,
                                            OutT* __restrict__ yrow, int32_t nvec,
                                            int32_t bulk_elems, int32_t cols, int t, int T,
                                            int gw, int group, int warp, int lane,
                                            float* red_m, float* red_s) {
    constexpr int V = VecOf<InT>::V;
    // FP32 input: the raw vectors stay in registers and the output pass
    // evaluates exp(x - m) again next to its stores (the row is bound by HBM,
    // and this order keeps the stores spread over the pass); 16-bit input:
    // each element is converted once and exp(x - m) is kept (the row is
    // bound by the per-element arithmetic).
    constexpr bool kKeepExp = sizeof(InT) == 2;
    float x[KV][V];
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int32_t v = t + k * T;
        if (v < nvec) {
            const uint4 u = *reinterpret_cast<const uint4*>(srow + static_cast<size_t>(v) * 16);
            const InT* q = reinterpret_cast<const InT*>(&u);
            #pragma unroll
            for (int e = 0; e < V; ++e) x[k][e] = to_f(q[e]);
        } else {
            #pragma unroll
            for (int e = 0; e < V; ++e) x[k][e] = -INFINITY;
        }
    }
    const int32_t te = bulk_elems + t;                  // at most one tail element each
    float xt = te < cols ? to_f(grow[te]) : -INFINITY;

    float m = xt;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        #pragma unroll
        for (int e = 0; e < V; ++e) m = fmax_nan(m, x[k][e]);
    }
    m = warp_max(m);
    if (gw > 1) {
        if (lane == 0) red_m[warp] = m;
        group_sync(gw, group);
        m = red_m[group * gw];
        for (int w = 1; w < gw; ++w) m = fmax_nan(m, red_m[group * gw + w]);
    }
    // padding entries are -inf: exp gives 0 unless m is -inf or +inf or NaN,
    // in which case the row is NaN anyway
    float s = 0.0f;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        #pragma unroll
        for (int e = 0; e < V; ++e) {
            const float ex = __expf(x[k][e] - m);
            if constexpr (kKeepExp) x[k][e] = ex;
            s += ex;
        }
    }
    xt = __expf(xt - m);
    if (te < cols) s += xt;
    s = warp_sum(s);
    if (gw > 1) {
        if (lane == 0) red_s[warp] = s;
        group_sync(gw, group);
        s = red_s[group * gw];
        for (int w = 1; w < gw; ++w) s += red_s[group * gw + w];
    }
    const float inv_s = 1.0f / s;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int32_t v = t + k * T;
        if (v < nvec) {
            float o[V];
            #pragma unroll
            for (int e = 0; e < V; ++e)
                o[e] = (kKeepExp ? x[k][e] : __expf(x[k][e] - m)) * inv_s;
            store_vec16<InT, OutT>(yrow + static_cast<int64_t>(v) * V, o);
        }
    }
    if (te < cols) yrow[te] = from_f<OutT>(xt * inv_s);
}

template <typename InT, typename OutT, int KV>
__global__ void __launch_bounds__(kTmaThreads, 1)
    softmax_tma_kernel(const __grid_constant__ TmaSoftmaxParams p) {
    constexpr int V = VecOf<InT>::V;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ float red_m[16], red_s[16];      // per warp, reduced within its group
    const InT* __restrict__ X = static_cast<const InT*>(p.X);
    OutT* __restrict__ Y = static_cast<OutT*>(p.Y);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int GW = p.group_warps;
    const int GT = GW * 32;
    const int NG = (blockDim.x >> 5) / GW;
    const int group = warp / GW;
    const int gt = threadIdx.x - group * GT;     // thread index within the group
    const int D = p.depth;
    const int32_t nvec = p.bulk_elems / V;
    // layout: [barriers: one per slot, 128 B aligned][slots]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint8_t* slots = smem_raw + ((NG * D * 8 + 127) / 128) * 128;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NG * D; ++i) gemm103::mbar_init(&bars[i], 1);
        gemm103::fence_barrier_init();
    }
    __syncthreads();
    gemm103::grid_dependency_wait();      // inputs of the previous kernel are visible
    const uint64_t policy = gemm103::l2_policy_evict_first();

    // this group's units (slots' worth of rows): u0, u0 + stride, ...; n in all
    const int64_t units = (p.rows + p.unit_rows - 1) / p.unit_rows;
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * NG + group;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * NG;
    const int64_t n = u0 < units ? (units - 1 - u0) / stride + 1 : 0;
    uint64_t* pb = bars + group * D;
    uint8_t* ps = slots + static_cast<size_t>(group) * D * p.slot_bytes;
    const bool issuer = (gt == 0);
    const bool skip_first = (p.debug_flags & kSmxDebugSkipFirstLoad) && blockIdx.x == 0 && group == 0;
    const int wg = warp - group * GW;                 // warp index within the group

    if (issuer) {
        for (int64_t i = 0; i < n && i < D - 1; ++i)
            issue_unit<InT>(p, X, p.bulk_elems, ps + (i % D) * p.slot_bytes, u0 + i * stride,
                            &pb[i % D], policy, skip_first && i == 0);
    }
    int64_t i = 0;
    for (; i < n; ++i) {
        // the slot of unit i - 1 is free (the group is past it): refill it
        // with unit i + D - 1
        const int64_t nxt = i + D - 1;
        if (issuer && nxt < n)
            issue_unit<InT>(p, X, p.bulk_elems, ps + (nxt % D) * p.slot_bytes, u0 + nxt * stride,
                            &pb[nxt % D], policy, false);
        bool ok = gemm103::mbar_wait(&pb[i % D], static_cast<uint32_t>((i / D) & 1),
                                     p.wait_limit_ns);
        ok = group_all(GW, group, ok);
        if (!ok) {
            if (issuer) atomicExch(p.err, 1);
            break;
        }
        const int64_t first = (u0 + i * stride) * p.unit_rows;
        const uint8_t* sunit = ps + (i % D) * p.slot_bytes;
        if (p.unit_rows == 1) {
            // the group shares the row
            process_row<InT, OutT, KV>(sunit, X + first * p.ldx, Y + first * p.ldy, nvec,
                                       p.bulk_elems, p.cols, gt, GT, GW, group, warp, lane, red_m,
                                       red_s);
        } else {
            // each warp of the group takes its own rows of the unit
            const int64_t left = p.rows - first;
            const int nr = static_cast<int>(left < p.unit_rows ? left : p.unit_rows);
            for (int j = wg; j < nr; j += GW)
                process_row<InT, OutT, KV>(sunit + static_cast<size_t>(j) * p.row_stride,
                                           X + (first + j) * p.ldx, Y + (first + j) * p.ldy,
                                           nvec, p.bulk_elems, p.cols, lane, 32, 1, group, warp,
                                           lane, red_m, red_s);
        }
        // every thread is past this unit's slot and reduction words
        group_sync(GW, group);
    }
    if (i < n && issuer) {
        // a wait ran out: let the copies already issued into this group's slots (units i .. i + D - 1)
        // land before shared memory is released
        const int64_t last = i + D < n ? i + D : n;
        for (int64_t j = i; j < last; ++j)
            gemm103::mbar_wait(&pb[j % D], static_cast<uint32_t>((j / D) & 1), p.wait_limit_ns);
    }
}

template <typename InT, typename OutT, int KV>
cudaError_t launch_softmax_tma_kv(const TmaSoftmaxParams& p, int grid, size_t smem,
                                  cudaStream_t stream) {
    auto kern = softmax_tma_kernel<InT, OutT, KV>;
    {
        static std::mutex mu;
        static size_t raised = 0;
        std::lock_guard<std::mutex> g(mu);
        if (smem > raised) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            raised = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename InT, typename OutT>
cudaError_t launch_softmax_tma(const TmaSoftmaxParams& p, int grid, size_t smem,
                               cudaStream_t stream) {
    constexpr int kMaxKV = kTmaMaxElems / VecOf<InT>::V;
    switch (p.kv) {
        case 1: return launch_softmax_tma_kv<InT, OutT, 1>(p, grid, smem, stream);
        case 2: return launch_softmax_tma_kv<InT, OutT, 2>(p, grid, smem, stream);
        case 4: return launch_softmax_tma_kv<InT, OutT, 4>(p, grid, smem, stream);
        case 8:
            if constexpr (kMaxKV >= 8)
                return launch_softmax_tma_kv<InT, OutT, 8>(p, grid, smem, stream);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace smx
