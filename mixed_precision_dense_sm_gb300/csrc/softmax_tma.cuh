// softmax_tma.cuh -- the row softmax with rows staged in shared memory by
// bulk copies (TMA), for rows of 256 bytes to 64 KB whose starts are 16-byte
// aligned.
//
// One CTA per SM: 16 compute warps in groups of `group_warps` warps (1 to 16,
// sized so that a row fits in the group's registers at <= 8 16-byte vectors
// per thread: 32 FP32 or 64 16-bit elements) and one producer warp.  Each
// group owns a ring of `depth` row slots, each slot with a "full" mbarrier
// (the bulk copy's bytes) and an "empty" one (one arrival per warp of the
// group once it has read the slot).  The producer's first thread keeps the
// rings filled: the groups take equal rows at the same pace, so it refills in
// one fixed order (unit i of every group, then unit i + 1), waiting on each
// slot's empty barrier in turn, and no barrier ties the warps of a group
// together between units.  An SM keeps ~130-190 KB of loads in flight
// without registers holding them.
//
// A row is moved from its slot into registers once, as FP32; the slot is
// released right then; the maximum (NaN-propagating), e = exp(x - m) with its
// sum, and the output e / s then run on the registers -- the three steps of
// the SGEMM tutorial page, section 2.1, with HBM and shared memory each read
// once.  A row shared by several warps merges its warps' (max, sum) pairs
// through shared memory at one group barrier.  When a row is whole in the
// vectors the threads hold (no 16-byte tail, every vector slot used) the
// kernel runs a variant without per-vector bounds checks.  The last
// (cols * size) % 16 bytes of a row, which a bulk copy cannot move, are read
// from global memory directly.
//
// Every wait is bounded; a wait that runs out sets the error word.  Compute
// warps that give up leave their loop; the producer stops refilling once a
// slot stays unread past the limit and, before the CTA exits, waits
// (bounded) for every copy it issued to land.
#pragma once
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "softmax_kern.cuh"

namespace smx {

constexpr int kTmaComputeWarps = 16;
constexpr int kTmaThreads = (kTmaComputeWarps + 1) * 32;    // + the producer warp
constexpr int kTmaMaxDepth = 8;
constexpr int kTmaMaxGroups = kTmaComputeWarps;
constexpr int kTmaMaxVec = 8;           // 16-byte row vectors per thread: 32 FP32 or 64 16-bit
                                         // elements, held as FP32
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
    int32_t whole;          // 1: bulk_elems == cols and every thread holds kv vectors
    int32_t long_rows;      // 1: rows streamed twice in chunks (softmax_long_kernel)
    int32_t cluster;        // long rows: CTAs per row (a thread-block cluster when > 1)
    int32_t slice;          // long rows: elements of a row per CTA (a multiple of 8)
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

// true on every thread of the group iff `pred` is true on all of them (a
// group barrier as well)
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

// Eight 16-bit values of a 16-byte vector as FP32 (a BF16 is the top half of
// its FP32; FP16 converts by pairs), or four FP32 values as they are.
template <typename InT>
__device__ __forceinline__ void unpack16(const uint4 u, float* x);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 u, float* x) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void unpack16<__half>(const uint4 u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// V (one input vector's worth of) FP32 outputs, cast and stored with
// streaming 16-byte (or 8-byte) stores.
template <typename InT, typename OutT>
__device__ __forceinline__ void store_vec16(OutT* dst, const float (&o)[VecOf<InT>::V]) {
    constexpr int V = VecOf<InT>::V;
    if constexpr (sizeof(OutT) == 2) {
        uint32_t w[V / 2];
        #pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            if constexpr (std::is_same<OutT, __nv_bfloat16>::value) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __half2 h = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        if constexpr (V == 8) __stcs(reinterpret_cast<uint4*>(dst), make_uint4(w[0], w[1], w[2], w[3]));
        else __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
    } else {
        #pragma unroll
        for (int h = 0; h < V / 4; ++h)
            __stcs(reinterpret_cast<float4*>(dst + 4 * h),
                   make_float4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]));
    }
}

// e^t per element.  Rows of 16-bit inputs use the identity e^t = 2^(t log2 e):
// the product rounded once to FP32, then the hardware base-2 exponential
// (PTX ex2.approx.ftz.f32), so the error is the exponential's own plus
// |t| 2^-24 relative from the product -- the same form as the bound of
// __expf, which rows of FP32 inputs keep (measured faster on them).
// Results below 2^-126 flush to zero.
template <typename InT>
__device__ __forceinline__ float exp_elem(float t) {
    if constexpr (sizeof(InT) == 2) {
        float r;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t * 1.4426950408889634f));
        return r;
    } else {
        return __expf(t);
    }
}

// Arm `bar` for the rows of unit u and issue their copies: one copy when the
// rows are adjacent in X, else one per row (unless the test hook says not to).
template <typename InT>
__device__ __forceinline__ void issue_unit(const TmaSoftmaxParams& p, const InT* X, uint8_t* slot,
                                           int64_t u, uint64_t* bar, uint64_t policy, bool skip) {
    const int64_t first = u * p.unit_rows;
    const int64_t left = p.rows - first;
    const uint32_t nr = static_cast<uint32_t>(left < p.unit_rows ? left : p.unit_rows);
    const uint32_t bytes = static_cast<uint32_t>(p.bulk_elems) * sizeof(InT);
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

// The row's values held by this thread: KV 16-byte vectors (vector k of
// thread t is vector t + k * T of the row) converted to FP32 once, plus at
// most one tail element past the bulk-copied part.  WHOLE: every vector slot
// is inside the row and there is no tail.
template <typename InT, int KV, bool WHOLE>
__device__ __forceinline__ void load_row(const uint8_t* srow, const InT* __restrict__ grow,
                                         int32_t nvec, int32_t bulk_elems, int32_t cols, int t,
                                         int T, float (&x)[KV][VecOf<InT>::V], float& xt) {
    constexpr int V = VecOf<InT>::V;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int32_t v = t + k * T;
        if (WHOLE || v < nvec) {
            unpack16<InT>(*reinterpret_cast<const uint4*>(srow + static_cast<size_t>(v) * 16), x[k]);
        } else {
            #pragma unroll
            for (int e = 0; e < V; ++e) x[k][e] = -INFINITY;
        }
    }
    xt = -INFINITY;
    if (!WHOLE) {
        const int32_t te = bulk_elems + t;
        if (te < cols) xt = to_f(grow[te]);
    }
}

// The rest of one row from registers: maximum, exponentials and their sum,
// output.  One exponential per element: e = exp(x - m) replaces x.  The T
// threads are one warp (gw = 1, shuffles only) or the group's gw warps.  A
// group meets once per row: each warp exponentiates against its own maximum
// m_w and publishes (m_w, s_w) in red_m / red_s (buffer `buf`, alternating
// between consecutive rows, so a warp that runs ahead never overwrites pairs
// another warp has yet to read); after the group barrier every warp merges
// the pairs by the online rule (SGEMM tutorial page, section 2.2):
//     M = max m_w,  S = sum_w s_w exp(m_w - M)   (a warp whose elements are
//     all -inf contributes 0),
// and scales its e by exp(m_w - M) / S.  NaN in any m_w makes the row NaN,
// as do +inf (inf - inf) and a fully masked row (S = 0).  `ok` (the slot's
// data arrived) is combined over the group at that barrier and the row is
// abandoned unless it holds everywhere.  Returns that.
template <typename InT, typename OutT, int KV, bool WHOLE>
__device__ __forceinline__ bool finish_row(float (&x)[KV][VecOf<InT>::V], float xt, bool ok,
                                           OutT* __restrict__ yrow, int32_t nvec,
                                           int32_t bulk_elems, int32_t cols, int t, int T, int gw,
                                           int group, int warp, int lane, float* red_m,
                                           float* red_s) {
    constexpr int V = VecOf<InT>::V;
    float m = xt;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        #pragma unroll
        for (int e = 0; e < V; ++e) m = fmax_nan(m, x[k][e]);
    }
    m = warp_max(m);
    // this warp's elements are all -inf: its e are 0 (not exp(-inf - -inf))
    const float mz = (m == -INFINITY) ? 0.0f : m;
    float s = 0.0f;
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        #pragma unroll
        for (int e = 0; e < V; ++e) {
            x[k][e] = exp_elem<InT>(x[k][e] - mz);
            s += x[k][e];
        }
    }
    if (!WHOLE) {
        xt = exp_elem<InT>(xt - mz);
        if (bulk_elems + t < cols) s += xt;
    }
    s = warp_sum(s);
    float scale;
    if (gw > 1) {
        if (lane == 0) {
            red_m[warp] = m;
            red_s[warp] = s;
        }
        ok = group_all(gw, group, ok);
        if (!ok) return false;
        // lanes 0 .. gw-1 merge the gw pairs by a butterfly over log2(gw)
        // levels, (m1, s1) + (m2, s2) = (M, s1 e^(m1 - M) + s2 e^(m2 - M)),
        // a side with m = -inf contributing 0; lane 0's result is everyone's
        // (every lane of the butterfly ends with the same bits)
        const int li = lane & (gw - 1);
        float Mi = red_m[group * gw + li];
        float Si = red_s[group * gw + li];
        for (int off = gw >> 1; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, Mi, off);
            const float so = __shfl_xor_sync(0xffffffffu, Si, off);
            const float mm = fmax_nan(Mi, mo);
            const float mmz = (mm == -INFINITY) ? 0.0f : mm;
            Si = (Mi == -INFINITY ? 0.0f : Si * __expf(Mi - mmz)) +
                 (mo == -INFINITY ? 0.0f : so * __expf(mo - mmz));
            Mi = mm;
        }
        const float Mz = (Mi == -INFINITY) ? 0.0f : Mi;
        scale = (m == -INFINITY ? 0.0f : __expf(m - Mz)) / Si;
    } else {
        ok = __all_sync(0xffffffffu, ok) != 0;
        if (!ok) return false;
        scale = 1.0f / s;
    }
    #pragma unroll
    for (int k = 0; k < KV; ++k) {
        const int32_t v = t + k * T;
        if (WHOLE || v < nvec) {
            float o[V];
            #pragma unroll
            for (int e = 0; e < V; ++e) o[e] = x[k][e] * scale;
            store_vec16<InT, OutT>(yrow + static_cast<int64_t>(v) * V, o);
        }
    }
    if (!WHOLE) {
        const int32_t te = bulk_elems + t;
        if (te < cols) yrow[te] = from_f<OutT>(xt * scale);
    }
    return true;
}

template <typename InT, typename OutT, int KV, bool WHOLE>
__global__ void __launch_bounds__(kTmaThreads, 1)
    softmax_tma_kernel(const __grid_constant__ TmaSoftmaxParams p) {
    constexpr int V = VecOf<InT>::V;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // per warp (m_w, s_w) of a shared row, two buffers alternating by row
    __shared__ float red_m[2][kTmaComputeWarps], red_s[2][kTmaComputeWarps];
    const InT* __restrict__ X = static_cast<const InT*>(p.X);
    OutT* __restrict__ Y = static_cast<OutT*>(p.Y);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int GW = p.group_warps;
    const int GT = GW * 32;
    const int NG = kTmaComputeWarps / GW;
    const int D = p.depth;
    const int32_t nvec = p.bulk_elems / V;
    // layout: [full barriers NG * D][empty barriers NG * D] (128-byte aligned) [slots]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw);
    uint64_t* empty = full + NG * D;
    uint8_t* slots = smem_raw + ((2 * NG * D * 8 + 127) / 128) * 128;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NG * D; ++i) {
            gemm103::mbar_init(&full[i], 1);
            gemm103::mbar_init(&empty[i], GW);
        }
        gemm103::fence_barrier_init();
    }
    __syncthreads();
    gemm103::grid_dependency_wait();      // inputs of the previous kernel are visible

    // group g's units (slots' worth of rows): g0, g0 + stride, ... with
    // g0 = blockIdx.x * NG + g; n(g) of them
    const int64_t units = (p.rows + p.unit_rows - 1) / p.unit_rows;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * NG;
    auto units_of = [&](int g) -> int64_t {
        const int64_t u0 = static_cast<int64_t>(blockIdx.x) * NG + g;
        return u0 < units ? (units - 1 - u0) / stride + 1 : 0;
    };

    if (warp == kTmaComputeWarps) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t policy = gemm103::l2_policy_evict_first();
        const bool skip_first = (p.debug_flags & kSmxDebugSkipFirstLoad) && blockIdx.x == 0;
        // Every group's i-th unit goes to its slot i % D, and the groups
        // consume at the same pace (equal rows), so the refills run in one
        // fixed order -- unit i of group 0, 1, ..., NG - 1, then unit i + 1 --
        // each waiting (bounded, the thread suspended in the barrier's
        // try_wait) for its slot's "empty" phase.  The loop's state is a few
        // scalars: no per-group tables to reload on every poll.
        int64_t issued[kTmaMaxGroups];    // per group; read only at the end
        // every slot starts free: the first D units of each group at once
        for (int g = 0; g < NG; ++g) {
            const int64_t n = units_of(g);
            const int64_t u0 = static_cast<int64_t>(blockIdx.x) * NG + g;
            for (int64_t i = 0; i < n && i < D; ++i)
                issue_unit<InT>(p, X, slots + (static_cast<size_t>(g) * D + i) * p.slot_bytes,
                                u0 + i * stride, &full[g * D + i], policy,
                                skip_first && g == 0 && i == 0);
            issued[g] = n < D ? n : D;
        }
        int d = 0;                        // slot of unit i; unit i - D's "empty" parity
        uint32_t par = 0;
        bool alive = true;
        for (int64_t i = D; alive; ++i) {
            bool any = false;
            for (int g = 0; g < NG; ++g) {
                const int64_t u = static_cast<int64_t>(blockIdx.x) * NG + g + i * stride;
                if (u >= units) break;    // nor for the groups after g
                any = true;
                if (!gemm103::mbar_wait(&empty[g * D + d], par, p.wait_limit_ns)) {
                    // the slot was never read: the consumers gave up
                    atomicExch(p.err, 1);
                    alive = false;
                    break;
                }
                issue_unit<InT>(p, X, slots + (static_cast<size_t>(g) * D + d) * p.slot_bytes, u,
                                &full[g * D + d], policy, false);
                issued[g] = i + 1;
            }
            if (!any) break;
            if (++d == D) {
                d = 0;
                par ^= 1u;
            }
        }
        // every copy issued lands before the CTA (and its shared memory) goes
        for (int g = 0; g < NG; ++g) {
            const int64_t n = issued[g];
            for (int64_t i = n > D ? n - D : 0; i < n; ++i)
                gemm103::mbar_wait(&full[g * D + static_cast<int>(i % D)],
                                   static_cast<uint32_t>((i / D) & 1), p.wait_limit_ns);
        }
        return;
    }

    // ------------------------------------------------------------ compute
    const int group = warp / GW;
    const int gt = threadIdx.x - group * GT;     // thread index within the group
    const int wg = warp - group * GW;            // warp index within the group
    const int64_t n = units_of(group);
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * NG + group;
    uint64_t* pf = full + group * D;
    uint64_t* pe = empty + group * D;
    const uint8_t* ps = slots + static_cast<size_t>(group) * D * p.slot_bytes;
    int d = 0;                                   // slot of unit i, and its "full" parity
    uint32_t par = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (i > 0 && ++d == D) {
            d = 0;
            par ^= 1u;
        }
        bool ok = gemm103::mbar_wait(&pf[d], par, p.wait_limit_ns);
        const int64_t first = (u0 + i * stride) * p.unit_rows;
        const uint8_t* sunit = ps + static_cast<size_t>(d) * p.slot_bytes;
        float x[KV][V];
        float xt;
        if (p.unit_rows == 1) {
            // the group shares the row: read it, release the slot, finish it
            load_row<InT, KV, WHOLE>(sunit, X + first * p.ldx, nvec, p.bulk_elems, p.cols, gt, GT,
                                     x, xt);
            __syncwarp();
            if (lane == 0) gemm103::mbar_arrive(&pe[d]);
            ok = finish_row<InT, OutT, KV, WHOLE>(x, xt, ok, Y + first * p.ldy, nvec, p.bulk_elems,
                                                  p.cols, gt, GT, GW, group, warp, lane,
                                                  red_m[i & 1], red_s[i & 1]);
        } else {
            // each warp of the group takes its own rows of the unit
            ok = __all_sync(0xffffffffu, ok) != 0;
            if (ok) {
                const int64_t left = p.rows - first;
                const int nr = static_cast<int>(left < p.unit_rows ? left : p.unit_rows);
                for (int j = wg; j < nr; j += GW) {
                    load_row<InT, KV, WHOLE>(sunit + static_cast<size_t>(j) * p.row_stride,
                                             X + (first + j) * p.ldx, nvec, p.bulk_elems, p.cols,
                                             lane, 32, x, xt);
                    if (j + GW >= nr) {
                        // this warp's last read of the slot
                        __syncwarp();
                        if (lane == 0) gemm103::mbar_arrive(&pe[d]);
                    }
                    finish_row<InT, OutT, KV, WHOLE>(x, xt, true, Y + (first + j) * p.ldy, nvec,
                                                     p.bulk_elems, p.cols, lane, 32, 1, group, warp,
                                                     lane, red_m[0], red_s[0]);
                }
                if (wg >= nr) {
                    __syncwarp();
                    if (lane == 0) gemm103::mbar_arrive(&pe[d]);
                }
            }
        }
        if (!ok) {
            if (gt == 0) atomicExch(p.err, 1);
            break;
        }
    }
}

// ------------------------------------------------------------ long rows
// Rows longer than the staged kernel holds (more than 64 KB or more vectors
// than its threads keep), 16-byte aligned, whose slices on all SMs fit the
// L2 budget: one CTA of 16 compute warps and a producer warp per SM takes
// rows in turn and streams each twice through a ring of kLongDepth slots of
// kLongChunkBytes -- the two-pass scheme of the SGEMM tutorial page, section
// 2.2, with the loads moved by bulk copies instead of registers.  Pass 1
// folds the row chunk by chunk into per-thread (m, s) by the online rule
// (m' = max(m, c), s' = s e^(m - m') + sum e^(x - m') over the chunk), and
// the CTA merges its 512 pairs (warp butterflies, then the 16 warps' pairs
// in one fixed order, so every thread holds the same (M, S)).  Pass 2 reads
// the chunks again -- from L2: pass 1's copies are evict-normal, pass 2's
// evict-first -- and writes y = e^(x - M) / S.
constexpr int kLongKV = 4;                                          // vectors per thread per chunk
constexpr int kLongChunkBytes = kTmaComputeWarps * 32 * kLongKV * 16;  // 32 KB
constexpr int kLongDepth = 6;
constexpr int kMaxLongCluster = 8;

// Bounded wait that also gives up once another thread of the CTA has set
// `abort` (the clock is read every 64 tries).
__device__ __forceinline__ bool wait_abortable(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
    const uint32_t a = gemm103::smem_addr(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (gemm103::mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            const uint64_t now = gemm103::global_timer_ns();
            if (i == 64u) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// (m, s) of this CTA's part of a row sent to every CTA of the cluster: the
// pair into the peer's receive buffer (slot `rank`), then a release-arrive on
// the peer's exchange barrier, which counts one arrival per CTA.
__device__ __forceinline__ void send_pair(float m, float s, float* recv_m, float* recv_s,
                                          uint64_t* xbar, uint32_t rank, int cl) {
    const uint32_t am = gemm103::smem_addr(recv_m + rank);
    const uint32_t as = gemm103::smem_addr(recv_s + rank);
    const uint32_t ab = gemm103::smem_addr(xbar);
    for (int q = 0; q < cl; ++q) {
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(gemm103::map_to_rank(am, q)), "f"(m)
                     : "memory");
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(gemm103::map_to_rank(as, q)), "f"(s)
                     : "memory");
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                     ::"r"(gemm103::map_to_rank(ab, q)) : "memory");
    }
}

// Bounded wait on a barrier that peers of the cluster arrive on.
__device__ __forceinline__ bool wait_peers(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           uint64_t limit_ns) {
    const uint32_t a = gemm103::smem_addr(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (gemm103::mbar_try_wait_cluster(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            const uint64_t now = gemm103::global_timer_ns();
            if (i == 64u) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// A row longer than one CTA's share of L2 is split over a cluster of
// p.cluster CTAs (slice p.slice elements each); after pass 1 every CTA sends
// its (m, s) to all the others, and each merges the cluster's pairs in rank
// order, so all hold the same (M, S).  Every loop of every thread is bounded
// and no thread leaves early: the rows, chunks and exchanges of a cluster
// run the same count on all its CTAs whatever fails, and the CTAs meet once
// more before they exit, so no CTA can go while a peer still writes to it.
template <typename InT, typename OutT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    softmax_long_kernel(const __grid_constant__ TmaSoftmaxParams p) {
    constexpr int V = VecOf<InT>::V;
    constexpr int T = kTmaComputeWarps * 32;                 // compute threads
    constexpr int D = kLongDepth;
    constexpr int32_t kChunkElems = kLongChunkBytes / static_cast<int>(sizeof(InT));
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ float red_m[2][kTmaComputeWarps], red_s[2][kTmaComputeWarps];
    __shared__ float recv_m[2][kMaxLongCluster], recv_s[2][kMaxLongCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ int abort_flag;
    const InT* __restrict__ X = static_cast<const InT*>(p.X);
    OutT* __restrict__ Y = static_cast<OutT*>(p.Y);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int CL = p.cluster;
    const uint32_t rank = CL > 1 ? gemm103::cluster_ctarank() : 0u;
    const int64_t cid = blockIdx.x / CL;                       // this CTA's cluster
    const int64_t nclusters = gridDim.x / CL;
    // this CTA's part of every row: elements [e_lo, e_lo + nb) by bulk copies,
    // and the tail [bulk_elems, cols) in the CTA whose part ends the row
    const int32_t e_lo = static_cast<int32_t>(rank) * p.slice;
    const int32_t e_hi = p.cols - e_lo < p.slice ? p.cols : e_lo + p.slice;
    const bool ends_row = e_hi == p.cols;
    const int32_t b_hi = ends_row ? p.bulk_elems : e_hi;
    const int32_t nb = b_hi > e_lo ? b_hi - e_lo : 0;
    const int32_t C = (nb + kChunkElems - 1) / kChunkElems;   // chunks per pass
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw);
    uint64_t* empty = full + D;
    uint8_t* slots = smem_raw + 1024;
    if (threadIdx.x == 0) {
        for (int i = 0; i < D; ++i) {
            gemm103::mbar_init(&full[i], 1);
            gemm103::mbar_init(&empty[i], kTmaComputeWarps);
        }
        gemm103::mbar_init(&xbar[0], CL);
        gemm103::mbar_init(&xbar[1], CL);
        abort_flag = 0;
        gemm103::fence_barrier_init();
    }
    // every CTA's barriers are initialised before a peer arrives on them
    if (CL > 1) gemm103::cluster_sync_all();
    else __syncthreads();
    gemm103::grid_dependency_wait();      // inputs of the previous kernel are visible

    if (warp == kTmaComputeWarps) {
        // ------------------------------------------------------- producer
        // unit i of this CTA: row cid + (i / 2C) nclusters, pass (i % 2C) / C,
        // chunk (i % 2C) % C; slot i % D
        if (lane == 0) {
            const uint64_t keep = gemm103::l2_policy_evict_normal();
            const uint64_t last = gemm103::l2_policy_evict_first();
            const bool skip_first = (p.debug_flags & kSmxDebugSkipFirstLoad) && blockIdx.x == 0;
            int64_t issued = 0;
            int d = 0;
            uint32_t round = 0;               // times slot 0 has been reached
            bool ok = true;
            for (int64_t row = cid; ok && row < p.rows; row += nclusters) {
                for (int32_t j = 0; j < 2 * C; ++j) {
                    if (round > 0 &&
                        !wait_abortable(&empty[d], (round - 1) & 1u, &abort_flag, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    const int32_t c = j < C ? j : j - C;
                    const int32_t e0 = c * kChunkElems;
                    const int32_t n = nb - e0 < kChunkElems ? nb - e0 : kChunkElems;
                    const uint32_t bytes = static_cast<uint32_t>(n) * sizeof(InT);
                    gemm103::mbar_arrive_expect_tx(&full[d], bytes);
                    if (!(skip_first && issued == 0))
                        gemm103::bulk_load_1d(slots + static_cast<size_t>(d) * kLongChunkBytes,
                                              X + row * p.ldx + e_lo + e0, bytes, &full[d],
                                              j < C ? keep : last);
                    ++issued;
                    if (++d == D) {
                        d = 0;
                        ++round;
                    }
                }
            }
            if (!ok) {
                atomicExch(p.err, 1);
                abort_flag = 1;
            }
            // every copy issued lands before the CTA (and its shared memory) goes
            for (int64_t i = issued > D ? issued - D : 0; i < issued; ++i)
                gemm103::mbar_wait(&full[static_cast<int>(i % D)],
                                   static_cast<uint32_t>((i / D) & 1), p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- compute
        const int t = threadIdx.x;
        const int32_t tail = ends_row ? p.cols - p.bulk_elems : 0;   // < V elements
        int d = 0;
        uint32_t round = 0;
        bool ok = true;
        uint32_t iter = 0;                // rows done by this CTA
        // wait for slot dd's data; a wait that runs out tells every other
        // waiter of the CTA (and the producer) to give up too
        auto take = [&](int dd, uint32_t rr) {
            if (!ok) return;
            ok = wait_abortable(&full[dd], rr & 1u, &abort_flag, p.wait_limit_ns);
            if (!ok) abort_flag = 1;
        };
        // the warp has read slot dd: one arrival, and only when every lane
        // got its data (a slot whose copy never landed is never refilled)
        auto release = [&](int dd) {
            const bool wok = __all_sync(0xffffffffu, ok) != 0;
            if (lane == 0 && wok) gemm103::mbar_arrive(&empty[dd]);
        };
        for (int64_t row = cid; row < p.rows; row += nclusters, ++iter) {
            const InT* __restrict__ xrow = X + row * p.ldx + e_lo;
            OutT* __restrict__ yrow = Y + row * p.ldy + e_lo;
            const int pb = static_cast<int>(iter & 1u);
            // pass 1: (m, s) of this thread's elements, chunk by chunk
            float m = -INFINITY, s = 0.0f;
            for (int32_t c = 0; c < C; ++c) {
                take(d, round);
                const int32_t e0 = c * kChunkElems;
                const int32_t nv = (nb - e0 < kChunkElems ? nb - e0 : kChunkElems) / V;
                const uint8_t* slot = slots + static_cast<size_t>(d) * kLongChunkBytes;
                float x[kLongKV][V];
                #pragma unroll
                for (int k = 0; k < kLongKV; ++k) {
                    const int32_t v = t + k * T;
                    if (v < nv) {
                        unpack16<InT>(
                            *reinterpret_cast<const uint4*>(slot + static_cast<size_t>(v) * 16), x[k]);
                    } else {
                        #pragma unroll
                        for (int e = 0; e < V; ++e) x[k][e] = -INFINITY;
                    }
                }
                release(d);
                float cm = -INFINITY;
                #pragma unroll
                for (int k = 0; k < kLongKV; ++k) {
                    #pragma unroll
                    for (int e = 0; e < V; ++e) cm = fmax_nan(cm, x[k][e]);
                }
                const float mm = fmax_nan(m, cm);
                const float mmz = (mm == -INFINITY) ? 0.0f : mm;
                float add = 0.0f;
                #pragma unroll
                for (int k = 0; k < kLongKV; ++k) {
                    #pragma unroll
                    for (int e = 0; e < V; ++e) add += exp_elem<InT>(x[k][e] - mmz);
                }
                s = (m == -INFINITY ? 0.0f : s * __expf(m - mmz)) + add;
                m = mm;
                if (++d == D) {
                    d = 0;
                    ++round;
                }
            }
            float xt = -INFINITY;
            if (t < tail) {
                xt = to_f(X[row * p.ldx + p.bulk_elems + t]);
                merge(m, s, xt, 1.0f);
            }
            // the CTA's 512 pairs: warp butterflies, then the 16 warps' pairs
            // in warp order (the same bits in every thread)
            warp_merge(m, s);
            if (lane == 0) {
                red_m[pb][warp] = m;
                red_s[pb][warp] = s;
            }
            ok = group_all(kTmaComputeWarps, 0, ok);
            if (!ok && CL == 1) break;
            float M = red_m[pb][0], S = red_s[pb][0];
            #pragma unroll
            for (int w = 1; w < kTmaComputeWarps; ++w) merge(M, S, red_m[pb][w], red_s[pb][w]);
            if (CL > 1) {
                // the cluster's pairs, merged in rank order in every CTA
                if (t == 0) send_pair(M, S, recv_m[pb], recv_s[pb], &xbar[pb], rank, CL);
                if (!wait_peers(&xbar[pb], (iter >> 1) & 1u, &abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    abort_flag = 1;
                }
                M = recv_m[pb][0];
                S = recv_s[pb][0];
                for (int q = 1; q < CL; ++q) merge(M, S, recv_m[pb][q], recv_s[pb][q]);
            }
            const float Mz = (M == -INFINITY) ? 0.0f : M;
            const float inv = 1.0f / S;
            // pass 2: y = e^(x - M) / S, chunk by chunk
            for (int32_t c = 0; c < C; ++c) {
                take(d, round);
                const int32_t e0 = c * kChunkElems;
                const int32_t nv = (nb - e0 < kChunkElems ? nb - e0 : kChunkElems) / V;
                const uint8_t* slot = slots + static_cast<size_t>(d) * kLongChunkBytes;
                float x[kLongKV][V];
                #pragma unroll
                for (int k = 0; k < kLongKV; ++k) {
                    const int32_t v = t + k * T;
                    if (v < nv)
                        unpack16<InT>(
                            *reinterpret_cast<const uint4*>(slot + static_cast<size_t>(v) * 16), x[k]);
                }
                release(d);
                if (ok) {
                    #pragma unroll
                    for (int k = 0; k < kLongKV; ++k) {
                        const int32_t v = t + k * T;
                        if (v < nv) {
                            float o[V];
                            #pragma unroll
                            for (int e = 0; e < V; ++e) o[e] = exp_elem<InT>(x[k][e] - Mz) * inv;
                            store_vec16<InT, OutT>(yrow + e0 + static_cast<int64_t>(v) * V, o);
                        }
                    }
                }
                if (++d == D) {
                    d = 0;
                    ++round;
                }
            }
            if (t < tail && ok)
                Y[row * p.ldy + p.bulk_elems + t] = from_f<OutT>(exp_elem<InT>(xt - Mz) * inv);
        }
        if (!ok) {
            abort_flag = 1;
            atomicExch(p.err, 1);
        }
    }
    // no CTA leaves while a peer may still write to its shared memory
    if (CL > 1) gemm103::cluster_sync_all();
}

template <typename InT, typename OutT>
cudaError_t launch_softmax_long(const TmaSoftmaxParams& p, int grid, size_t smem,
                                cudaStream_t stream) {
    auto kern = softmax_long_kernel<InT, OutT>;
    const int cl = p.cluster;
    if (cl < 1 || cl > kMaxLongCluster || grid % cl != 0) return cudaErrorInvalidValue;
    int clusters_max = 0;                 // clusters of `cl` CTAs resident at once (cl > 1)
    {
        static std::mutex mu;
        static bool raised = false;
        static int resident[kMaxLongCluster + 1] = {};
        std::lock_guard<std::mutex> g(mu);
        if (!raised) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            if (cl > 1) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
            raised = true;
        }
        if (cl > 1 && resident[cl] == 0) {
            cudaLaunchConfig_t q = {};
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = cl;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.gridDim = dim3(grid, 1, 1);
            q.blockDim = dim3(kTmaThreads, 1, 1);
            q.dynamicSmemBytes = smem;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) {
                cudaGetLastError();
                n = 1;
            }
            resident[cl] = n;
        }
        clusters_max = cl > 1 ? resident[cl] : 0;
    }
    if (cl > 1 && grid > cl * clusters_max) grid = cl * clusters_max;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (cl > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename InT, typename OutT, int KV, bool WHOLE>
cudaError_t launch_softmax_tma_kv(const TmaSoftmaxParams& p, int grid, size_t smem,
                                  cudaStream_t stream) {
    auto kern = softmax_tma_kernel<InT, OutT, KV, WHOLE>;
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

template <typename InT, typename OutT, int KV>
cudaError_t launch_softmax_tma_w(const TmaSoftmaxParams& p, int grid, size_t smem,
                                 cudaStream_t stream) {
    return p.whole ? launch_softmax_tma_kv<InT, OutT, KV, true>(p, grid, smem, stream)
                   : launch_softmax_tma_kv<InT, OutT, KV, false>(p, grid, smem, stream);
}

template <typename InT, typename OutT>
cudaError_t launch_softmax_tma(const TmaSoftmaxParams& p, int grid, size_t smem,
                               cudaStream_t stream) {
    if (p.long_rows) return launch_softmax_long<InT, OutT>(p, grid, smem, stream);
    switch (p.kv) {
        case 1: return launch_softmax_tma_w<InT, OutT, 1>(p, grid, smem, stream);
        case 2: return launch_softmax_tma_w<InT, OutT, 2>(p, grid, smem, stream);
        case 4: return launch_softmax_tma_w<InT, OutT, 4>(p, grid, smem, stream);
        case 8: return launch_softmax_tma_w<InT, OutT, 8>(p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace smx
