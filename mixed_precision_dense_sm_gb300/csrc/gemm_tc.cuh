// gemm_tc.cuh -- persistent, warp-specialised tcgen05 GEMM mainloop for sm_103a.
//
// Computes D = op(A) * op(B) over 128 x BN output tiles, K in blocks of 64,
// with FP16/BF16 operands and an FP32 accumulator in tensor memory, then
// applies the epilogue r = alpha * D + beta * C and the output cast.
//
// How it maps the pages' GEMM structure onto GB300:
//  * Tiling (DeepGEMM page, section 3.1; CATLASS page, section 2.1): one CTA
//    owns a 128 x BN output tile and walks K; the accumulator lives in TMEM
//    (128 lanes x BN FP32 columns) instead of per-thread registers.
//  * Multi-stage pipelining (DeepGEMM page, sections 4.1 and 5.1-5.4; SGEMM
//    page, section 3.4): a ring of `stages` shared-memory slots.  Warp 0
//    (producer) waits for a free slot, arms its "full" mbarrier with the byte
//    count and issues TMA tile loads; warp 1 (MMA issuer) waits on "full",
//    issues 4 tcgen05.mma (K = 16 each) and commits to the slot's "empty"
//    mbarrier, which frees it once the tensor core has read it.  The
//    prologue/steady-state/epilogue structure of the pages falls out of the
//    ring: the producer runs ahead by up to `stages` slots.
//  * Bank conflicts and padding (SGEMM page, section 3.3; DeepGEMM page,
//    sections 4.2-4.3): TMA writes every tile with the 128-byte swizzle that
//    the tensor core's shared-memory descriptor expects; no padding.
//  * Ragged edges (DeepGEMM page, section 3.4): TMA fills elements outside
//    the matrix with zeros, so a K tail contributes nothing; rows/columns past
//    M/N are computed but never stored.
//  * FP32 accumulation (DeepGEMM page, section 6.2): kind::f16 with an F32 D.
//  * Grid fill (SGEMM page, section 4.3): the grid is at most one CTA per SM;
//    each CTA walks a sequence of work segments (below).  Warps 2-5 drain the
//    other TMEM accumulator buffer while the next segment's MMAs run.
//
// Work segments.  A segment is (tile, first k-block, last k-block).
//  * Data-parallel mode: CTA g takes tiles g, g + G, g + 2G, ... whole.
//  * Stream-K mode (fewer tiles than SMs): the (tile, k-block) space is cut
//    into G contiguous ranges of L k-blocks, one per CTA.  A segment that
//    covers a whole tile is stored directly; a partial one writes its raw
//    FP32 sums to a workspace slot, and a separate fixup kernel adds a tile's
//    slots in increasing CTA order (deterministic) and applies the epilogue.
//
// CTA pairs.  For large problems two CTAs of a cluster share one 256 x BN
// tile through tcgen05's cta_group::2 form (see gemm_tc_kernel below): each SM
// reads half of B, which halves the B traffic and shared-memory reads per SM.
//
// Swap-A/B.  For small M the host passes A' = op(B)^T and B' = op(A)^T, so the
// kernel computes D' = C^T and the epilogue stores D'(i, j) at C[j][i]
// (c_rs = 1, c_cs = ldc).  The kernel itself only sees "rows" M' and "columns"
// N' and the two strides.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gemm103 {

constexpr int kBlockM = 128;      // tcgen05 M (cta_group::1)
constexpr int kBlockK = 64;       // 64 16-bit elements = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K per tcgen05.mma kind::f16
constexpr int kThreads = 192;     // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiWarps = 4;
constexpr uint32_t kATileBytes = kBlockM * kBlockK * 2;   // 16 KB
constexpr uint32_t kChunkBytes = 64 * kBlockK * 2;        // one 64 x 64 MN-major box, 8 KB

enum : int { kErrTimeoutProducer = 1, kErrTimeoutMma = 2, kErrTimeoutEpilogue = 3 };

struct TcParams {
    int32_t M, N;               // logical rows (M') / columns (N') of D
    int32_t k_blocks;           // ceil(K / 64)
    int32_t tiles_m, tiles_n, num_tiles;
    int32_t group_m;            // raster: tiles walk down group_m tile-rows at a time
    int32_t stages;
    int32_t a_mn_major, b_mn_major;
    uint32_t idesc;
    // scheduling
    int32_t stream_k;           // 0: data-parallel, 1: stream-K
    int32_t sk_len;             // L: k-blocks per CTA in stream-K mode
    int32_t sk_max_seg;         // workspace slots per CTA
    // epilogue
    float alpha, beta;
    void* C;
    int64_t c_rs, c_cs;         // D'(i, j) -> C[i * c_rs + j * c_cs]
    int32_t c_vector;           // c_cs == 1 and rows 16-byte aligned
    float* partials;            // stream-K slots: [G * sk_max_seg][128][BN] FP32
    int* err;                   // device-visible error word (0 = ok)
    uint64_t ab_policy;         // unused placeholder for cache-policy selection
};

struct Segment {
    int32_t tile, kb0, kb1;
    int32_t slot;               // -1: whole tile (direct store), else workspace slot
};

// Iterates the segments of CTA `g` in order; identical in every role.
struct SegmentIter {
    int32_t g, G;
    int32_t pos, end;           // stream-K: linear (tile, k-block) positions
    int32_t next_tile;          // data-parallel
    __device__ SegmentIter(const TcParams& p, int32_t g_, int32_t G_) : g(g_), G(G_) {
        if (p.stream_k) {
            int64_t total = static_cast<int64_t>(p.num_tiles) * p.k_blocks;
            int64_t b = static_cast<int64_t>(g) * p.sk_len;
            int64_t e = b + p.sk_len;
            pos = static_cast<int32_t>(b < total ? b : total);
            end = static_cast<int32_t>(e < total ? e : total);
        } else {
            pos = end = 0;
        }
        next_tile = g;
    }
    __device__ bool next(const TcParams& p, Segment& s) {
        if (!p.stream_k) {
            if (next_tile >= p.num_tiles) return false;
            s.tile = next_tile;
            s.kb0 = 0;
            s.kb1 = p.k_blocks;
            s.slot = -1;
            next_tile += G;
            return true;
        }
        if (pos >= end) return false;
        const int32_t KB = p.k_blocks;
        s.tile = pos / KB;
        s.kb0 = pos - s.tile * KB;
        int32_t take = KB - s.kb0;
        if (take > end - pos) take = end - pos;
        s.kb1 = s.kb0 + take;
        pos += take;
        if (s.kb0 == 0 && s.kb1 == KB) {
            s.slot = -1;
        } else {
            const int32_t first_tile = static_cast<int32_t>(
                (static_cast<int64_t>(g) * p.sk_len) / KB);
            s.slot = g * p.sk_max_seg + (s.tile - first_tile);
        }
        return true;
    }
};

__device__ __forceinline__ void tile_coords(const TcParams& p, int32_t tile, int32_t& tm,
                                            int32_t& tn) {
    const int32_t per_group = p.group_m * p.tiles_n;
    const int32_t group = tile / per_group;
    const int32_t first_m = group * p.group_m;
    int32_t gsz = p.tiles_m - first_m;
    if (gsz > p.group_m) gsz = p.group_m;
    const int32_t local = tile - group * per_group;
    tm = first_m + local % gsz;
    tn = local / gsz;
}

__device__ __forceinline__ void record_error(const TcParams& p, int code, volatile int* abort_flag) {
    *abort_flag = 1;
    if (p.err) atomicCAS(p.err, 0, code);
}

// Bounded wait that also gives up early once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
        }
    }
}

template <typename OutT>
__device__ __forceinline__ OutT cvt_out(float v);
template <>
__device__ __forceinline__ float cvt_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half cvt_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

template <typename OutT>
__device__ __forceinline__ float load_out(const OutT* p);
template <>
__device__ __forceinline__ float load_out<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_out<__half>(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float load_out<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

// Store 32 consecutive values v[0..31] of one C row at `dst` (16-byte aligned,
// all in range), with optional beta * C read.
template <typename OutT>
__device__ __forceinline__ void store_row32_vec(OutT* dst, const float (&v)[32], float beta) {
    constexpr int kPer16 = 16 / sizeof(OutT);      // elements per 16-byte vector
    #pragma unroll
    for (int q = 0; q < 32 / kPer16; ++q) {
        float x[kPer16];
        #pragma unroll
        for (int e = 0; e < kPer16; ++e) x[e] = v[q * kPer16 + e];
        if (beta != 0.0f) {
            uint4 old = *reinterpret_cast<const uint4*>(dst + q * kPer16);
            const OutT* o = reinterpret_cast<const OutT*>(&old);
            #pragma unroll
            for (int e = 0; e < kPer16; ++e) x[e] = fmaf(beta, load_out<OutT>(o + e), x[e]);
        }
        uint4 pack;
        OutT* pk = reinterpret_cast<OutT*>(&pack);
        #pragma unroll
        for (int e = 0; e < kPer16; ++e) pk[e] = cvt_out<OutT>(x[e]);
        *reinterpret_cast<uint4*>(dst + q * kPer16) = pack;
    }
}

// Wait on a barrier that receives plain arrivals from the peer CTA (the odd
// CTA's epilogue releasing the accumulator): cluster-scope acquire, so the
// peer's TMEM reads are ordered before the MMAs that overwrite them.  Barriers
// completed by TMA transactions or tcgen05.commit are waited on at CTA scope.
template <int CG>
__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if constexpr (CG == 1) {
        return wait_or_abort(bar, parity, abort_flag);
    } else {
        const uint32_t a = smem_addr(bar);
        if (mbar_try_wait_cluster(a, parity)) return true;
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 1;; ++i) {
            if (mbar_try_wait_cluster(a, parity)) return true;
            if ((i & 63u) == 0) {
                if (*abort_flag) return false;
                if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
            }
        }
    }
}

// CG = 1: one CTA per 128 x BN tile (tcgen05 cta_group::1, M = 128).
// CG = 2: a cluster of two CTAs per 256 x BN tile (cta_group::2, M = 256).
//   Each CTA loads its own 128 rows of A and BN/2 rows of B; both CTAs'
//   loads count their bytes on the even CTA's "full" barrier, which the even
//   CTA alone arms with the pair's total (no cluster-scope arrive, and so no
//   memory barrier, on the per-k-block path); the even CTA
//   alone issues the MMAs, whose commits arrive on the "empty" / "acc_full"
//   barriers of both CTAs; both CTAs drain their own TMEM half (128 rows x BN)
//   and release the accumulator on the even CTA's "acc_empty" barrier.
template <int CG, int BN, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ TcParams p) {
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
    static_assert(CG == 1 || (CG == 2 && BN >= 128), "CG");
    constexpr int BM = kBlockM * CG;                      // rows per (pair) tile
    constexpr uint32_t kBRows = BN / CG;                  // B rows this CTA loads
    constexpr uint32_t kBTileBytes = kBRows * kBlockK * 2;
    constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
    constexpr uint32_t kTmemCols = 2 * BN;               // double-buffered accumulator

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const int32_t unit = blockIdx.x / CG;                 // CTA (pair) index
    const int32_t units = gridDim.x / CG;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);                      // the even CTA's producer arms it
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps * CG);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (CG == 1) {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        } else {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();            // peer barriers initialised
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0;                   // number of slot armings so far
            SegmentIter it(p, unit, units);
            Segment sg;
            bool ok = true;
            while (ok && it.next(p, sg)) {
                int32_t tm, tn;
                tile_coords(p, sg.tile, tm, tn);
                // Parts of a CTA's A / B tiles that lie wholly outside the
                // matrix only feed outputs that are never stored: not loaded.
                // tile_bytes(r) is what CTA r of the pair loads per k-block.
                auto a_parts = [&](int32_t m_first) {
                    if (!p.a_mn_major) return (m_first < p.M) ? 1 : 0;
                    int n = 0;
                    for (int c = 0; c < kBlockM / 64; ++c) n += (m_first + 64 * c < p.M);
                    return n;
                };
                auto b_parts = [&](int32_t n_first) {
                    if (!p.b_mn_major) return (n_first < p.N) ? 1 : 0;
                    int n = 0;
                    for (int c = 0; c < static_cast<int>(kBRows) / 64; ++c) n += (n_first + 64 * c < p.N);
                    return n;
                };
                auto tile_bytes = [&](uint32_t r) {
                    const int32_t mf = tm * BM + static_cast<int32_t>(r) * kBlockM;
                    const int32_t nf = tn * BN + static_cast<int32_t>(r * kBRows);
                    return static_cast<uint32_t>(a_parts(mf)) *
                               (p.a_mn_major ? kChunkBytes : kATileBytes) +
                           static_cast<uint32_t>(b_parts(nf)) *
                               (p.b_mn_major ? kChunkBytes : kBTileBytes);
                };
                const int32_t m0 = tm * BM + static_cast<int32_t>(rank) * kBlockM;
                const int32_t n0 = tn * BN + static_cast<int32_t>(rank * kBRows);
                const int na = a_parts(m0), nb = b_parts(n0);
                // The even CTA's "full" barrier counts the bytes of both CTAs;
                // the odd CTA's loads may land before it is armed (the
                // transaction count may go transiently negative).
                const uint32_t bytes = (CG == 1) ? tile_bytes(0)
                                                 : (rank == 0 ? tile_bytes(0) + tile_bytes(1) : 0u);
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!wait_or_abort(&empty[stage], phase ^ 1u, &abort_flag)) {
                        record_error(p, kErrTimeoutProducer, &abort_flag);
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * kStageBytes;
                    uint8_t* sb = sa + kATileBytes;
                    const int32_t k0 = kb * kBlockK;
                    if constexpr (CG == 1) {
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        if (p.a_mn_major) {
                            for (int c = 0; c < na; ++c)
                                tma_load_2d(sa + c * kChunkBytes, &tmA, &full[stage], m0 + 64 * c,
                                            k0, policy);
                        } else if (na) {
                            tma_load_2d(sa, &tmA, &full[stage], k0, m0, policy);
                        }
                        if (p.b_mn_major) {
                            for (int c = 0; c < nb; ++c)
                                tma_load_2d(sb + c * kChunkBytes, &tmB, &full[stage], n0 + 64 * c,
                                            k0, policy);
                        } else if (nb) {
                            tma_load_2d(sb, &tmB, &full[stage], k0, n0, policy);
                        }
                    } else {
                        const uint32_t fb = map_to_rank(smem_addr(&full[stage]), 0);
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], bytes);
                        if (p.a_mn_major) {
                            for (int c = 0; c < na; ++c)
                                tma_load_2d_pair(sa + c * kChunkBytes, &tmA, fb, m0 + 64 * c, k0,
                                                 policy);
                        } else if (na) {
                            tma_load_2d_pair(sa, &tmA, fb, k0, m0, policy);
                        }
                        if (p.b_mn_major) {
                            for (int c = 0; c < nb; ++c)
                                tma_load_2d_pair(sb + c * kChunkBytes, &tmB, fb, n0 + 64 * c, k0,
                                                 policy);
                        } else if (nb) {
                            tma_load_2d_pair(sb, &tmB, fb, k0, n0, policy);
                        }
                    }
                    ++armed;
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Wind-down: wait (bounded) until every TMA load issued into this
            // CTA pair has landed.  The even CTA's "full" barriers count the
            // bytes of both CTAs, so only the even CTA waits; the odd CTA is
            // held by the cluster barrier before exit until then.
            if (rank == 0) {
                for (int s = 0; s < S; ++s) {
                    if (armed <= static_cast<uint32_t>(s)) break;
                    const uint32_t last = ((armed - 1 - s) / S) * S + s;   // last arming of slot s
                    if (!mbar_wait(&full[s], (last / S) & 1u)) {
                        record_error(p, kErrTimeoutProducer, &abort_flag);
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0, acc_i = 0;
            SegmentIter it(p, unit, units);
            Segment sg;
            bool ok = true;
            const uint32_t a_lbo = p.a_mn_major ? kChunkBytes : 16u;
            const uint32_t b_lbo = p.b_mn_major ? kChunkBytes : 16u;
            const uint32_t a_kstep = p.a_mn_major ? kUmmaK * 128u : kUmmaK * 2u;
            const uint32_t b_kstep = p.b_mn_major ? kUmmaK * 128u : kUmmaK * 2u;
            const uint32_t smem_base = smem_addr(smem);
            while (ok && it.next(p, sg)) {
                const uint32_t buf = acc_i & 1u;
                if (!wait_role<CG>(&acc_empty[buf], ((acc_i >> 1) & 1u) ^ 1u, &abort_flag)) {
                    record_error(p, kErrTimeoutMma, &abort_flag);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!wait_or_abort(&full[stage], phase, &abort_flag)) {
                        record_error(p, kErrTimeoutMma, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = smem_base + stage * kStageBytes;
                    const uint32_t sb = sa + kATileBytes;
                    #pragma unroll
                    for (int kk = 0; kk < kBlockK / kUmmaK; ++kk) {
                        const uint64_t ad = smem_desc_sw128(sa + kk * a_kstep, a_lbo, 1024);
                        const uint64_t bd = smem_desc_sw128(sb + kk * b_kstep, b_lbo, 1024);
                        const uint32_t acc = (kb > sg.kb0 || kk > 0) ? 1u : 0u;
                        if constexpr (CG == 1) tc_mma_f16(d_tmem, ad, bd, p.idesc, acc);
                        else tc_mma_f16_pair(d_tmem, ad, bd, p.idesc, acc);
                    }
                    if constexpr (CG == 1) tc_commit(&empty[stage]);
                    else tc_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (CG == 1) tc_commit(&acc_full[buf]);
                else tc_commit_pair_multicast(&acc_full[buf], 0x3);
                ++acc_i;
            }
            // Wind-down: every MMA issued has completed before TMEM is freed.
            if constexpr (CG == 1) tc_commit(drain);
            else tc_commit_pair(drain);
            if (!mbar_wait(drain, 0)) record_error(p, kErrTimeoutMma, &abort_flag);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int quarter = warp & 3;                   // TMEM lanes 32*quarter..+31
        const int row_in_cta = quarter * 32 + lane;
        const int row_in_tile = static_cast<int>(rank) * kBlockM + row_in_cta;
        OutT* C = reinterpret_cast<OutT*>(p.C);
        uint32_t acc_i = 0;
        SegmentIter it(p, unit, units);
        Segment sg;
        while (it.next(p, sg)) {
            const uint32_t buf = acc_i & 1u;
            if (!wait_or_abort(&acc_full[buf], (acc_i >> 1) & 1u, &abort_flag)) {
                record_error(p, kErrTimeoutEpilogue, &abort_flag);
                break;
            }
            tc_fence_after_sync();
            int32_t tm, tn;
            tile_coords(p, sg.tile, tm, tn);
            const int32_t row = tm * BM + row_in_tile;              // D' row
            const int32_t col0 = tn * BN;                           // D' first column
            const uint32_t t_row = tmem_base + buf * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            #pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                __syncwarp();                      // tcgen05.ld is warp-collective
                tmem_ld_32x32b_x32(t_row + ch * 32, r);
                tmem_ld_wait();
                float v[32];
                #pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                const int32_t c0 = col0 + ch * 32;
                if (sg.slot >= 0) {
                    // stream-K partial: raw FP32 sums, [slot][row_in_tile][BN]
                    float4* dst = reinterpret_cast<float4*>(
                        p.partials + (static_cast<int64_t>(sg.slot) * BM + row_in_tile) * BN +
                        ch * 32);
                    #pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    continue;
                }
                #pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= p.alpha;
                if (row >= p.M) continue;
                if (p.c_vector && c0 + 32 <= p.N) {
                    store_row32_vec<OutT>(C + static_cast<int64_t>(row) * p.c_rs + c0, v, p.beta);
                } else {
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int32_t col = c0 + j;
                        if (col < p.N) {
                            OutT* dst = C + static_cast<int64_t>(row) * p.c_rs +
                                        static_cast<int64_t>(col) * p.c_cs;
                            float x = v[j];
                            if (p.beta != 0.0f) x = fmaf(p.beta, load_out<OutT>(dst), x);
                            *dst = cvt_out<OutT>(x);
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(&acc_empty[buf]);
                else mbar_arrive_cluster(map_to_rank(smem_addr(&acc_empty[buf]), 0));
            }
            ++acc_i;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();            // peer done with our smem / TMEM
    tc_fence_after_sync();
    if (warp == 1) {
        if constexpr (CG == 1) tmem_dealloc(tmem_base, kTmemCols);
        else tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// Stream-K fixup: for every tile that was split across CTAs, add its partial
// slots in increasing CTA order, then apply alpha/beta and the output cast.
// One thread per (tile, row, 4 columns).
template <int BM, int BN, typename OutT>
__global__ void __launch_bounds__(256)
    streamk_fixup_kernel(const __grid_constant__ TcParams p) {
    const int64_t per_tile = static_cast<int64_t>(BM) * (BN / 4);
    const int64_t total = per_tile * p.num_tiles;
    OutT* C = reinterpret_cast<OutT*>(p.C);
    const int32_t KB = p.k_blocks, L = p.sk_len;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t tile = static_cast<int32_t>(idx / per_tile);
        const int32_t rem = static_cast<int32_t>(idx - static_cast<int64_t>(tile) * per_tile);
        const int32_t r = rem / (BN / 4);
        const int32_t c4 = (rem - r * (BN / 4)) * 4;
        const int32_t g_first = static_cast<int32_t>((static_cast<int64_t>(tile) * KB) / L);
        const int32_t g_last = static_cast<int32_t>((static_cast<int64_t>(tile + 1) * KB - 1) / L);
        if (g_first == g_last) continue;           // stored whole by one CTA
        int32_t tm, tn;
        tile_coords(p, tile, tm, tn);
        const int32_t row = tm * BM + r;
        if (row >= p.M) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t g = g_first; g <= g_last; ++g) {
            const int32_t first_tile = static_cast<int32_t>((static_cast<int64_t>(g) * L) / KB);
            const int64_t slot = static_cast<int64_t>(g) * p.sk_max_seg + (tile - first_tile);
            const float4 v = *reinterpret_cast<const float4*>(
                p.partials + (slot * BM + r) * BN + c4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int32_t col = tn * BN + c4 + e;
            if (col >= p.N) break;
            OutT* dst = C + static_cast<int64_t>(row) * p.c_rs + static_cast<int64_t>(col) * p.c_cs;
            float x = p.alpha * vals[e];
            if (p.beta != 0.0f) x = fmaf(p.beta, load_out<OutT>(dst), x);
            *dst = cvt_out<OutT>(x);
        }
    }
}

}  // namespace gemm103
