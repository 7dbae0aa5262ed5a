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
//    covers a whole tile is stored directly; for a split tile the last CTA to
//    finish its part adds every contribution in increasing CTA order
//    (deterministic) -- its own from registers, the others' from workspace
//    slots -- and applies the epilogue.
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

#include "epilogue_ops.cuh"
#include "ptx.cuh"

namespace gemm103 {

constexpr int kBlockM = 128;      // tcgen05 M (cta_group::1)
// A K chunk is one 128-byte swizzle row of K per operand row: 64 16-bit
// elements (kind::f16, K = 16 per MMA) or 32 FP32 elements used as TF32
// (kind::tf32, K = 8 per MMA); either way 4 MMAs per chunk.  A pipeline stage
// holds KC chunks (1 or 2, a template parameter of the kernel).  The TMA unit completes about one box per
// 160 ns per SM whatever its size (8-32 KB), so two chunks per box halve the
// TMA operations per MMA: K-major operands are then read through a 3-D map
// (chunk of K, rows, chunk index) whose box spans both chunks, and MN-major
// boxes span kc * 64 rows of K.
template <int ES> struct Elem {
    static constexpr int kChunkK = 128 / ES;        // K elements per chunk
    static constexpr int kUmmaK = 32 / ES;          // K per tcgen05.mma
    static constexpr int kMNChunk = 128 / ES;       // M/N elements per MN-major box row
};
constexpr int kMaxKc = 2;
constexpr int kThreads = 320;     // warp 0 producer, warp 1 MMA, warps 2-9 epilogue
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter, splitting the columns
constexpr int kFinBatch = 2;      // stream-K finisher: partial slots loaded per batch
// Staging for C stores by TMA: 32 KB after the pipeline stages, two boxes of
// 128 rows x 128 bytes (128-byte swizzle), each 1024-byte aligned.
constexpr uint32_t kCStageBytes = 32768;
constexpr uint32_t kCBoxBytes = 16384;
constexpr uint32_t kATileBytes = kBlockM * 128;          // 16 KB: 128 rows of 128 bytes

enum : int { kErrTimeoutProducer = 1, kErrTimeoutMma = 2, kErrTimeoutEpilogue = 3 };

struct TcParams {
    int32_t M, N;               // logical rows (M') / columns (N') of D
    int32_t k_blocks;           // ceil(K / (KC * chunk)): pipeline stages of K per tile
    int32_t tiles_m, tiles_n, num_tiles;
    int32_t group;              // raster: tiles go in groups of `group` tile-rows (raster_n = 0)
    int32_t raster_n;           // or of `group` tile-columns (raster_n = 1)
    int32_t serpentine;         // data-parallel: odd tiles of a CTA walk K backwards
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
    int32_t c_tma;              // C stored through shared memory by TMA (tmC, plain epilogue)
    float* partials;            // stream-K slots: [G * sk_max_seg][BN / 4][BM] float4 (FP32)
    int* tile_counters;         // stream-K: per split tile and CTA of the pair, contributors
                                // written (self-resetting)
    int* err;                   // device-visible error word (0 = ok)
    int32_t a_policy;           // L2 policy of A's loads: kL2EvictLast / kL2EvictFirst / kL2EvictNormal
    int32_t b_policy;
    uint64_t wait_limit_ns;     // bound on every in-kernel wait
    uint32_t debug_flags;       // test hook (kDebugSkipFirstLoad), 0 in normal use
    // fused epilogue: r = act(alpha * acc + beta * C + bias)
    const void* bias;           // N elements or nullptr
    int32_t bias_dtype;         // 0 F16, 1 BF16, 2 F32
    int32_t bias_on_rows;       // 1: bias indexed by D' row (swapped problem), 0: by column
    int32_t act;                // 0 none, 1 ReLU, 2 GELU (erf), 3 SiLU
    // implicit-GEMM convolution (conv != 0): A is an im2col map over the
    // NHWC input; chunk j of K (64 channels, 16-bit inputs) is filter tap
    // j / cblocks with channels from (j % cblocks) * 64, chunks past the last
    // tap read channels past C (zeros); D row m is the output pixel (n, p, q)
    // of m = (n*P + p)*Q + q.  B is the KRSC filter: with one chunk per stage
    // a 3-D map (C, R*S, K) loaded by (channel, tap); with two (C a multiple
    // of 64) the filter as a K-major K x (R*S*C) matrix in chunks
    int32_t conv;
    int32_t conv_cblocks;       // ceil(C / 64)
    int32_t conv_taps;          // R * S
    int32_t conv_S;             // filter width
    int32_t conv_P, conv_Q;     // output height and width
    int32_t conv_stride_h, conv_stride_w, conv_pad_h, conv_pad_w, conv_dil_h, conv_dil_w;
    // conv_tiled (stride 1, single-CTA tiles): a tile is conv_rows whole
    // output rows of one image (tile row tm: image tm / conv_tpi, first row
    // (tm % conv_tpi) * conv_rows), and A is loaded per filter tap by a tiled
    // 4-D map over X (C, W, H, N) -- a box of 64 channels x Q x conv_rows
    // pixels at the tap's shifted window, zeros outside the image -- instead
    // of the im2col map; conv_a_bytes = one such box
    int32_t conv_tiled;
    int32_t conv_rows;
    int32_t conv_tpi;
    uint32_t conv_a_bytes;
    // conv_tiled == 2 (halo units): a tile's output pixel (p', q) is A row
    // p' * conv_pitch + q (conv_pitch = Q rounded up to 8; 1: conv_pitch = Q).
    // Pipeline step kb is filter column s = kb / conv_cblocks and channel
    // block kb % conv_cblocks: one tiled box of conv_rows + (R - 1) dil_h
    // image rows x conv_pitch pixels (the halo, conv_a_bytes) and the R
    // filter taps of that column (R boxes of BN rows); tap r's A is the box
    // from row r * dil_h * conv_pitch on.  The stage geometry is set at run
    // time: halo_a_region bytes of A, then R * BN * 128 of B, stage_bytes in all
    int32_t conv_pitch;
    int32_t conv_R;
    uint32_t halo_a_region;
    uint32_t halo_stage_bytes;
    // LayerNorm after the linear layer (kernels instantiated with EPI ==
    // kEpiLayerNorm): h = round_C(alpha * acc + beta * C + bias) per element;
    // ln_fused (the whole row in one tile): each row is normalised in the
    // epilogue, y = (h - mean) / sqrt(var + eps) * gamma + shift, and only y is
    // stored; otherwise h is stored and (sum, M2) of the tile's columns of
    // each row go to ln_stats[row * tiles_n + tile column] for a row pass
    const void* ln_gamma;       // N elements or nullptr (1)
    const void* ln_shift;       // N elements or nullptr (0)
    int32_t ln_dtype;           // 0 F16, 1 BF16, 2 F32
    int32_t ln_fused;
    float ln_eps;
    float2* ln_stats;
};

enum : int { kL2EvictLast = 0, kL2EvictFirst = 1, kL2EvictNormal = 2 };

__device__ __forceinline__ uint64_t l2_policy(int32_t which) {
    return which == kL2EvictFirst ? l2_policy_evict_first()
           : which == kL2EvictNormal ? l2_policy_evict_normal() : l2_policy_evict_last();
}

// Test hook: CTA 0's producer arms its first pipeline slot but issues no load
// into it, so the MMA's bounded wait on that slot runs out.
constexpr uint32_t kDebugSkipFirstLoad = 1u;

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

// Tile `tile` of the raster: groups of p.group tile-rows, each visited column
// by column (every column, the group's rows together), or -- raster_n --
// groups of p.group tile-columns visited row by row.  Consecutive tiles, which
// run in the same wave, share the group's strips of one operand.
__device__ __forceinline__ void tile_coords(const TcParams& p, int32_t tile, int32_t& tm,
                                            int32_t& tn) {
    const int32_t along = p.raster_n ? p.tiles_n : p.tiles_m;    // the grouped dimension
    const int32_t across = p.raster_n ? p.tiles_m : p.tiles_n;
    const int32_t per_group = p.group * across;
    const int32_t group = tile / per_group;
    const int32_t first = group * p.group;
    int32_t gsz = along - first;
    if (gsz > p.group) gsz = p.group;
    const int32_t local = tile - group * per_group;
    const int32_t g_idx = first + local % gsz;
    const int32_t a_idx = local / gsz;
    tm = p.raster_n ? a_idx : g_idx;
    tn = p.raster_n ? g_idx : a_idx;
}

__device__ __forceinline__ void record_error(const TcParams& p, int code, volatile int* abort_flag) {
    *abort_flag = 1;
    if (p.err) atomicCAS(p.err, 0, code);
}

// Bounded wait that also gives up early once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, uint64_t limit_ns) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
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

// Wait on a barrier that receives plain arrivals from the peer CTA (the odd
// CTA's epilogue releasing the accumulator): cluster-scope acquire, so the
// peer's TMEM reads are ordered before the MMAs that overwrite them.  Barriers
// completed by TMA transactions or tcgen05.commit are waited on at CTA scope.
template <int CG>
__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
    if constexpr (CG == 1) {
        return wait_or_abort(bar, parity, abort_flag, limit_ns);
    } else {
        const uint32_t a = smem_addr(bar);
        if (mbar_try_wait_cluster(a, parity)) return true;
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 1;; ++i) {
            if (mbar_try_wait_cluster(a, parity)) return true;
            if ((i & 63u) == 0) {
                if (*abort_flag) return false;
                if (global_timer_ns() - t0 > limit_ns) return false;
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
__device__ __forceinline__ float load_bias(const TcParams& p, int64_t idx) {
    return load_bias_elem(p.bias, p.bias_dtype, idx);
}

// Elements c0..c0+31 of a per-column vector (bias, gamma, shift) of type
// 0 = F16, 1 = BF16, 2 = F32; zeros past column N.
__device__ __forceinline__ void load_col_vec32(const void* vec, int32_t dtype, int32_t c0,
                                               int32_t N, float (&b)[32]) {
    const int esize = dtype == 2 ? 4 : 2;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(vec) + static_cast<uintptr_t>(c0) * esize;
    if (c0 + 32 <= N && (addr & 15u) == 0) {
        // 16-byte loads (every thread of the warp reads the same columns: one
        // L1 line serves the warp)
        const uint4* src = reinterpret_cast<const uint4*>(addr);
        if (dtype == 2) {
            #pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 t = __ldg(src + q);
                b[4 * q] = __uint_as_float(t.x);
                b[4 * q + 1] = __uint_as_float(t.y);
                b[4 * q + 2] = __uint_as_float(t.z);
                b[4 * q + 3] = __uint_as_float(t.w);
            }
        } else {
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 t = __ldg(src + q);
                const uint32_t w[4] = {t.x, t.y, t.z, t.w};
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t lo = static_cast<uint16_t>(w[e] & 0xFFFFu);
                    const uint16_t hi = static_cast<uint16_t>(w[e] >> 16);
                    if (dtype == 1) {
                        b[8 * q + 2 * e] = __bfloat162float(__ushort_as_bfloat16(lo));
                        b[8 * q + 2 * e + 1] = __bfloat162float(__ushort_as_bfloat16(hi));
                    } else {
                        b[8 * q + 2 * e] = __half2float(__ushort_as_half(lo));
                        b[8 * q + 2 * e + 1] = __half2float(__ushort_as_half(hi));
                    }
                }
            }
        }
    } else {
        #pragma unroll
        for (int j = 0; j < 32; ++j) b[j] = (c0 + j < N) ? load_bias_elem(vec, dtype, c0 + j) : 0.0f;
    }
}

// Adds the bias and applies the activation to one row's 32 values at D'
// columns c0..c0+31 (in place); the beta * C term is already in v.
__device__ __forceinline__ void bias_act(const TcParams& p, int32_t row, int32_t c0,
                                         float (&v)[32]) {
    if (p.bias != nullptr) {
        if (p.bias_on_rows) {
            const float b = load_bias(p, row);
            #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += b;
        } else {
            float b[32];
            load_col_vec32(p.bias, p.bias_dtype, c0, p.N, b);
            #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += b[j];
        }
    }
    act32(p.act, v);
}

// act(alpha * v + beta * C + bias) in place for one row of 32 columns at D'
// column c0, without the store (C is read only for columns < N; rows >= M,
// which are never stored, are left as they are).
template <typename OutT>
__device__ __forceinline__ void epilogue_values(const TcParams& p, int32_t row, int32_t c0,
                                                float (&v)[32]) {
    if (p.alpha != 1.0f) {
        #pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= p.alpha;
    }
    if (row >= p.M) return;                 // never stored
    if (p.beta != 0.0f) {
        const OutT* src = reinterpret_cast<const OutT*>(p.C) + static_cast<int64_t>(row) * p.c_rs;
        if (p.c_vector && c0 + 32 <= p.N) {
            constexpr int kPer16 = 16 / sizeof(OutT);
            uint4 raw[32 / kPer16];
            #pragma unroll
            for (int q = 0; q < 32 / kPer16; ++q)
                raw[q] = *reinterpret_cast<const uint4*>(src + c0 + q * kPer16);
            #pragma unroll
            for (int q = 0; q < 32 / kPer16; ++q) {
                const OutT* o = reinterpret_cast<const OutT*>(&raw[q]);
                #pragma unroll
                for (int e = 0; e < kPer16; ++e)
                    v[q * kPer16 + e] = fmaf(p.beta, load_out<OutT>(o + e), v[q * kPer16 + e]);
            }
        } else {
            #pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < p.N)
                    v[j] = fmaf(p.beta, load_out<OutT>(src + static_cast<int64_t>(c0 + j) * p.c_cs),
                                v[j]);
        }
    }
    bias_act(p, row, c0, v);
}

// Writes v[0..31], cast to the output type, to row r of a staging box whose
// rows are 128 bytes with the 128-byte swizzle (16-byte unit u of row r sits
// at unit u ^ (r % 8)), from 16-byte unit u0 of the row on.  Eight
// consecutive rows write eight different bank groups.
template <typename OutT>
__device__ __forceinline__ void stage_row32(uint8_t* box, int r, int u0, const float (&v)[32]) {
    constexpr int kPer16 = 16 / sizeof(OutT);
    uint8_t* base = box + r * 128;
    #pragma unroll
    for (int q = 0; q < 32 / kPer16; ++q) {
        uint4 pack;
        OutT* pk = reinterpret_cast<OutT*>(&pack);
        #pragma unroll
        for (int e = 0; e < kPer16; ++e) pk[e] = cvt_out<OutT>(v[q * kPer16 + e]);
        *reinterpret_cast<uint4*>(base + (((u0 + q) ^ (r & 7)) << 4)) = pack;
    }
}

// Stores v[0..31] (final values), cast to the output type, to C row `row`
// at D' columns c0..c0+31: 16-byte vector stores when the chunk is whole and
// C's rows are aligned, element stores (columns < N) otherwise; rows >= M
// are not stored.
template <typename OutT>
__device__ __forceinline__ void store_row32(const TcParams& p, int32_t row, int32_t c0,
                                            const float (&v)[32]) {
    if (row >= p.M) return;
    OutT* base = reinterpret_cast<OutT*>(p.C) + static_cast<int64_t>(row) * p.c_rs;
    if (p.c_vector && c0 + 32 <= p.N) {
        constexpr int kPer16 = 16 / sizeof(OutT);
        #pragma unroll
        for (int q = 0; q < 32 / kPer16; ++q) {
            uint4 pack;
            OutT* pk = reinterpret_cast<OutT*>(&pack);
            #pragma unroll
            for (int e = 0; e < kPer16; ++e) pk[e] = cvt_out<OutT>(v[q * kPer16 + e]);
            *reinterpret_cast<uint4*>(base + c0 + q * kPer16) = pack;
        }
    } else {
        #pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j < p.N) base[static_cast<int64_t>(c0 + j) * p.c_cs] = cvt_out<OutT>(v[j]);
    }
}

// Spin (bounded) until the global counter reaches `target`.
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, volatile int* abort_flag,
                                             uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((i & 63u) == 63u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
        }
        __nanosleep(32);
    }
}

// Named barrier 1 among the four epilogue warps.
__device__ __forceinline__ void epilogue_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// All four epilogue warps agree on `ok` (logical AND), so that after a
// bounded wait either every epilogue warp carries on or every one stops --
// none is left behind at a later named barrier.
__device__ __forceinline__ bool epilogue_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "n"(kEpiWarps * 32)
        : "memory");
    return r != 0;
}

// ----------------------------------------- LayerNorm after the linear layer

constexpr int kEpiPlain = 0;
constexpr int kEpiLayerNorm = 1;

// A value as the output type holds it (rounded to nearest even, read back).
template <typename OutT>
__device__ __forceinline__ float round_to_out(float v) {
    const OutT t = cvt_out<OutT>(v);
    return load_out<OutT>(&t);
}

// Stores 32 values of one C row at D' columns c0..c0+31 (the columns < N),
// cast to the output type; vector stores when the chunk is whole and aligned.
template <typename OutT>
__device__ __forceinline__ void store_out32(const TcParams& p, int32_t row, int32_t c0,
                                            const float (&v)[32]) {
    OutT* base = reinterpret_cast<OutT*>(p.C) + static_cast<int64_t>(row) * p.c_rs;
    if (p.c_vector && c0 + 32 <= p.N) {
        constexpr int kPer16 = 16 / sizeof(OutT);
        #pragma unroll
        for (int q = 0; q < 32 / kPer16; ++q) {
            uint4 pack;
            OutT* pk = reinterpret_cast<OutT*>(&pack);
            #pragma unroll
            for (int e = 0; e < kPer16; ++e) pk[e] = cvt_out<OutT>(v[q * kPer16 + e]);
            *reinterpret_cast<uint4*>(base + c0 + q * kPer16) = pack;
        }
    } else {
        #pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j < p.N) base[static_cast<int64_t>(c0 + j) * p.c_cs] = cvt_out<OutT>(v[j]);
    }
}

// Warp-collective: v[0..31] = TMEM row `taddr`, 32 consecutive columns.
__device__ __forceinline__ void tmem_row32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld_32x32b_x32(taddr, r);
    tmem_ld_wait();
    #pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// h for one row's 32 columns c0..c0+31 of the accumulator at TMEM address
// `taddr`: round_C(alpha * acc + beta * C + bias), 0 past column N.  The
// residual C and the bias are read only for rows inside the matrix (`rv`).
// Warp-collective (tcgen05.ld).
template <typename OutT>
__device__ __forceinline__ void ln_chunk_h(const TcParams& p, uint32_t taddr, int32_t row, bool rv,
                                           int32_t c0, float (&v)[32]) {
    tmem_row32(taddr, v);
    #pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= p.alpha;
    if (rv && c0 < p.N) {
        const OutT* base = reinterpret_cast<const OutT*>(p.C) + static_cast<int64_t>(row) * p.c_rs;
        if (p.beta != 0.0f) {
            if (p.c_vector && c0 + 32 <= p.N) {
                constexpr int kPer16 = 16 / sizeof(OutT);
                uint4 old[32 / kPer16];
                #pragma unroll
                for (int q = 0; q < 32 / kPer16; ++q)
                    old[q] = *reinterpret_cast<const uint4*>(base + c0 + q * kPer16);
                #pragma unroll
                for (int q = 0; q < 32 / kPer16; ++q) {
                    const OutT* o = reinterpret_cast<const OutT*>(&old[q]);
                    #pragma unroll
                    for (int e = 0; e < kPer16; ++e)
                        v[q * kPer16 + e] = fmaf(p.beta, load_out<OutT>(o + e), v[q * kPer16 + e]);
                }
            } else {
                #pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.N)
                        v[j] = fmaf(p.beta, load_out<OutT>(base + static_cast<int64_t>(c0 + j) * p.c_cs),
                                    v[j]);
            }
        }
        if (p.bias != nullptr) {
            float b[32];
            load_col_vec32(p.bias, p.bias_dtype, c0, p.N, b);
            #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += b[j];
        }
    }
    #pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (c0 + j < p.N) ? round_to_out<OutT>(v[j]) : 0.0f;
}

// The LayerNorm epilogue of one tile.  Each row's columns are split between
// two warps (alternate 32-column chunks); their partial sums meet in shared
// memory (red[0..2*kBlockM) for the mean, red[2*kBlockM..4*kBlockM) for M2).
// Pass 1 forms h = round_C(alpha * acc + beta * C + bias) (0 past column N),
// sums it and writes it back over the accumulator in TMEM: the later passes
// read TMEM only, and C (the residual) is read once, by the thread that
// overwrites it.  Pass 2 sums the squared deviations from the tile mean
// (two-pass, no cancellation) and, when a row spans several tiles, stores h.
// Pass 3 -- the row whole in this tile -- stores
// y = (h - mean) / sqrt(M2 / N + eps) * gamma + shift; otherwise the tile's
// (sum, M2) of each row go to ln_stats for the row pass.
template <typename OutT, int BN>
__device__ __forceinline__ void ln_tile(const TcParams& p, uint32_t t_row, int32_t row,
                                        int row_in_cta, int half, int32_t col0, int32_t tn,
                                        float* red) {
    const bool rv = row < p.M;
    const int32_t nvalid = (p.N - col0) < BN ? (p.N - col0) : BN;
    float s = 0.0f;
    #pragma unroll 1
    for (int ch = half; ch < BN / 32; ch += 2) {
        float v[32];
        ln_chunk_h<OutT>(p, t_row + ch * 32, row, rv, col0 + ch * 32, v);
        #pragma unroll
        for (int j = 0; j < 32; ++j) s += v[j];
        uint32_t r[32];
        #pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
        __syncwarp();                              // tcgen05.st is warp-collective
        tmem_st_32x32b_x32(t_row + ch * 32, r);
    }
    tmem_st_wait();                                // h is in TMEM before it is read back
    red[half * kBlockM + row_in_cta] = s;
    epilogue_bar_sync();
    const float mean = (red[row_in_cta] + red[kBlockM + row_in_cta]) / static_cast<float>(nvalid);
    float q = 0.0f;
    #pragma unroll 1
    for (int ch = half; ch < BN / 32; ch += 2) {
        float v[32];
        const int32_t c0 = col0 + ch * 32;
        tmem_row32(t_row + ch * 32, v);
        #pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float d = (c0 + j < p.N) ? v[j] - mean : 0.0f;
            q = fmaf(d, d, q);
        }
        if (!p.ln_fused && rv && c0 < p.N) store_out32<OutT>(p, row, c0, v);
    }
    red[(2 + half) * kBlockM + row_in_cta] = q;
    epilogue_bar_sync();
    const float m2 = red[2 * kBlockM + row_in_cta] + red[3 * kBlockM + row_in_cta];
    if (p.ln_fused) {
        const float rstd = 1.0f / sqrtf(m2 / static_cast<float>(nvalid) + p.ln_eps);
        #pragma unroll 1
        for (int ch = half; ch < BN / 32; ch += 2) {
            const int32_t c0 = col0 + ch * 32;
            float v[32];
            tmem_row32(t_row + ch * 32, v);
            if (rv && c0 < p.N) {
                #pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (v[j] - mean) * rstd;
                if (p.ln_gamma != nullptr) {
                    float g[32];
                    load_col_vec32(p.ln_gamma, p.ln_dtype, c0, p.N, g);
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= g[j];
                }
                if (p.ln_shift != nullptr) {
                    float t[32];
                    load_col_vec32(p.ln_shift, p.ln_dtype, c0, p.N, t);
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += t[j];
                }
                store_out32<OutT>(p, row, c0, v);
            }
        }
    } else if (half == 0 && rv) {
        const float sum = red[row_in_cta] + red[kBlockM + row_in_cta];
        p.ln_stats[static_cast<int64_t>(row) * p.tiles_n + tn] = make_float2(sum, m2);
    }
}

// MH = 2 (single CTA, plain epilogue, BN <= 128, data-parallel schedules):
//   a 256 x BN tile in one CTA, as two M = 128 halves.  One A box of 256 rows
//   per K chunk feeds both halves' MMAs, which share the chunk's B tile and
//   accumulate into two TMEM accumulators (columns [0, BN) and [BN, 2 BN) of
//   each buffer): twice the MMA per TMA box of a 128-row tile.  Epilogue warps
//   2-5 drain the first half, 6-9 the second.
template <int CG, int BN, typename OutT, int ES, int EPI = kEpiPlain, int KC = 1, int MH = 1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ TcParams p) {
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
    static_assert(EPI == kEpiPlain || EPI == kEpiLayerNorm, "epilogue");
    static_assert(KC == 1 || KC == 2, "K chunks per stage");
    static_assert(CG == 1 || (CG == 2 && BN >= 128), "CG");
    static_assert(ES == 2 || ES == 4, "element size");
    static_assert(MH == 1 || (MH == 2 && CG == 1 && EPI == kEpiPlain && BN <= 128), "MH");
    constexpr int kChunkK = Elem<ES>::kChunkK;
    constexpr int kUmmaK = Elem<ES>::kUmmaK;
    constexpr int kMNChunk = Elem<ES>::kMNChunk;
    constexpr int BM = kBlockM * CG * MH;                 // rows per (pair) tile
    constexpr int kARows = kBlockM * MH;                  // A rows this CTA loads
    constexpr uint32_t kBRows = BN / CG;                  // B rows this CTA loads
    // per stage: kc chunks of A (kBlockM rows) and of B (kBRows rows), each
    // chunk a 128-byte-wide swizzled tile; an MN-major box is 128 bytes of
    // M/N by kc * kChunkK rows of K
    constexpr int kc = KC;
    constexpr int32_t kBlockK = kc * kChunkK;             // K elements per stage
    constexpr uint32_t kATile = static_cast<uint32_t>(kc) * kARows * 128u;
    constexpr uint32_t kBTile = static_cast<uint32_t>(kc) * kBRows * 128u;
    constexpr uint32_t kStageBytes = kATile + kBTile;
    static_assert(kStageBytes % 1024 == 0, "stages keep the C staging boxes 1024-byte aligned");
    constexpr uint32_t kChunkBytes = static_cast<uint32_t>(kBlockK) * 128u;   // one MN-major box
    constexpr uint32_t kTmemCols = 2 * MH * BN;          // double-buffered accumulator(s)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    // whole-row convolution tiles (conv_tiled) run on 256-row tiles only
    const bool whole_rows = MH == 2 && p.conv_tiled != 0;
    const bool halo = MH == 2 && p.conv_tiled == 2;
    const uint32_t stage_bytes = halo ? p.halo_stage_bytes : kStageBytes;
    const uint32_t a_region = halo ? p.halo_a_region : kATile;
    // [stages][C staging, when C is stored by TMA][barriers]
    uint8_t* cstage = smem + S * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(cstage + (p.c_tma ? kCStageBytes : 0u));
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
        if (p.c_tma) tma_prefetch_desc(&tmC);
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
    // Everything above (barrier set-up, TMEM allocation, descriptor prefetch)
    // may overlap the previous kernel on the stream; nothing below touches
    // global memory before that kernel has completed.
    grid_dependency_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // Operands that every tile re-reads stay in L2 (evict-last); an
            // operand streamed once (the weights of a skinny GEMM) is marked
            // evict-first so it does not push the reused one out.
            const uint64_t pol_a = l2_policy(p.a_policy);
            const uint64_t pol_b = l2_policy(p.b_policy);
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0;                   // number of slot armings so far
            uint32_t seg_i = 0;                   // segments (tiles) so far
            SegmentIter it(p, unit, units);
            Segment sg;
            bool ok = true;
            while (ok && it.next(p, sg)) {
                int32_t tm, tn;
                tile_coords(p, sg.tile, tm, tn);
                // Serpentine K: a CTA's odd tiles walk K backwards.  The CTAs
                // run their j-th tiles together (one wave), so a wave starts
                // where the previous one ended: on the k-blocks it left most
                // recently in L2, which the next wave's tiles that share its
                // strips then find there.  (The MMA warp only counts k-blocks.)
                const bool rev = p.serpentine && (seg_i & 1u);
                ++seg_i;
                // Parts of a CTA's A / B tiles that lie wholly outside the
                // matrix only feed outputs that are never stored: not loaded.
                // tile_bytes(r) is what CTA r of the pair loads per k-block.
                auto a_parts = [&](int32_t m_first) {
                    if (!p.a_mn_major) return (m_first < p.M) ? 1 : 0;
                    int n = 0;
                    for (int c = 0; c < kARows / kMNChunk; ++c) n += (m_first + kMNChunk * c < p.M);
                    return n;
                };
                auto b_parts = [&](int32_t n_first) {
                    if (!p.b_mn_major) return (n_first < p.N) ? 1 : 0;
                    int n = 0;
                    for (int c = 0; c < static_cast<int>(kBRows) / kMNChunk; ++c)
                        n += (n_first + kMNChunk * c < p.N);
                    return n;
                };
                auto tile_bytes = [&](uint32_t r) {
                    const int32_t mf = tm * BM + static_cast<int32_t>(r) * kARows;
                    const int32_t nf = tn * BN + static_cast<int32_t>(r * kBRows);
                    if (halo)
                        return p.conv_a_bytes +
                               static_cast<uint32_t>(b_parts(nf)) * p.conv_R * kBRows * 128u;
                    if (whole_rows)
                        return static_cast<uint32_t>(kc) * p.conv_a_bytes +
                               static_cast<uint32_t>(b_parts(nf)) * kBTile;
                    return static_cast<uint32_t>(a_parts(mf)) *
                               (p.a_mn_major ? kChunkBytes : kATile) +
                           static_cast<uint32_t>(b_parts(nf)) *
                               (p.b_mn_major ? kChunkBytes : kBTile);
                };
                const int32_t m0 = tm * BM + static_cast<int32_t>(rank) * kARows;
                const int32_t n0 = tn * BN + static_cast<int32_t>(rank * kBRows);
                const int na = a_parts(m0), nb = b_parts(n0);
                // The even CTA's "full" barrier counts the bytes of both CTAs;
                // the odd CTA's loads may land before it is armed (the
                // transaction count may go transiently negative).
                const uint32_t bytes = (CG == 1) ? tile_bytes(0)
                                                 : (rank == 0 ? tile_bytes(0) + tile_bytes(1) : 0u);
                // convolution: the first window of this CTA's rows (output
                // pixel m0) as the input coordinates of its top-left pixel
                int32_t cn = 0, ch = 0, cw = 0;
                if (whole_rows) {
                    // the tile's image and first output row
                    cn = tm / p.conv_tpi;
                    ch = (tm - cn * p.conv_tpi) * p.conv_rows - p.conv_pad_h;
                    cw = -p.conv_pad_w;
                } else if (p.conv) {
                    const int32_t pq = p.conv_P * p.conv_Q;
                    cn = m0 / pq;
                    const int32_t rem = m0 - cn * pq;
                    const int32_t pp = rem / p.conv_Q;
                    ch = pp * p.conv_stride_h - p.conv_pad_h;
                    cw = (rem - pp * p.conv_Q) * p.conv_stride_w - p.conv_pad_w;
                }
                for (int32_t kbi = sg.kb0; kbi < sg.kb1; ++kbi) {
                    const int32_t kb = rev ? sg.kb0 + sg.kb1 - 1 - kbi : kbi;
                    if (!wait_or_abort(&empty[stage], phase ^ 1u, &abort_flag, p.wait_limit_ns)) {
                        record_error(p, kErrTimeoutProducer, &abort_flag);
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * stage_bytes;
                    uint8_t* sb = sa + a_region;
                    const int32_t k0 = kb * kBlockK;
                    if ((p.debug_flags & kDebugSkipFirstLoad) && armed == 0 && blockIdx.x == 0) {
                        // test hook: arm the slot, load nothing into it
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], bytes > 0 ? bytes : 16u);
                        ++armed;
                        if (++stage == static_cast<uint32_t>(S)) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    if (MH == 2 && halo) {
                        // filter column s, channel block cb: the halo box, then
                        // the column's R taps (3-D filter map, one box per tap)
                        if constexpr (CG == 1 && MH == 2) {
                            mbar_arrive_expect_tx(&full[stage], bytes);
                            const int32_t sc = kb / p.conv_cblocks;
                            const int32_t cb0 = (kb - sc * p.conv_cblocks) * kChunkK;
                            tma_load_4d(sa, &tmA, &full[stage], cb0, cw + sc * p.conv_dil_w, ch, cn,
                                        pol_a);
                            if (nb) {
                                for (int32_t r = 0; r < p.conv_R; ++r)
                                    tma_load_3d(sb + r * kBRows * 128u, &tmB, &full[stage], cb0,
                                                r * p.conv_S + sc, n0, pol_b);
                            }
                        }
                    } else if (p.conv) {
                        // chunk j = kb * kc + q: channels c0 .. c0 + 63 of filter
                        // tap (r, s), the channel blocks of one tap back to back
                        uint32_t fb = 0;                       // the even CTA's barrier (pairs)
                        if constexpr (CG == 2) fb = map_to_rank(smem_addr(&full[stage]), 0);
                        if (CG == 1 || rank == 0) mbar_arrive_expect_tx(&full[stage], bytes);
                        int32_t c0 = 0, tap = 0;
                        #pragma unroll
                        for (int q = 0; q < kc; ++q) {
                            const int32_t j = kb * kc + q;
                            tap = j / p.conv_cblocks;
                            c0 = (j - tap * p.conv_cblocks) * kChunkK;
                            if (tap >= p.conv_taps) {          // past the last tap: zeros
                                tap = 0;
                                c0 = p.conv_cblocks * kChunkK;
                            }
                            const int32_t r = tap / p.conv_S;
                            const uint16_t ow = static_cast<uint16_t>((tap - r * p.conv_S) * p.conv_dil_w);
                            const uint16_t oh = static_cast<uint16_t>(r * p.conv_dil_h);
                            if (whole_rows) {
                                // the tap's window of the tile's output rows:
                                // input (cw + ow + q', ch + oh + p') for output (p', q')
                                if constexpr (CG == 1)
                                    tma_load_4d(sa + q * kARows * 128, &tmA, &full[stage], c0,
                                                cw + ow, ch + oh, cn, pol_a);
                            } else if (na) {
                                if constexpr (CG == 1)
                                    tma_load_im2col_4d(sa + q * kARows * 128, &tmA, &full[stage], c0, cw,
                                                       ch, cn, ow, oh, pol_a);
                                else
                                    tma_load_im2col_4d_pair(sa + q * kARows * 128, &tmA, fb, c0, cw, ch,
                                                            cn, ow, oh, pol_a);
                            }
                        }
                        if (nb) {
                            if constexpr (kc == 1) {
                                if constexpr (CG == 1) tma_load_3d(sb, &tmB, &full[stage], c0, tap, n0, pol_b);
                                else tma_load_3d_pair(sb, &tmB, fb, c0, tap, n0, pol_b);
                            } else {
                                if constexpr (CG == 1) tma_load_3d(sb, &tmB, &full[stage], 0, n0, kb * kc, pol_b);
                                else tma_load_3d_pair(sb, &tmB, fb, 0, n0, kb * kc, pol_b);
                            }
                        }
                    } else if constexpr (CG == 1) {
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        if (p.a_mn_major) {
                            for (int c = 0; c < na; ++c)
                                tma_load_2d(sa + c * kChunkBytes, &tmA, &full[stage], m0 + kMNChunk * c,
                                            k0, pol_a);
                        } else if (na) {
                            if constexpr (kc == 1) tma_load_2d(sa, &tmA, &full[stage], k0, m0, pol_a);
                            else tma_load_3d(sa, &tmA, &full[stage], 0, m0, kb * kc, pol_a);
                        }
                        if (p.b_mn_major) {
                            for (int c = 0; c < nb; ++c)
                                tma_load_2d(sb + c * kChunkBytes, &tmB, &full[stage], n0 + kMNChunk * c,
                                            k0, pol_b);
                        } else if (nb) {
                            if constexpr (kc == 1) tma_load_2d(sb, &tmB, &full[stage], k0, n0, pol_b);
                            else tma_load_3d(sb, &tmB, &full[stage], 0, n0, kb * kc, pol_b);
                        }
                    } else {
                        const uint32_t fb = map_to_rank(smem_addr(&full[stage]), 0);
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], bytes);
                        if (p.a_mn_major) {
                            for (int c = 0; c < na; ++c)
                                tma_load_2d_pair(sa + c * kChunkBytes, &tmA, fb, m0 + kMNChunk * c, k0,
                                                 pol_a);
                        } else if (na) {
                            if constexpr (kc == 1) tma_load_2d_pair(sa, &tmA, fb, k0, m0, pol_a);
                            else tma_load_3d_pair(sa, &tmA, fb, 0, m0, kb * kc, pol_a);
                        }
                        if (p.b_mn_major) {
                            for (int c = 0; c < nb; ++c)
                                tma_load_2d_pair(sb + c * kChunkBytes, &tmB, fb, n0 + kMNChunk * c, k0,
                                                 pol_b);
                        } else if (nb) {
                            if constexpr (kc == 1) tma_load_2d_pair(sb, &tmB, fb, k0, n0, pol_b);
                            else tma_load_3d_pair(sb, &tmB, fb, 0, n0, kb * kc, pol_b);
                        }
                    }
                    ++armed;
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every load of this CTA is issued: the next kernel on the stream
            // may begin its own set-up on SMs as they free up.
            grid_dependents_launch();
            // Wind-down: wait (bounded) until every TMA load issued into this
            // CTA pair has landed.  The even CTA's "full" barriers count the
            // bytes of both CTAs, so only the even CTA waits; the odd CTA is
            // held by the cluster barrier before exit until then.
            if (rank == 0) {
                for (int s = 0; s < S; ++s) {
                    if (armed <= static_cast<uint32_t>(s)) break;
                    const uint32_t last = ((armed - 1 - s) / S) * S + s;   // last arming of slot s
                    if (!mbar_wait(&full[s], (last / S) & 1u, p.wait_limit_ns))
                        record_error(p, kErrTimeoutProducer, &abort_flag);
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
            // advance per MMA: K-major 32 bytes within the 128-byte row, and
            // the next chunk's tile after four; MN-major kUmmaK rows of 128 bytes
            const uint32_t a_kstep = p.a_mn_major ? kUmmaK * 128u : kUmmaK * ES;
            const uint32_t b_kstep = p.b_mn_major ? kUmmaK * 128u : kUmmaK * ES;
            const uint32_t a_cstep = p.a_mn_major ? 4u * a_kstep : kARows * 128u;
            // MH = 2: the second half's A rows, 128 rows on (K-major) or two
            // 64-row MN-major boxes on
            const uint32_t a_hstep = p.a_mn_major ? 2u * kChunkBytes : kATileBytes;
            const uint32_t b_cstep = p.b_mn_major ? 4u * b_kstep : kBRows * 128u;

            const uint32_t smem_base = smem_addr(smem);
            while (ok && it.next(p, sg)) {
                const uint32_t buf = acc_i & 1u;
                if (!wait_role<CG>(&acc_empty[buf], ((acc_i >> 1) & 1u) ^ 1u, &abort_flag, p.wait_limit_ns)) {
                    record_error(p, kErrTimeoutMma, &abort_flag);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * (MH * BN);
                for (int32_t kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!wait_or_abort(&full[stage], phase, &abort_flag, p.wait_limit_ns)) {
                        record_error(p, kErrTimeoutMma, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = smem_base + stage * stage_bytes;
                    const uint32_t sb = sa + a_region;
                    if (MH == 2 && halo) {
                        // tap r of this filter column: A from halo row
                        // r * dil_h * pitch on (a multiple of 8 rows, so the
                        // swizzle atoms line up), its own B tile.  The
                        // descriptors advance by (byte offset >> 4) added to
                        // their start-address field (shared-memory offsets
                        // never overflow its 14 bits): one add per MMA
                        const uint32_t a_tap = static_cast<uint32_t>(p.conv_dil_h * p.conv_pitch) * 8u;
                        const uint64_t a_desc = smem_desc_sw128(sa, 16u, 1024);
                        const uint64_t b_desc = smem_desc_sw128(sb, 16u, 1024);
                        // A and B share the high word (stride offset, layout)
                        const uint32_t hi = static_cast<uint32_t>(a_desc >> 32);
                        uint32_t ar = static_cast<uint32_t>(a_desc);
                        uint32_t br = static_cast<uint32_t>(b_desc);
                        uint32_t acc = kb > sg.kb0 ? 1u : 0u;
                        for (int32_t r = 0; r < p.conv_R; ++r, ar += a_tap, br += kBRows * 8u) {
                            #pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                if constexpr (ES == 2 && CG == 1 && MH == 2)
                                    tc_mma_f16_x2(d_tmem, d_tmem + BN, ar + kk * 2u,
                                                  ar + kk * 2u + (kATileBytes >> 4), br + kk * 2u, hi,
                                                  p.idesc, acc);
                                acc = 1u;
                            }
                        }
                    } else {
                    #pragma unroll
                    for (int kk = 0; kk < kc * 4; ++kk) {
                        const uint32_t ka = (kk >> 2) * a_cstep + (kk & 3) * a_kstep;
                        const uint32_t kb2 = (kk >> 2) * b_cstep + (kk & 3) * b_kstep;
                        const uint64_t ad = smem_desc_sw128(sa + ka, a_lbo, 1024);
                        const uint64_t bd = smem_desc_sw128(sb + kb2, b_lbo, 1024);
                        const uint32_t acc = (kb > sg.kb0 || kk > 0) ? 1u : 0u;
                        if constexpr (ES == 4) {
                            if constexpr (CG == 1) tc_mma_tf32(d_tmem, ad, bd, p.idesc, acc);
                            else tc_mma_tf32_pair(d_tmem, ad, bd, p.idesc, acc);
                        } else {
                            if constexpr (CG == 1) tc_mma_f16(d_tmem, ad, bd, p.idesc, acc);
                            else tc_mma_f16_pair(d_tmem, ad, bd, p.idesc, acc);
                        }
                        if constexpr (MH == 2) {
                            // the second half: its A rows, the same B, its accumulator
                            const uint64_t ad2 = ad + (a_hstep >> 4);
                            if constexpr (ES == 4) tc_mma_tf32(d_tmem + BN, ad2, bd, p.idesc, acc);
                            else tc_mma_f16(d_tmem + BN, ad2, bd, p.idesc, acc);
                        }
                    }
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
            if (!mbar_wait(drain, 0, p.wait_limit_ns)) record_error(p, kErrTimeoutMma, &abort_flag);
        }
    } else {
        // --------------------------------------------------------- epilogue
        // Warp w may read TMEM lanes 32*(w%4)..+31: two epilogue warps share each
        // lane quarter and take alternate 32-column chunks of the tile (MH = 2:
        // the two warps of a lane quarter take the two halves' accumulators,
        // every chunk of each).
        const int quarter = warp & 3;                   // TMEM lanes 32*quarter..+31
        const int half = (warp - 2) >> 2;               // 0: even chunks, 1: odd chunks (MH = 2: M half)
        const int row_in_cta = quarter * 32 + lane;
        const int row_in_tile = (MH == 2 ? half : static_cast<int>(rank)) * kBlockM + row_in_cta;
        const int ch_first = MH == 2 ? 0 : half;        // this warp's first chunk and step
        const int ch_step = MH == 2 ? 1 : 2;
        uint32_t acc_i = 0;
        uint32_t cstep = 0;                     // TMA-store steps so far (the same in every warp)
        SegmentIter it(p, unit, units);
        Segment sg;
        __shared__ int wait_ok;
        // LayerNorm: the two warps of each row exchange partial sums here
        __shared__ float ln_red[EPI == kEpiLayerNorm ? 4 * kBlockM : 1];
        while (it.next(p, sg)) {
            const uint32_t buf = acc_i & 1u;
            int32_t tm, tn;
            tile_coords(p, sg.tile, tm, tn);
            int32_t row = tm * BM + row_in_tile;                    // D' row
            if (whole_rows) {
                // output pixel row_in_tile of the tile's conv_rows image rows
                // (rows past the image's last output row are not stored)
                const int32_t n = tm / p.conv_tpi;
                const int32_t p0 = (tm - n * p.conv_tpi) * p.conv_rows;
                const int32_t nrow = p.conv_P - p0 < p.conv_rows ? p.conv_P - p0 : p.conv_rows;
                const int32_t pl = row_in_tile / p.conv_pitch;
                const int32_t q = row_in_tile - pl * p.conv_pitch;
                row = (pl < nrow && q < p.conv_Q) ? (n * p.conv_P + p0 + pl) * p.conv_Q + q : p.M;
            }
            const int32_t col0 = tn * BN;                           // D' first column
            const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            const uint32_t t_row = t_lane + buf * (MH * BN) + (MH == 2 ? half * BN : 0);  // this tile's sums
            const uint32_t t_spare = t_lane + (buf ^ 1u) * BN;     // the other buffer (MH = 1)

            // Stream-K tile split across CTAs g_first..g_last.  g_first, which
            // holds the tile's first k-blocks, finishes it.  For g_first this
            // segment is the last of its range (a range is at most one tile
            // long), so it ends last, the MMA warp will not write the other
            // TMEM buffer again, and the epilogue warps are idle until its sums
            // arrive.  They use that time: wait (bounded) until every other
            // contributor has stored its sums and counted itself on the tile's
            // counter, add those sums in increasing CTA order and park the
            // total in the spare TMEM buffer.  When the finisher's own sums
            // land, total + own goes through the epilogue -- the same order on
            // every run.  The others store their sums to their slot.
            const int32_t KB = p.k_blocks, L = p.sk_len;
            int32_t g_first = 0, g_last = -1;
            bool finisher = false;
            bool ok = true;
            if (MH == 1 && sg.slot >= 0) {                        // (MH = 2: never split)
                g_first = static_cast<int32_t>((static_cast<int64_t>(sg.tile) * KB) / L);
                g_last = static_cast<int32_t>((static_cast<int64_t>(sg.tile + 1) * KB - 1) / L);
                finisher = (unit == g_first);
            }
            if (MH == 1 && finisher) {
                // one counter per tile and CTA of the pair: CTA r of a pair
                // finishes rows r * 128.. of the tile from the sums that CTA
                // r of each contributing pair stored
                int* written = p.tile_counters + sg.tile * CG + static_cast<int32_t>(rank);
                if (warp == 2 && lane == 0) {
                    const bool w = wait_counter(written, g_last - g_first, &abort_flag, p.wait_limit_ns);
                    if (w) *written = 0;                    // self-resetting for the next call
                    else record_error(p, kErrTimeoutEpilogue, &abort_flag);
                    wait_ok = w ? 1 : 0;
                }
                epilogue_bar_sync();
                ok = (wait_ok != 0);
                __threadfence();
                if (ok) {
                    #pragma unroll 1
                    for (int ch = half; ch < BN / 32; ch += 2) {
                        float acc[32];
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
                        // 16 columns at a time, up to kFinBatch slots' loads in
                        // flight together; each warp load is 512 contiguous bytes
                        #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            for (int32_t g0 = g_first + 1; g0 <= g_last; g0 += kFinBatch) {
                                float x[kFinBatch][16];
                                #pragma unroll
                                for (int u = 0; u < kFinBatch; ++u) {
                                    const int32_t g = g0 + u;
                                    if (g > g_last) continue;
                                    const int32_t first_tile =
                                        static_cast<int32_t>((static_cast<int64_t>(g) * L) / KB);
                                    const float4* s4 =
                                        reinterpret_cast<const float4*>(
                                            p.partials + (static_cast<int64_t>(g) * p.sk_max_seg +
                                                          (sg.tile - first_tile)) * BM * BN) +
                                        (ch * 8 + h * 4) * BM + row_in_tile;
                                    #pragma unroll
                                    for (int q = 0; q < 4; ++q) {
                                        const float4 t = __ldcg(s4 + q * BM);
                                        x[u][4 * q] = t.x;
                                        x[u][4 * q + 1] = t.y;
                                        x[u][4 * q + 2] = t.z;
                                        x[u][4 * q + 3] = t.w;
                                    }
                                }
                                #pragma unroll
                                for (int u = 0; u < kFinBatch; ++u) {
                                    if (g0 + u > g_last) break;
                                    #pragma unroll
                                    for (int j = 0; j < 16; ++j) acc[h * 16 + j] += x[u][j];
                                }
                            }
                        }
                        uint32_t r[32];
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
                        __syncwarp();                  // tcgen05.st is warp-collective
                        tmem_st_32x32b_x32(t_spare + ch * 32, r);
                    }
                    tmem_st_wait();
                }
            }
            ok = ok && wait_or_abort(&acc_full[buf], (acc_i >> 1) & 1u, &abort_flag, p.wait_limit_ns);
            // stream-K, LayerNorm and the TMA store of C use named barriers below
            if (p.stream_k || EPI == kEpiLayerNorm || p.c_tma) ok = epilogue_all(ok);
            if (!ok) {
                record_error(p, kErrTimeoutEpilogue, &abort_flag);
                break;
            }
            tc_fence_after_sync();
            if constexpr (EPI == kEpiLayerNorm) {
                // data-parallel only (the planner gives LayerNorm no stream-K)
                ln_tile<OutT, BN>(p, t_row, row, row_in_cta, half, col0, tn, ln_red);
            } else {
                float* my_slot = (MH == 1 && sg.slot >= 0 && !finisher)
                                     ? p.partials + static_cast<int64_t>(sg.slot) * BM * BN
                                     : nullptr;
                #pragma unroll 1
                for (int ch = ch_first; ch < BN / 32; ch += ch_step) {
                    uint32_t r[32];
                    __syncwarp();                      // tcgen05.ld is warp-collective
                    tmem_ld_32x32b_x32(t_row + ch * 32, r);
                    tmem_ld_wait();
                    float v[32];
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (MH == 1 && finisher) {
                        uint32_t o[32];
                        __syncwarp();
                        tmem_ld_32x32b_x32(t_spare + ch * 32, o);
                        tmem_ld_wait();
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(o[j]) + v[j];
                    }
                    const int32_t c0 = col0 + ch * 32;
                    if (my_slot == nullptr) epilogue_values<OutT>(p, row, c0, v);
                    if (MH == 1 && my_slot == nullptr && p.c_tma) {
                        // C through shared memory: step ch / 2 of the tile is
                        // 64 columns (one 32-column chunk per half); the eight
                        // warps fill the staging box(es) and one thread stores
                        // them by TMA
                        uint8_t* box;
                        int u0;
                        if constexpr (sizeof(OutT) == 4) {
                            box = cstage + half * kCBoxBytes;      // 32 columns per box
                            u0 = 0;
                        } else {
                            box = cstage + (cstep & 1u) * kCBoxBytes;   // 64 columns, two buffers
                            u0 = 4 * half;
                        }
                        if (warp == 2 && lane == 0) {
                            // the box's previous store has finished reading it
                            if constexpr (sizeof(OutT) == 4) bulk_wait_group_read<0>();
                            else bulk_wait_group_read<1>();
                        }
                        epilogue_bar_sync();
                        stage_row32<OutT>(box, row_in_cta, u0, v);
                        fence_proxy_async_shared();
                        epilogue_bar_sync();
                        if (warp == 2 && lane == 0) {
                            const int32_t y = tm * BM + static_cast<int32_t>(rank) * kBlockM;
                            const int32_t x = col0 + (ch >> 1) * 64;
                            if (y < p.M) {
                                if constexpr (sizeof(OutT) == 4) {
                                    if (x < p.N) tma_store_2d(&tmC, cstage, x, y);
                                    if (x + 32 < p.N) tma_store_2d(&tmC, cstage + kCBoxBytes, x + 32, y);
                                } else {
                                    if (x < p.N) tma_store_2d(&tmC, box, x, y);
                                }
                            }
                            bulk_commit_group();
                        }
                        ++cstep;
                    } else if (my_slot == nullptr) {
                        store_row32<OutT>(p, row, c0, v);
                    } else {
                        // raw FP32 sums as float4s of four columns, laid out
                        // [column / 4][row]: the 32 rows of a warp store (and of
                        // the finisher's load) are 512 contiguous bytes
                        float4* dst = reinterpret_cast<float4*>(my_slot) + (ch * 8) * BM + row_in_tile;
                        #pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q * BM] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
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
            if (sg.slot >= 0) {
                if (!finisher) {
                    __threadfence();                       // this thread's slot stores
                    epilogue_bar_sync();
                    if (warp == 2 && lane == 0)
                        atomicAdd(p.tile_counters + sg.tile * CG + static_cast<int32_t>(rank), 1);
                }
                epilogue_bar_sync();                       // wait_ok is reused by the next tile
            }
        }
        // the C stores have written global memory and released the staging
        // boxes before the CTA moves on to exit
        if (p.c_tma && warp == 2 && lane == 0) bulk_wait_group_all();
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

}  // namespace gemm103
