// api.cu -- the C ABI (include/gemm_sm103.h): argument validation, the host
// planner that picks a kernel path, TMA descriptor encoding, workspace
// management and the launches.
//
// The planner follows the pages' measurement-first split between
// compute-bound and memory-bound GEMMs (SGEMM page, section 1.2; DeepGEMM
// page, section 2.4; CATLASS page, section 3.1): large problems run the
// data-parallel persistent tensor-core kernel; problems with fewer output
// tiles than SMs spread their K loop across SMs (stream-K) so the whole GPU
// streams the operands; very small M swaps the operands so the 128-row MMA
// dimension is filled by the large side (the skinny, memory-bound path).
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_sm103.h"
#include "conv_sm103.h"
#include "aux_kernels.cuh"
#include "launch.h"

using namespace gemm103;

namespace {

constexpr int kMaxStages = 8;
constexpr int kGroupM = 8;
// Raster (raster_columns): the B strips that one group of tile-columns keeps
// in L2 fit in this many bytes (half of GB300's L2: each die's half caches
// what that die's SMs read), and a group has at most kRasterMaxColumns.
constexpr int64_t kRasterResidentBytes = 64ll << 20;
constexpr int64_t kRasterMaxColumns = 16;
// Data-parallel tiles alternate their K direction from wave to wave.
constexpr bool kSerpentineK = true;
// Workspace header: one stream-K counter (int32: contributors that have
// stored their sums) per output tile; the planner uses stream-K only for
// schedules of at most 1024 tiles.
constexpr int64_t kWsHeaderBytes = 4096;
constexpr int64_t kMaxCounterTiles = kWsHeaderBytes / 4;
// Stream-K thresholds: tiles at least this many k-blocks long, and data-parallel
// schedules whose last wave leaves more than 1 - kMinWaveFill of the GPU idle.
constexpr int32_t kLongK = 32;
constexpr double kMinWaveFill = 0.8;
// An operand read once and at least this large (about three quarters of the
// GB300 L2) is loaded evict-first so that it does not push reused data out.
constexpr int64_t kStreamOnceBytes = 96ll << 20;
// Convolutions with at most 128 output channels run 256-row single-CTA tiles
// (make_plan's mh2): the im2col box of 256 output pixels feeds two MMAs.
constexpr bool kConvTwoHalves = true;
// ... and, at stride 1, tiles of whole output rows loaded by tiled boxes,
// as halo units (one box per filter column) where they fit.
constexpr bool kConvWholeRows = true;
constexpr bool kConvHalo = true;
// Stream-K fix-up: one FP32 partial tile read back by the finisher costs about
// as long as this many k-blocks of 256 bytes per row (128 BF16 / FP16 or 64
// TF32 elements) of the tile's MMA (measured on GB300).
constexpr double kSkFixupKBlocks = 8.0;

struct OperandDesc {
    // stored matrix: rows x cols with pitch ld (elements); K-major means the
    // contiguous direction is K (cols == K), MN-major means it is M or N.
    const void* ptr;
    int64_t rows, cols, ld;
    bool mn_major;
    bool pack;          // needs a 16-byte-aligned copy
    bool transpose;     // the copy also transposes (FP32 MN-major -> K-major)
    int64_t packed_ld;
};

struct Plan {
    gemm_plan_t pub;
    OperandDesc a, b;   // kernel operands (after an optional swap)
    int64_t Mk, Nk;     // kernel rows / columns (M', N')
    int64_t K;
    int64_t c_rs, c_cs;
    int32_t k_blocks, tiles_m, tiles_n;
    int32_t kc;         // K chunks (128-byte rows of K) per pipeline stage
    int32_t cta_group;
    int32_t mh;         // M halves per single-CTA tile: 1 (128 rows) or 2 (256 rows)
    int32_t esize;      // input element bytes: 2 (FP16/BF16) or 4 (FP32 as TF32)
    int32_t sk_len, sk_max_seg;
    int64_t pack_a_bytes, pack_b_bytes, partial_bytes;
    size_t smem_bytes;
    // LayerNorm after the linear layer: whole rows in one tile (normalised in
    // the epilogue), else per-tile row statistics for a row pass
    bool ln;
    bool ln_fused;
    int64_t ln_stats_bytes;
    // the plain epilogue stores C through shared memory by TMA (C rows
    // 16-byte aligned, not swapped): kCStageBytes of staging after the stages
    bool c_tma;
    // convolution on whole-row tiles (conv_plan): output rows per tile and
    // tiles per image; 0 for im2col tiles.  conv_halo: halo units (pitch,
    // the halo box's bytes, the A region and the whole stage)
    int32_t conv_rows, conv_tpi;
    bool conv_halo;
    int32_t conv_pitch;
    uint32_t halo_box_bytes, halo_a_region, halo_stage_bytes;
};

bool is_n(char t) { return t == 'N' || t == 'n'; }
bool is_t(char t) { return t == 'T' || t == 't'; }
int64_t max1(int64_t v) { return v > 1 ? v : 1; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
size_t out_elem_bytes(int32_t c) { return c == GEMM_F32 ? 4 : 2; }
int32_t in_elem_bytes(int32_t ab) { return ab == GEMM_F32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

gemm_status_t check_args(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                         const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                         const void* C, int64_t ldc, gemm_dtypes_t dt) {
    if (!(is_n(transA) || is_t(transA)) || !(is_n(transB) || is_t(transB)))
        return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    // TMA coordinates and tile indices are 32-bit.
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_VALUE;
    if (dt.a != dt.b || (dt.a != GEMM_F16 && dt.a != GEMM_BF16 && dt.a != GEMM_F32))
        return GEMM_ERR_INVALID_VALUE;
    if (dt.c != GEMM_F32 && dt.c != GEMM_F16 && dt.c != GEMM_BF16) return GEMM_ERR_INVALID_VALUE;
    const int64_t a_cols = is_n(transA) ? K : M;
    const int64_t b_cols = is_n(transB) ? N : K;
    if (lda < max1(a_cols) || ldb < max1(b_cols) || ldc < max1(N)) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr || !aligned_to(C, out_elem_bytes(dt.c))) return GEMM_ERR_INVALID_VALUE;
    const bool reads_ab = (K > 0 && alpha != 0.0f);
    if (reads_ab && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_VALUE;
    // Every element must sit on its own size's boundary (the pack pre-pass
    // reads the operands element by element).
    const size_t es = static_cast<size_t>(in_elem_bytes(dt.a));
    if (reads_ab && (!aligned_to(A, es) || !aligned_to(B, es))) return GEMM_ERR_INVALID_VALUE;
    (void)beta;
    return GEMM_OK;
}

// Pick the kernel path, tile shape, schedule and workspace for a problem.
gemm_status_t make_plan(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                        const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                        const void* C, int64_t ldc, gemm_dtypes_t dt, int32_t num_sms,
                        int32_t smem_optin, Plan& pl, bool allow_swap = true, bool ln = false,
                        int32_t max_kc = kMaxKc, int32_t min_kc2_stages = 3,
                        bool allow_sk = true, int32_t max_sk_units = 0, bool mh2 = false) {
    gemm_status_t st = check_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt);
    if (st != GEMM_OK) return st;
    if (num_sms < 1 || smem_optin < 64 * 1024) return GEMM_ERR_INVALID_VALUE;
    std::memset(&pl, 0, sizeof pl);
    pl.pub.split_k = 1;
    pl.K = K;
    pl.ln = ln;
    if (M == 0 || N == 0) {
        pl.pub.path = GEMM_PATH_NOOP;
        return GEMM_OK;
    }
    if (K == 0 || alpha == 0.0f) {
        pl.pub.path = GEMM_PATH_SCALE;
        return GEMM_OK;
    }

    // Operand descriptions in the problem's own orientation.
    OperandDesc opA, opB;
    opA.ptr = A;
    opA.mn_major = is_t(transA);            // stored K x M
    opA.rows = opA.mn_major ? K : M;
    opA.cols = opA.mn_major ? M : K;
    opA.ld = lda;
    opB.ptr = B;
    opB.mn_major = is_n(transB);            // stored K x N
    opB.rows = opB.mn_major ? K : N;
    opB.cols = opB.mn_major ? N : K;
    opB.ld = ldb;

    // Skinny M: compute C^T = op(B)^T op(A)^T so the large N fills the
    // 128-row MMA side and the small M becomes the MMA's N.  Always for
    // M <= 64; for M <= 128 (one tile row either way) only when the unswapped
    // one-row plan would leave its single wave of 128-wide tiles under 80 %
    // full and balance it by stream-K over 256-wide tiles, which the swapped
    // stream-K beats (measured on GB300, FP16, weights N x K: M = 80-128 x
    // 14336 x 4096 32 -> 27 us swapped, while 16384 x 8192 (one wave 84 %
    // full) and 4096 x 4096 (too few tiles for a wave) ran 10-25 % faster
    // unswapped).
    const int64_t one_row_tiles = ceil_div(N, 128);
    const double one_row_fill =
        static_cast<double>(one_row_tiles) /
        static_cast<double>(ceil_div(one_row_tiles, num_sms) * num_sms);
    const bool mid_swap = M > 64 && M <= 128 && K >= kLongK * 64 &&
                          one_row_tiles >= (num_sms + 1) / 2 && one_row_fill < kMinWaveFill;
    const bool swap = allow_swap && !ln && N >= 128 && (M <= 64 || mid_swap);
    pl.pub.swap_ab = swap ? 1 : 0;
    if (swap) {
        pl.a = opB;
        pl.b = opA;
        pl.Mk = N;
        pl.Nk = M;
        pl.c_rs = 1;
        pl.c_cs = ldc;
    } else {
        pl.a = opA;
        pl.b = opB;
        pl.Mk = M;
        pl.Nk = N;
        pl.c_rs = ldc;
        pl.c_cs = 1;
    }
    // A K chunk is one 128-byte swizzle row of K: 64 16-bit or 32 32-bit
    // elements.  A stage holds kc chunks (below).
    const int32_t esize = in_elem_bytes(dt.a);
    const int64_t chunk_k = 128 / esize;
    pl.esize = esize;
    for (OperandDesc* o : {&pl.a, &pl.b}) {
        o->pack = !aligned16(o->ptr) || ((o->ld * esize) % 16) != 0;
        o->transpose = false;
        o->packed_ld = o->pack ? round_up(o->cols, 16 / esize) : o->ld;
        if (esize == 4 && o->mn_major) {
            // kind::tf32 takes K-major operands only: a pre-pass rewrites the
            // stored K x MN matrix as MN x K.  From here on rows/cols/mn_major
            // describe the rewritten copy the kernel reads.
            o->transpose = true;
            o->pack = true;
            o->mn_major = false;
            const int64_t k = o->rows;
            o->rows = o->cols;
            o->cols = k;
            o->packed_ld = round_up(k, 16 / esize);
        }
    }
    pl.pub.transpose_ab = ((swap ? pl.b.transpose : pl.a.transpose) ? 1 : 0) |
                          ((swap ? pl.a.transpose : pl.b.transpose) ? 2 : 0);
    pl.pub.a_mn_major = pl.a.mn_major;
    pl.pub.b_mn_major = pl.b.mn_major;
    pl.pub.pack_a = (swap ? pl.b.pack : pl.a.pack) ? 1 : 0;
    pl.pub.pack_b = (swap ? pl.a.pack : pl.b.pack) ? 1 : 0;
    pl.pack_a_bytes = pl.a.pack ? pl.a.rows * pl.a.packed_ld * esize : 0;
    pl.pack_b_bytes = pl.b.pack ? pl.b.rows * pl.b.packed_ld * esize : 0;
    pl.pub.c_vector = (!swap && aligned16(C) && (ldc * (int64_t)out_elem_bytes(dt.c)) % 16 == 0) ? 1 : 0;

    // Two K chunks per stage halve the TMA operations per MMA (the TMA unit
    // completes about one box per 160 ns per SM, nearly independent of the
    // box's size).  A K-major operand is then read through a 3-D view
    // (chunk, rows, chunk index) whose chunks must not run past K: one chunk
    // per stage unless K is a whole number of chunks.  The choice is final
    // once the tile width is known (below: at least 3 stages must fit).
    const bool kc2_ok = max_kc >= 2 && !((!pl.a.mn_major || !pl.b.mn_major) && K % chunk_k != 0);
    const int64_t k_chunks = ceil_div(K, chunk_k);
    // Tile shape.  Enough 256 x 256 tiles to give every SM pair one: CTA-pair
    // tiles (tcgen05 cta_group::2).  Otherwise single-CTA 128-row tiles, 256
    // columns wide when that still fills the GPU, else narrower ones with
    // stream-K over K for more parallelism (on CTA pairs for 256-wide tiles).
    //
    // Wave quantisation: when the last wave of a data-parallel schedule would
    // leave more than kMinWaveFill of the SMs idle and each tile is long in K,
    // single-CTA stream-K over the widest tiles balances the work instead
    // (the fix-up of a split tile costs one FP32 tile through L2, small beside
    // a K loop of kLongK or more k-blocks).
    // (LayerNorm needs each tile's rows complete in one CTA: no stream-K)
    // (allow_sk = false: data-parallel only, for callers with bounded scratch)
    // 256-row single-CTA tiles (two M = 128 halves sharing each B tile) for
    // N <= 128 when asked (convolutions): twice the MMA per A box of a
    // 128-row tile; data-parallel, plain epilogue, 16-bit inputs.
    const bool use_mh2 = mh2 && !swap && !ln && esize == 2 && pl.Nk <= 128 && pl.Mk > kBlockM;
    const bool long_k = allow_sk && !use_mh2 && !swap && !ln && k_chunks >= kLongK;
    auto wave_fill = [](int64_t tiles, int64_t units) {
        return static_cast<double>(tiles) / static_cast<double>(ceil_div(tiles, units) * units);
    };
    const int64_t pair_tiles = ceil_div(pl.Mk, 2 * kBlockM) * ceil_div(pl.Nk, 256);
    bool pairs = !use_mh2 && !swap && pl.Mk >= 2 * kBlockM && pl.Nk >= 256 && num_sms >= 2 &&
                 pair_tiles >= num_sms / 2;
    if (ln && pl.Nk <= 128) pairs = false;
    bool balance_sk = false;
    if (pairs && long_k && wave_fill(pair_tiles, num_sms / 2) < kMinWaveFill) {
        pairs = false;
        balance_sk = true;
    }
    int cg = pairs ? 2 : 1;
    pl.mh = use_mh2 ? 2 : 1;
    int64_t block_m = static_cast<int64_t>(kBlockM) * cg * pl.mh;
    int64_t tiles_m = ceil_div(pl.Mk, block_m);
    // Single-CTA tiles: the widest of 256 / 128 / 64 columns that still gives
    // every SM a tile (256) or at least half a wave (128, 64).
    int bn;
    const int64_t half_wave = (num_sms + 1) / 2;
    if (pairs || (pl.Nk > 128 && tiles_m * ceil_div(pl.Nk, 256) >= num_sms)) {
        bn = 256;
    } else if (pl.Nk > 64 && tiles_m * ceil_div(pl.Nk, 128) >= half_wave) {
        bn = 128;
    } else if (pl.Nk > 64 && tiles_m * ceil_div(pl.Nk, 64) < half_wave) {
        bn = 128;                           // too few tiles either way: stream-K below
    } else {
        bn = 64;
    }
    if (use_mh2) bn = pl.Nk <= 64 ? 64 : 128;
    if (ln) {
        // LayerNorm kernels come in widths 128 and 256: a row of up to 256
        // columns is whole in one tile
        if (pl.Nk <= 256) bn = (pl.Nk <= 128 && !pairs) ? 128 : 256;
        else if (bn < 128) bn = 128;
        pl.ln_fused = (pl.Nk <= bn);
    }
    if (!pairs && long_k) {
        const int64_t t = tiles_m * ceil_div(pl.Nk, bn);
        if (t >= half_wave && wave_fill(t, num_sms) < kMinWaveFill) balance_sk = true;
        if (balance_sk) {
            bn = pl.Nk > 128 ? 256 : (pl.Nk > 64 ? 128 : 64);
            if (tiles_m * ceil_div(pl.Nk, bn) > kMaxCounterTiles) balance_sk = false;
        }
    }
    // Stream-K over single-CTA 256-wide tiles (below) runs on CTA pairs
    // instead when M allows: per MMA a pair tile loads two thirds of the
    // operand bytes of a single-CTA 128 x 256 tile, and that is the limit
    // once the operands come from L2 (each re-read by several tiles).
    bool pair_sk = false;
    if (!use_mh2 && !pairs && !ln && !swap && bn == 256 && pl.Mk >= 2 * kBlockM && num_sms >= 2) {
        const int64_t t1 = tiles_m * ceil_div(pl.Nk, bn);
        // one counter per tile and CTA of the pair
        const bool fits = pair_tiles * 2 <= kMaxCounterTiles;
        if (fits && t1 <= kMaxCounterTiles && (balance_sk || (t1 < half_wave && long_k))) {
            pair_sk = pairs = true;
            cg = 2;
            block_m = 2 * kBlockM;
            tiles_m = ceil_div(pl.Mk, block_m);
        }
    }
    const int64_t tiles_n = ceil_div(pl.Nk, bn);
    const int64_t tiles = tiles_m * tiles_n;
    pl.cta_group = cg;
    pl.tiles_m = static_cast<int32_t>(tiles_m);
    pl.tiles_n = static_cast<int32_t>(tiles_n);
    pl.pub.block_m = static_cast<int32_t>(block_m);
    pl.pub.block_n = bn;
    pl.pub.num_tiles = static_cast<int32_t>(tiles);

    const uint32_t chunk_bytes = kATileBytes * static_cast<uint32_t>(pl.mh) +
                                 static_cast<uint32_t>(bn / cg) * 128u;
    const int64_t barrier_bytes = 256;
    // static shared memory of the kernel: flags, and the LayerNorm exchange
    const int64_t static_bytes = 64 + (ln ? 4 * kBlockM * 4 : 4);
    // C may be stored by TMA from a 32 KB staging area (decided below, with
    // the schedule): 128-row boxes of 128 bytes, full lines and one store per
    // box, where per-thread row stores each write 16 bytes of 32 different
    // lines.  The K chunks per stage are chosen with the staging set aside;
    // without it the stages are counted again (shared memory the kernel does
    // not use is left to the L1 cache).
    const bool c_stage_ok = pl.pub.c_vector && !ln && !use_mh2;
    const int64_t avail_all = smem_optin - 1024 - barrier_bytes - static_bytes;
    const int64_t avail = avail_all - (c_stage_ok ? kCStageBytes : 0);
    pl.kc = (kc2_ok && avail / (2 * static_cast<int64_t>(chunk_bytes)) >= min_kc2_stages) ? 2 : 1;
    const int64_t block_k = chunk_k * pl.kc;
    pl.k_blocks = static_cast<int32_t>(ceil_div(K, block_k));
    pl.pub.block_k = static_cast<int32_t>(block_k);
    const uint32_t stage_bytes = static_cast<uint32_t>(pl.kc) * chunk_bytes;
    int64_t stages = avail / stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return GEMM_ERR_NOT_SUPPORTED;
    pl.pub.stages = static_cast<int32_t>(stages);
    pl.smem_bytes = static_cast<size_t>(stages * stage_bytes + 1024 + barrier_bytes);

    const int64_t work = tiles * pl.k_blocks;
    // Stream-K spreads the K loop of too few tiles (or of a badly filled last
    // wave, above) over all SMs.  It pays for itself only when the tiles are
    // long in K; the swapped skinny path (a weight-streaming GEMM) always uses it.
    const bool stream_k = allow_sk && !use_mh2 && work < INT32_MAX &&
                          (pair_sk || (!pairs && !ln && (tiles <= kMaxCounterTiles) &&
                                       (balance_sk || ((tiles < num_sms) &&
                                        (swap ? k_chunks >= 4 : (tiles < half_wave && long_k))))));
    if (stream_k) {
        int64_t units = num_sms / cg;                  // CTAs or CTA pairs
        if (max_sk_units > 0 && units > max_sk_units) units = max_sk_units;
        int64_t G = units < work ? units : work;
        int64_t L = ceil_div(work, G);
        if (!swap) {
            // A tile split s ways saves (1 - 1/s) of its K loop and costs its
            // finisher s - 1 partial tiles read back through L2, each about
            // `fixup` k-blocks of MMA time: beyond sqrt(k_blocks / fixup) ways a
            // split costs more than it saves, and the ranges stay at least
            // k_blocks / that long.
            const double fixup = kSkFixupKBlocks * 256.0 / static_cast<double>(block_k * esize);
            int64_t s_max = static_cast<int64_t>(
                std::floor(std::sqrt(static_cast<double>(pl.k_blocks) / fixup)));
            if (s_max < 1) s_max = 1;
            const int64_t l_min = ceil_div(pl.k_blocks, s_max);
            if (L < l_min) L = l_min;
        }
        G = ceil_div(work, L);
        pl.sk_len = static_cast<int32_t>(L);
        pl.sk_max_seg = static_cast<int32_t>((L + pl.k_blocks - 2) / pl.k_blocks + 1);
        pl.pub.grid = static_cast<int32_t>(G * cg);
        pl.pub.split_k = static_cast<int32_t>(ceil_div(pl.k_blocks, L));
        pl.partial_bytes = G * pl.sk_max_seg * block_m * bn * 4;
    } else {
        const int64_t units = num_sms / cg;
        pl.pub.grid = static_cast<int32_t>(cg * (tiles < units ? tiles : units));
    }
    // TMA stores of C pay off where a tile's stores overlap later tiles'
    // mainloops (data-parallel, two or more tiles per CTA or pair) and for
    // FP32 C (a chunk is 32 rows of 128 bytes) once K is long enough (2048)
    // that the steps' latency after a lone or last tile is small beside its
    // mainloop; with a residual (beta != 0) the reads of C come first and the
    // steps' barriers serialise them: row stores there.
    pl.c_tma = c_stage_ok && beta == 0.0f &&
               ((dt.c == GEMM_F32 && K >= 2048) || (!stream_k && tiles >= 2 * (num_sms / cg)));
    pl.pub.c_tma = pl.c_tma ? 1 : 0;
    if (pl.c_tma) {
        pl.smem_bytes += kCStageBytes;
    } else if (c_stage_ok) {
        int64_t s_all = avail_all / stage_bytes;
        if (s_all > kMaxStages) s_all = kMaxStages;
        pl.pub.stages = static_cast<int32_t>(s_all);
        pl.smem_bytes = static_cast<size_t>(s_all * stage_bytes + 1024 + barrier_bytes);
    }
    pl.pub.path = swap ? GEMM_PATH_SKINNY : (pairs ? GEMM_PATH_TILED_2SM : GEMM_PATH_TILED_1SM);
    pl.pub.sk_len = pl.sk_len;
    pl.pub.sk_max_seg = pl.sk_max_seg;
    pl.pub.k_blocks = pl.k_blocks;
    pl.pub.tiles_m = pl.tiles_m;
    pl.pub.tiles_n = pl.tiles_n;
    if (ln && !pl.ln_fused) pl.ln_stats_bytes = pl.Mk * tiles_n * 8;
    const int64_t body = round_up(pl.pack_a_bytes, 256) + round_up(pl.pack_b_bytes, 256) +
                         round_up(pl.partial_bytes, 256) + round_up(pl.ln_stats_bytes, 256);
    pl.pub.workspace_bytes = body > 0 ? kWsHeaderBytes + body : 0;
    return GEMM_OK;
}

// Raster of a data-parallel GEMM schedule: groups of g tile-columns, each
// visited row by row, so the tiles of one wave (consecutive tiles) cover a
// few tile-rows across the group's g columns.  The group's g column strips of
// B (g x block_n rows, each K long) are reused by every tile of the group and
// stay in L2, while each row strip of A serves the g tiles of its row in one
// wave and comes back once per group.  g = 16 columns, fewer where their
// strips would pass kRasterResidentBytes.  (The pages' advice to reuse tiles
// through fast memory, applied to L2: CATLASS page, section 2.2; SGEMM page,
// section 1.2.)  Chosen by measurement on GB300 over groups of 4-16
// tile-rows or tile-columns, either L2 policy for the streamed operand and
// either K direction: see the tuning log.
int32_t raster_columns(int64_t tiles_n, int64_t b_strip_bytes) {
    int64_t g = b_strip_bytes > 0 ? kRasterResidentBytes / b_strip_bytes : kRasterMaxColumns;
    if (g > kRasterMaxColumns) g = kRasterMaxColumns;
    if (g > tiles_n) g = tiles_n;
    if (g < 1) g = 1;
    return static_cast<int32_t>(g);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                   cuuint32_t, cuuint32_t, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A forward 2-D convolution seen as a GEMM (M = N*P*Q output pixels, N = K
// output channels, the reduction over filter taps x channels).
struct ConvDesc {
    int64_t N, H, W, C, K, R, S, P, Q;
    int64_t pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
    const void* X;
    const void* Wt;
    EncodeIm2colFn encode_im2col;
};

}  // namespace

struct gemm_ctx {
    uint32_t debug_flags;     // test hook (gemm_debug_set)
    uint64_t wait_limit_ns;   // 0: the default bound
    int device;
    int num_sms;
    int smem_optin;
    int* err_host;        // mapped pinned error word (host view)
    int* err_dev;         // device view of the same word
    void* ws;             // device workspace
    size_t ws_bytes;
    EncodeTiledFn encode;
    EncodeIm2colFn encode_im2col;
};

namespace {

// Tiled map over a stored matrix (row pitch ld elements), 128-byte swizzle,
// zero fill out of range.  FP32 is moved as plain FP32: the tensor core itself
// takes it as TF32.
//  * chunks == 1: 2-D, dims {inner, outer}, a box of one 128-byte row (64
//    16-bit or 32 FP32 elements) by box_outer rows.
//  * chunks > 1 (K-major operands, inner a whole number of 128-byte chunks):
//    3-D, dims {chunk, outer, inner / chunk} with the chunk index striding 128
//    bytes along the row, a box of `chunks` chunks of box_outer rows -- in
//    shared memory one swizzled box_outer x 128-byte tile per chunk, back to
//    back.
bool encode_operand(EncodeTiledFn encode, CUtensorMap* map, int32_t dtype, const void* ptr,
                    int64_t inner, int64_t outer, int64_t ld, uint32_t box_outer,
                    int32_t chunks = 1) {
    const int64_t es = in_elem_bytes(dtype);
    const int64_t chunk = 128 / es;
    const CUtensorMapDataType ty = dtype == GEMM_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r;
    if (chunks == 1) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(chunk), box_outer};
        const cuuint32_t estr[2] = {1, 1};
        r = encode(map, ty, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        if (inner % chunk != 0) return false;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(chunk), static_cast<cuuint64_t>(outer),
                                    static_cast<cuuint64_t>(inner / chunk)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es), 128u};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk), box_outer,
                                   static_cast<cuuint32_t>(chunks)};
        const cuuint32_t estr[3] = {1, 1, 1};
        r = encode(map, ty, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// C (rows x cols, row pitch ld elements) for the epilogue's TMA stores:
// boxes of 128 bytes of a row (64 16-bit or 32 FP32 elements) by 128 rows,
// 128-byte swizzle; the parts of a box outside C are not written.
bool encode_c_store(EncodeTiledFn encode, CUtensorMap* map, int32_t dtype, const void* ptr,
                    int64_t cols, int64_t rows, int64_t ld) {
    const int64_t es = out_elem_bytes(dtype);
    const CUtensorMapDataType ty = dtype == GEMM_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(kBlockM)};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, ty, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The input X (N, H, W, C) as an im2col map: windows traversed W, H, N with
// the convolution's stride, 64 channels x 128 windows per load, 128-byte
// swizzle, zeros outside the image.  The box corners make the traversal
// visit exactly the windows of the output (P x Q per image); `pixels` windows
// (the tile's rows) per load.
bool encode_conv_input(const ConvDesc& cd, CUtensorMap* map, int32_t dtype, uint32_t pixels) {
    const int64_t es = 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cd.C), static_cast<cuuint64_t>(cd.W),
                                static_cast<cuuint64_t>(cd.H), static_cast<cuuint64_t>(cd.N)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(cd.C * es),
                                   static_cast<cuuint64_t>(cd.W * cd.C * es),
                                   static_cast<cuuint64_t>(cd.H * cd.W * cd.C * es)};
    const int lower[2] = {static_cast<int>(-cd.pad_w), static_cast<int>(-cd.pad_h)};
    const int upper[2] = {static_cast<int>(cd.pad_w - (cd.S - 1) * cd.dil_w),
                          static_cast<int>(cd.pad_h - (cd.R - 1) * cd.dil_h)};
    const cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(cd.stride_w),
                                static_cast<cuuint32_t>(cd.stride_h), 1};
    CUresult r = cd.encode_im2col(map,
                                  dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                  4, const_cast<void*>(cd.X), dims, strides, lower, upper,
                                  64u /* channels per 128-byte row */, pixels, estr,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The input X (N, H, W, C) as a tiled 4-D map (C, W, H, N) for whole-row
// convolution tiles: a box is 64 channels x `pixels` pixels x `rows` image
// rows of one image (stride 1), in shared memory rows x pixels rows of 128
// bytes in the 128-byte swizzle -- the K-major A tile the MMA reads;
// positions outside the image (the padding, or a window past the last row
// or column) read zeros.
bool encode_conv_rows(EncodeTiledFn encode, const ConvDesc& cd, CUtensorMap* map, int32_t dtype,
                      uint32_t rows, uint32_t pixels) {
    const int64_t es = 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cd.C), static_cast<cuuint64_t>(cd.W),
                                static_cast<cuuint64_t>(cd.H), static_cast<cuuint64_t>(cd.N)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(cd.C * es),
                                   static_cast<cuuint64_t>(cd.W * cd.C * es),
                                   static_cast<cuuint64_t>(cd.H * cd.W * cd.C * es)};
    const cuuint32_t box[4] = {64u, pixels, rows, 1u};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode(map,
                  dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(cd.X), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The filter (K, R, S, C) as a 3-D map (C, R*S, K): a box is 64 channels of
// one tap for box_rows output channels; channels past C read zeros.
bool encode_conv_filter(EncodeTiledFn encode, const ConvDesc& cd, CUtensorMap* map,
                        int32_t dtype, uint32_t box_rows) {
    const int64_t es = 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cd.C),
                                static_cast<cuuint64_t>(cd.R * cd.S),
                                static_cast<cuuint64_t>(cd.K)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cd.C * es),
                                   static_cast<cuuint64_t>(cd.R * cd.S * cd.C * es)};
    const cuuint32_t box[3] = {64, 1, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map,
                        dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(cd.Wt), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

gemm_status_t ensure_workspace(gemm_ctx* h, size_t bytes) {
    if (bytes <= h->ws_bytes) return GEMM_OK;
    if (h->ws) {
        cudaFree(h->ws);          // implicit device synchronisation: no user of the old buffer remains
        h->ws = nullptr;
        h->ws_bytes = 0;
    }
    size_t want = bytes + (bytes >> 2);
    if (cudaMalloc(&h->ws, want) != cudaSuccess) {
        cudaGetLastError();
        h->ws = nullptr;
        return GEMM_ERR_ALLOC;
    }
    // The stream-K tile counters must start at zero; every call leaves them
    // at zero again.
    if (cudaMemset(h->ws, 0, kWsHeaderBytes) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->ws);
        h->ws = nullptr;
        return GEMM_ERR_ALLOC;
    }
    h->ws_bytes = want;
    return GEMM_OK;
}

gemm_status_t take_device_error(gemm_ctx* h) {
    volatile int* e = h->err_host;
    if (*e != 0) {
        // A kernel that gave up may have left stream-K tile counters
        // half-counted: clear them before the handle is used again.
        cudaDeviceSynchronize();
        if (h->ws) cudaMemset(h->ws, 0, kWsHeaderBytes);
        cudaGetLastError();
        *e = 0;
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

int grid_for(int64_t elems_per_thread_unit, int num_sms) {
    int64_t blocks = ceil_div(elems_per_thread_unit, 256);
    int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}


// The LayerNorm row pass over C (M x N, row pitch ldc): from per-tile
// statistics, or (stats == nullptr) computing them.
template <typename OutT>
void launch_ln_rows(int64_t M, int64_t N, OutT* C, int64_t ldc, const float2* stats,
                    int32_t tiles_n, int32_t block_n, const gemm_layernorm_t* ln, int32_t ldt,
                    int num_sms, cudaStream_t stream) {
    if (stats != nullptr) {
        const int64_t want = static_cast<int64_t>(num_sms) * 8;   // resident CTAs
        const int grid = static_cast<int>(M < want ? M : want);
        ln_rows_stats_kernel<OutT><<<grid, kLnRowThreads, 0, stream>>>(C, ldc, M, N, stats, tiles_n,
                                                             block_n, ln->gamma, ln->shift, ldt,
                                                             ln->eps);
    } else {
        const int64_t want = static_cast<int64_t>(num_sms) * 8;
        const int grid = static_cast<int>(M < want ? M : want);
        ln_rows_kernel<OutT><<<grid, 256, 0, stream>>>(C, ldc, M, N, ln->gamma, ln->shift, ldt,
                                                       ln->eps);
    }
}

gemm_status_t enqueue_ln_rows(int64_t M, int64_t N, void* C, int64_t ldc, gemm_dtypes_t dt,
                              const float2* stats, int32_t tiles_n, int32_t block_n,
                              const gemm_layernorm_t* ln, int num_sms, cudaStream_t stream) {
    const int32_t ldt = (ln->gamma || ln->shift) ? ln->ln_dtype : GEMM_F32;
    if (dt.c == GEMM_F32)
        launch_ln_rows(M, N, static_cast<float*>(C), ldc, stats, tiles_n, block_n, ln, ldt,
                       num_sms, stream);
    else if (dt.c == GEMM_F16)
        launch_ln_rows(M, N, static_cast<__half*>(C), ldc, stats, tiles_n, block_n, ln, ldt,
                       num_sms, stream);
    else
        launch_ln_rows(M, N, static_cast<__nv_bfloat16*>(C), ldc, stats, tiles_n, block_n, ln,
                       ldt, num_sms, stream);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// Everything gemm_run enqueues after planning: the optional pack pre-passes,
// the TMA descriptors and the GEMM kernel.  `ws` is the workspace laid out as
// [tile counters (4 KB)][packed A][packed B][partial slots]; with
// clear_counters the counters are zeroed on the stream first.
gemm_status_t enqueue_plan(const Plan& pl, EncodeTiledFn encode, int num_sms, uint8_t* ws,
                           int* err_dev, float alpha, float beta, void* C, gemm_dtypes_t dt,
                           cudaStream_t stream, bool clear_counters, uint32_t debug_flags = 0,
                           uint64_t wait_limit_ns = 0, const gemm_epilogue_t* ep = nullptr,
                           const ConvDesc* conv = nullptr, const gemm_layernorm_t* ln = nullptr) {
    // kind::tf32 reads K-major operands only; the planner transposes the rest.
    if (pl.esize == 4 && (pl.a.mn_major || pl.b.mn_major)) return GEMM_ERR_NOT_SUPPORTED;
    int* counters = reinterpret_cast<int*>(ws);
    if (clear_counters && pl.sk_len > 0 &&
        cudaMemsetAsync(counters, 0, kWsHeaderBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    uint8_t* ws_a = ws + kWsHeaderBytes;
    uint8_t* ws_b = ws_a + round_up(pl.pack_a_bytes, 256);
    float* ws_part = reinterpret_cast<float*>(ws_b + round_up(pl.pack_b_bytes, 256));
    float2* ws_stats = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws_part) +
                                                 round_up(pl.partial_bytes, 256));

    // Pack operands whose rows TMA cannot address (pitch or base not 16-byte aligned).
    const void* a_ptr = pl.a.ptr;
    const void* b_ptr = pl.b.ptr;
    auto pack = [&](const OperandDesc& o, uint8_t* dst) {
        if (o.transpose) {
            // source: o.cols (K) rows of o.rows (MN) elements, pitch o.ld
            const int64_t tiles = ceil_div(o.rows, 32) * ceil_div(o.cols, 32);
            const int64_t cap = static_cast<int64_t>(num_sms) * 8;
            const int grid = static_cast<int>(tiles < cap ? tiles : cap);
            transpose_rows_kernel<<<grid, 256, 0, stream>>>(
                static_cast<const uint32_t*>(o.ptr), o.ld, o.cols, o.rows,
                reinterpret_cast<uint32_t*>(dst), o.packed_ld);
            return;
        }
        const int grid = grid_for(o.rows * o.packed_ld * pl.esize / 16, num_sms);
        if (pl.esize == 4)
            pack_rows_kernel<uint32_t><<<grid, 256, 0, stream>>>(
                static_cast<const uint32_t*>(o.ptr), o.ld, o.rows, o.cols,
                reinterpret_cast<uint32_t*>(dst), o.packed_ld);
        else
            pack_rows_kernel<uint16_t><<<grid, 256, 0, stream>>>(
                static_cast<const uint16_t*>(o.ptr), o.ld, o.rows, o.cols,
                reinterpret_cast<uint16_t*>(dst), o.packed_ld);
    };
    if (pl.a.pack) {
        pack(pl.a, ws_a);
        a_ptr = ws_a;
    }
    if (pl.b.pack) {
        pack(pl.b, ws_b);
        b_ptr = ws_b;
    }
    if ((pl.a.pack || pl.b.pack) && cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;

    TcLaunch l;
    std::memset(&l, 0, sizeof l);
    const int bn = pl.pub.block_n;
    const int cg = pl.cta_group;
    // MN-major boxes are one 128-byte row of M/N by block_k rows of K;
    // K-major ones kc chunks of 128 bytes of K by the tile's rows.
    const uint32_t mn_box = static_cast<uint32_t>(pl.pub.block_k);
    bool ok;
    if (conv != nullptr && pl.conv_halo) {
        ok = encode_conv_rows(encode, *conv, &l.tmA, dt.a,
                              static_cast<uint32_t>(pl.conv_rows + (conv->R - 1) * conv->dil_h),
                              static_cast<uint32_t>(pl.conv_pitch));
        ok = ok && encode_conv_filter(encode, *conv, &l.tmB, dt.b, static_cast<uint32_t>(bn / cg));
    } else if (conv != nullptr && pl.conv_rows > 0) {
        ok = encode_conv_rows(encode, *conv, &l.tmA, dt.a, static_cast<uint32_t>(pl.conv_rows),
                              static_cast<uint32_t>(conv->Q));
        if (pl.kc == 1)
            ok = ok && encode_conv_filter(encode, *conv, &l.tmB, dt.b, static_cast<uint32_t>(bn / cg));
        else
            ok = ok && encode_operand(encode, &l.tmB, dt.b, conv->Wt, conv->R * conv->S * conv->C,
                                      conv->K, conv->R * conv->S * conv->C,
                                      static_cast<uint32_t>(bn / cg), pl.kc);
    } else if (conv != nullptr) {
        ok = encode_conv_input(*conv, &l.tmA, dt.a, static_cast<uint32_t>(kBlockM * pl.mh));
        if (pl.kc == 1)
            ok = ok && encode_conv_filter(encode, *conv, &l.tmB, dt.b, static_cast<uint32_t>(bn / cg));
        else
            ok = ok && encode_operand(encode, &l.tmB, dt.b, conv->Wt, conv->R * conv->S * conv->C,
                                      conv->K, conv->R * conv->S * conv->C,
                                      static_cast<uint32_t>(bn / cg), pl.kc);
    } else {
        ok = encode_operand(encode, &l.tmA, dt.a, a_ptr, pl.a.cols, pl.a.rows, pl.a.packed_ld,
                            pl.a.mn_major ? mn_box : static_cast<uint32_t>(kBlockM * pl.mh),
                            pl.a.mn_major ? 1 : pl.kc);
        ok = ok && encode_operand(encode, &l.tmB, dt.b, b_ptr, pl.b.cols, pl.b.rows,
                                  pl.b.packed_ld,
                                  pl.b.mn_major ? mn_box : static_cast<uint32_t>(bn / cg),
                                  pl.b.mn_major ? 1 : pl.kc);
    }
    if (!ok) return GEMM_ERR_LAUNCH;
    const bool c_tma = pl.c_tma && encode_c_store(encode, &l.tmC, dt.c, C, pl.Nk, pl.Mk, pl.c_rs);

    TcParams& p = l.p;
    p.M = static_cast<int32_t>(pl.Mk);
    p.N = static_cast<int32_t>(pl.Nk);
    p.k_blocks = pl.k_blocks;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.num_tiles = pl.pub.num_tiles;
    p.group = kGroupM;
    p.raster_n = 0;
    p.stages = pl.pub.stages;
    p.a_mn_major = pl.a.mn_major ? 1 : 0;
    p.b_mn_major = pl.b.mn_major ? 1 : 0;
    // A/B format field: 0 F16, 1 BF16 (kind::f16); 2 TF32 (kind::tf32).
    const uint32_t ab_format = dt.a == GEMM_F32 ? 2u : (dt.a == GEMM_BF16 ? 1u : 0u);
    p.idesc = instr_desc(ab_format, pl.a.mn_major, pl.b.mn_major,
                         static_cast<uint32_t>(kBlockM * cg), static_cast<uint32_t>(bn));
    p.stream_k = pl.sk_len > 0 ? 1 : 0;
    p.sk_len = pl.sk_len;
    p.sk_max_seg = pl.sk_max_seg;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.c_rs = pl.c_rs;
    p.c_cs = pl.c_cs;
    p.c_vector = pl.pub.c_vector;
    p.c_tma = c_tma ? 1 : 0;
    p.partials = pl.partial_bytes > 0 ? ws_part : nullptr;
    p.tile_counters = pl.partial_bytes > 0 ? counters : nullptr;
    p.err = err_dev;
    // In the swapped skinny path each tile of A' (the large operand) is read
    // by exactly one CTA while B' (the few rows of the original A) is re-read
    // by every CTA.  Likewise a GEMM with one tile column reads each row
    // panel of A once, and one with one tile row each column panel of B (a
    // convolution re-reads its input once per filter tap: never).  A smaller
    // operand read once stays evict-last: it fits in L2 beside the rest, and a
    // caller that runs the GEMM again on it finds it there.
    const bool a_big = pl.a.rows * pl.a.cols * pl.esize >= kStreamOnceBytes;
    const bool b_big = pl.b.rows * pl.b.cols * pl.esize >= kStreamOnceBytes;
    const bool a_once = pl.pub.swap_ab || (conv == nullptr && pl.tiles_n == 1 && a_big);
    const bool b_once = !pl.pub.swap_ab && conv == nullptr && pl.tiles_m == 1 && b_big;
    p.a_policy = a_once ? kL2EvictFirst : kL2EvictLast;
    p.b_policy = b_once ? kL2EvictFirst : kL2EvictLast;
    // Data-parallel GEMMs: groups of tile-columns (raster_columns); every
    // wave reverses the K direction of the last.
    p.serpentine = 0;
    if (conv == nullptr && p.stream_k == 0 && !pl.pub.swap_ab) {
        const int64_t kpad = static_cast<int64_t>(pl.k_blocks) * pl.pub.block_k * pl.esize;
        p.raster_n = 1;
        p.group = raster_columns(pl.tiles_n, static_cast<int64_t>(bn) * kpad);
        p.serpentine = kSerpentineK ? 1 : 0;
    }
    p.wait_limit_ns = wait_limit_ns ? wait_limit_ns : kWaitTimeoutNs;
    p.debug_flags = debug_flags;
    p.bias = ep ? ep->bias : nullptr;
    p.bias_dtype = (ep && ep->bias) ? ep->bias_dtype : GEMM_F32;
    p.bias_on_rows = pl.pub.swap_ab ? 1 : 0;      // swapped: C columns are D' rows
    p.act = ep ? ep->activation : GEMM_ACT_NONE;
    if (pl.ln) {
        l.epi = kEpiLayerNorm;
        p.bias = ln->bias;
        p.bias_dtype = ln->bias ? ln->bias_dtype : GEMM_F32;
        p.act = GEMM_ACT_NONE;
        p.ln_gamma = ln->gamma;
        p.ln_shift = ln->shift;
        p.ln_dtype = (ln->gamma || ln->shift) ? ln->ln_dtype : GEMM_F32;
        p.ln_eps = ln->eps;
        p.ln_fused = pl.ln_fused ? 1 : 0;
        p.ln_stats = pl.ln_fused ? nullptr : ws_stats;
    }
    if (conv != nullptr) {
        p.conv = 1;
        p.conv_cblocks = static_cast<int32_t>(ceil_div(conv->C, 64));
        p.conv_taps = static_cast<int32_t>(conv->R * conv->S);
        p.conv_S = static_cast<int32_t>(conv->S);
        p.conv_P = static_cast<int32_t>(conv->P);
        p.conv_Q = static_cast<int32_t>(conv->Q);
        p.conv_stride_h = static_cast<int32_t>(conv->stride_h);
        p.conv_stride_w = static_cast<int32_t>(conv->stride_w);
        p.conv_pad_h = static_cast<int32_t>(conv->pad_h);
        p.conv_pad_w = static_cast<int32_t>(conv->pad_w);
        p.conv_dil_h = static_cast<int32_t>(conv->dil_h);
        p.conv_dil_w = static_cast<int32_t>(conv->dil_w);
        if (pl.conv_rows > 0) {
            p.conv_tiled = pl.conv_halo ? 2 : 1;
            p.conv_rows = pl.conv_rows;
            p.conv_tpi = pl.conv_tpi;
            p.conv_pitch = pl.conv_pitch;
            p.conv_R = static_cast<int32_t>(conv->R);
            p.conv_a_bytes = pl.conv_halo ? pl.halo_box_bytes
                                          : static_cast<uint32_t>(conv->Q * pl.conv_rows * 128);
            p.halo_a_region = pl.halo_a_region;
            p.halo_stage_bytes = pl.halo_stage_bytes;
        }
    }
    l.grid = pl.pub.grid;
    l.cta_group = cg;
    l.block_n = bn;
    l.esize = pl.esize;
    l.kc = pl.kc;
    l.mh = pl.mh;
    l.smem_bytes = pl.smem_bytes;
    l.stream = stream;

    cudaError_t e;
    if (pl.esize == 4) {
        if (dt.c == GEMM_F32) e = launch_tc_tf32_f32(l);
        else if (dt.c == GEMM_F16) e = launch_tc_tf32_f16(l);
        else e = launch_tc_tf32_bf16(l);
    } else {
        if (dt.c == GEMM_F32) e = launch_tc_f32(l);
        else if (dt.c == GEMM_F16) e = launch_tc_f16(l);
        else e = launch_tc_bf16(l);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (pl.ln && !pl.ln_fused)
        return enqueue_ln_rows(pl.Mk, pl.Nk, C, pl.c_rs, dt, ws_stats, pl.tiles_n, bn, ln, num_sms,
                               stream);
    return GEMM_OK;
}

gemm_status_t enqueue_scale(int64_t M, int64_t N, void* C, int64_t ldc, float beta,
                            gemm_dtypes_t dt, int num_sms, cudaStream_t stream,
                            const gemm_epilogue_t* ep = nullptr) {
    const int grid = grid_for(M * N, num_sms);
    const void* bias = ep ? ep->bias : nullptr;
    const int32_t bdt = (ep && ep->bias) ? ep->bias_dtype : GEMM_F32;
    const int32_t act = ep ? ep->activation : GEMM_ACT_NONE;
    if (dt.c == GEMM_F32)
        scale_c_kernel<float><<<grid, 256, 0, stream>>>(static_cast<float*>(C), M, N, ldc, beta,
                                                        bias, bdt, act);
    else if (dt.c == GEMM_F16)
        scale_c_kernel<__half><<<grid, 256, 0, stream>>>(static_cast<__half*>(C), M, N, ldc, beta,
                                                         bias, bdt, act);
    else
        scale_c_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<__nv_bfloat16*>(C), M, N, ldc, beta, bias, bdt, act);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

int64_t conv_dim(int64_t in, int64_t pad, int64_t dil, int64_t f, int64_t stride) {
    const int64_t span = in + 2 * pad - dil * (f - 1) - 1;
    return span < 0 ? 0 : span / stride + 1;
}

// Checks a convolution and fills its descriptor; then the GEMM plan of
// M = N*P*Q by K with R*S*ceil(C/64) k-blocks (both operands K-major, never
// swapped: the im2col load fills the MMA's 128-row side).
gemm_status_t conv_plan(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                        int64_t S, int64_t pad_h, int64_t pad_w, int64_t stride_h,
                        int64_t stride_w, int64_t dil_h, int64_t dil_w, float alpha,
                        const void* X, const void* Wt, float beta, const void* Y,
                        gemm_dtypes_t dt, int32_t num_sms, int32_t smem_optin, ConvDesc& cd,
                        Plan& pl) {
    if (N < 0 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1) return GEMM_ERR_INVALID_VALUE;
    if (pad_h < 0 || pad_w < 0 || stride_h < 1 || stride_w < 1 || dil_h < 1 || dil_w < 1)
        return GEMM_ERR_INVALID_VALUE;
    if (dt.a != dt.b || (dt.a != GEMM_F16 && dt.a != GEMM_BF16)) return GEMM_ERR_INVALID_VALUE;
    if (dt.c != GEMM_F32 && dt.c != GEMM_F16 && dt.c != GEMM_BF16) return GEMM_ERR_INVALID_VALUE;
    if (N > INT32_MAX || H > INT32_MAX || W > INT32_MAX || C > INT32_MAX || K > INT32_MAX ||
        R > 65535 || S > 65535 || dil_h > 65535 || dil_w > 65535)
        return GEMM_ERR_INVALID_VALUE;
    const int64_t P = conv_dim(H, pad_h, dil_h, R, stride_h);
    const int64_t Q = conv_dim(W, pad_w, dil_w, S, stride_w);
    const int64_t M = N * P * Q;
    if (M > INT32_MAX) return GEMM_ERR_INVALID_VALUE;
    // limits of the im2col load: 16-byte pixel rows, traversal strides up to
    // 8, window corners in [-128, 127], 16-bit tap offsets
    const int64_t up_w = pad_w - (S - 1) * dil_w, up_h = pad_h - (R - 1) * dil_h;
    if (C % 8 != 0 || stride_h > 8 || stride_w > 8 || pad_h > 128 || pad_w > 128 ||
        up_w < -128 || up_w > 127 || up_h < -128 || up_h > 127 ||
        (R - 1) * dil_h > 65535 || (S - 1) * dil_w > 65535)
        return GEMM_ERR_NOT_SUPPORTED;
    cd = ConvDesc{N, H, W, C, K, R, S, P, Q, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w,
                  X, Wt, nullptr};
    if (M > 0 && alpha != 0.0f && (!aligned16(X) || !aligned16(Wt))) {
        if (X == nullptr || Wt == nullptr) return GEMM_ERR_INVALID_VALUE;
        return GEMM_ERR_NOT_SUPPORTED;
    }
    const int64_t kfake = R * S * ceil_div(C, 64) * 64;
    // Two chunks per stage take two im2col boxes (64 channels of one tap
    // each) and one filter box, when C is a whole number of 64-channel blocks
    // (the KRSC filter is then a K-major K x (R*S*C) matrix whose chunks never
    // straddle taps); otherwise one chunk.  Two such stages suffice here (the
    // single-CTA 256-wide tile): the im2col boxes re-read X from L2 (R*S
    // times) and the filter stays in L2, so one stage in flight covers the
    // load latency, where a GEMM streaming an operand from DRAM needs three.
    gemm_status_t st = make_plan('N', 'T', M, K, kfake, alpha, X, kfake, Wt, kfake, beta, Y, K,
                                 dt, num_sms, smem_optin, pl, false, false,
                                 C % 64 == 0 ? kMaxKc : 1, 2, true, 0, kConvTwoHalves);
    if (st != GEMM_OK || pl.pub.path != GEMM_PATH_TILED_1SM || pl.mh != 2) return st;
    // Stride 1 on 256-row tiles: a tile is T whole output rows of one image,
    // and A is loaded by tiled boxes of the input instead of im2col boxes.
    //  * Halo units (kConvHalo): the tile's rows sit at a pitch of Q rounded
    //    up to 8 pixels (T pitch <= 256); pipeline step = (filter column s,
    //    64-channel block): one box of T + (R - 1) dil_h image rows x pitch
    //    pixels at the column's shifted window, and the column's R filter
    //    taps; tap r's A starts r dil_h pitch rows into the box (a multiple of
    //    8 rows: the swizzle atoms line up).  Each input pixel is fetched once
    //    per filter column, not once per tap.
    //  * Otherwise one box per tap of T rows x Q pixels (pitch Q).
    // The images' rows are split evenly: tiles per image = ceil(P / Tmax),
    // T = ceil(P / that).
    if (kConvWholeRows && stride_h == 1 && stride_w == 1 && Q <= 256 && P > 0) {
        const int64_t pitch = kConvHalo ? round_up(Q, 8) : Q;
        const int64_t tmax = (kBlockM * 2) / pitch;
        const int64_t tpi = ceil_div(P, tmax);
        const int64_t T = ceil_div(P, tpi);
        const int64_t tiles_m = N * tpi;
        bool halo = kConvHalo && pitch <= 256 && T + (R - 1) * dil_h <= 256;
        uint32_t box = 0, a_region = 0, stage = 0;
        int64_t stages = 0;
        if (halo) {
            const int64_t rows = T + (R - 1) * dil_h;
            box = static_cast<uint32_t>(rows * pitch * 128);
            // the MMAs of the last tap read 256 rows from (R - 1) dil_h pitch
            // on: the A region covers them (rows past the box are junk that
            // feeds only masked output rows)
            const int64_t span = ((R - 1) * dil_h * pitch + 2 * kBlockM) * 128;
            a_region = static_cast<uint32_t>(round_up(box > span ? box : span, 1024));
            stage = a_region + static_cast<uint32_t>(R * pl.pub.block_n * 128);
            stages = (smem_optin - 1024 - 256 - 64 - 4) / stage;
            if (stages > kMaxStages) stages = kMaxStages;
            halo = stages >= 2;
        }
        if (tiles_m <= INT32_MAX / pl.tiles_n) {
            pl.conv_rows = static_cast<int32_t>(T);
            pl.conv_tpi = static_cast<int32_t>(tpi);
            pl.pub.conv_rows = pl.conv_rows;
            pl.tiles_m = static_cast<int32_t>(tiles_m);
            pl.pub.tiles_m = pl.tiles_m;
            pl.pub.num_tiles = static_cast<int32_t>(tiles_m * pl.tiles_n);
            const int64_t units = num_sms;
            pl.pub.grid = static_cast<int32_t>(pl.pub.num_tiles < units ? pl.pub.num_tiles : units);
            pl.conv_pitch = static_cast<int32_t>(halo ? pitch : Q);
            pl.pub.conv_pitch = pl.conv_pitch;
            if (halo) {
                pl.conv_halo = true;
                pl.halo_box_bytes = box;
                pl.halo_a_region = a_region;
                pl.halo_stage_bytes = stage;
                pl.k_blocks = static_cast<int32_t>(S * ceil_div(C, 64));
                pl.pub.k_blocks = pl.k_blocks;
                pl.pub.block_k = 64;
                pl.pub.stages = static_cast<int32_t>(stages);
                pl.smem_bytes = static_cast<size_t>(stages * stage + 1024 + 256);
            }
        }
    }
    return GEMM_OK;
}

bool dtype16or32(int32_t t) { return t == GEMM_F16 || t == GEMM_BF16 || t == GEMM_F32; }

bool layernorm_ok(const gemm_layernorm_t* ln) {
    if (ln == nullptr) return false;
    if (ln->bias != nullptr && !dtype16or32(ln->bias_dtype)) return false;
    if ((ln->gamma != nullptr || ln->shift != nullptr) && !dtype16or32(ln->ln_dtype)) return false;
    if (!(ln->eps > 0.0f) || !std::isfinite(ln->eps)) return false;
    return true;
}

bool epilogue_ok(const gemm_epilogue_t* ep) {
    if (ep == nullptr) return true;
    if (ep->activation < GEMM_ACT_NONE || ep->activation > GEMM_ACT_SILU) return false;
    if (ep->bias != nullptr && ep->bias_dtype != GEMM_F16 && ep->bias_dtype != GEMM_BF16 &&
        ep->bias_dtype != GEMM_F32)
        return false;
    return true;
}

}  // namespace

extern "C" {

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
        case GEMM_ERR_NOT_SUPPORTED: return "GEMM_ERR_NOT_SUPPORTED";
        case GEMM_ERR_ALLOC: return "GEMM_ERR_ALLOC";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

gemm_status_t gemm_check_args(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                              float beta, const void* C, int64_t ldc, gemm_dtypes_t dt) {
    return check_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt);
}

gemm_status_t gemm_plan_query(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                              float beta, const void* C, int64_t ldc, gemm_dtypes_t dt,
                              int32_t num_sms, int32_t smem_optin, gemm_plan_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
    Plan pl;
    gemm_status_t st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt,
                                 num_sms, smem_optin, pl);
    if (st != GEMM_OK) return st;
    *out = pl.pub;
    return GEMM_OK;
}

gemm_status_t gemm_create(gemm_handle_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    int major = 0, minor = 0, sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NOT_SUPPORTED;

    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    gemm_ctx* h = new (std::nothrow) gemm_ctx();
    if (h == nullptr) return GEMM_ERR_ALLOC;
    h->device = dev;
    h->num_sms = sms;
    h->smem_optin = smem;
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);
    void* fn2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn2, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn2 == nullptr) {
        cudaGetLastError();
        delete h;
        return GEMM_ERR_LAUNCH;
    }
    h->encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn2);
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->err_host), 64, cudaHostAllocMapped) !=
            cudaSuccess ||
        cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->err_dev), h->err_host, 0) !=
            cudaSuccess) {
        cudaGetLastError();
        if (h->err_host) cudaFreeHost(h->err_host);
        delete h;
        return GEMM_ERR_ALLOC;
    }
    *h->err_host = 0;
    *out = h;
    return GEMM_OK;
}

gemm_status_t gemm_debug_set(gemm_handle_t h, uint32_t flags, uint64_t wait_limit_ns) {
    if (h == nullptr || (flags & ~static_cast<uint32_t>(GEMM_DEBUG_SKIP_FIRST_LOAD)) != 0)
        return GEMM_ERR_INVALID_VALUE;
    h->debug_flags = flags;
    h->wait_limit_ns = wait_limit_ns;
    return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
    if (h == nullptr) return GEMM_OK;
    cudaDeviceSynchronize();
    if (h->ws) cudaFree(h->ws);
    if (h->err_host) cudaFreeHost(h->err_host);
    delete h;
    cudaGetLastError();
    return GEMM_OK;
}

gemm_status_t gemm_sync(gemm_handle_t h, gemm_stream_t stream) {
    if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    gemm_status_t st = take_device_error(h);
    if (st != GEMM_OK) return st;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

gemm_status_t gemm_run_ex(gemm_handle_t h, char transA, char transB, int64_t M, int64_t N,
                          int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                          int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtypes_t dt,
                          const gemm_epilogue_t* ep, gemm_stream_t stream_) {
    if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = take_device_error(h);
    if (st != GEMM_OK) return st;
    if (!epilogue_ok(ep)) return GEMM_ERR_INVALID_VALUE;
    Plan pl;
    st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt, h->num_sms,
                   h->smem_optin, pl);
    if (st != GEMM_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    if (pl.pub.path == GEMM_PATH_NOOP) return GEMM_OK;
    if (pl.pub.path == GEMM_PATH_SCALE)
        return enqueue_scale(M, N, C, ldc, beta, dt, h->num_sms, stream, ep);
    st = ensure_workspace(h, static_cast<size_t>(pl.pub.workspace_bytes));
    if (st != GEMM_OK) return st;
    return enqueue_plan(pl, h->encode, h->num_sms, static_cast<uint8_t*>(h->ws), h->err_dev, alpha,
                        beta, C, dt, stream, false, h->debug_flags, h->wait_limit_ns, ep);
}

gemm_status_t gemm_run(gemm_handle_t h, char transA, char transB, int64_t M, int64_t N, int64_t K,
                       float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                       float beta, void* C, int64_t ldc, gemm_dtypes_t dt, gemm_stream_t stream) {
    return gemm_run_ex(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt,
                       nullptr, stream);
}

gemm_status_t gemm_layernorm_plan_query(char transA, char transB, int64_t M, int64_t N, int64_t K,
                                        float alpha, const void* A, int64_t lda, const void* B,
                                        int64_t ldb, float beta, const void* C, int64_t ldc,
                                        gemm_dtypes_t dt, const gemm_layernorm_t* ln,
                                        int32_t num_sms, int32_t smem_optin, gemm_plan_t* out,
                                        int32_t* fused) {
    if (out == nullptr || !layernorm_ok(ln)) return GEMM_ERR_INVALID_VALUE;
    Plan pl;
    gemm_status_t st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt,
                                 num_sms, smem_optin, pl, false, true);
    if (st != GEMM_OK) return st;
    if (dt.a == GEMM_F32) return GEMM_ERR_NOT_SUPPORTED;
    *out = pl.pub;
    if (fused) *fused = pl.ln_fused ? 1 : 0;
    return GEMM_OK;
}

gemm_status_t gemm_run_layernorm(gemm_handle_t h, char transA, char transB, int64_t M, int64_t N,
                                 int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtypes_t dt,
                                 const gemm_layernorm_t* ln, gemm_stream_t stream_) {
    if (h == nullptr || !layernorm_ok(ln)) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = take_device_error(h);
    if (st != GEMM_OK) return st;
    Plan pl;
    st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt, h->num_sms,
                   h->smem_optin, pl, false, true);
    if (st != GEMM_OK) return st;
    if (dt.a == GEMM_F32) return GEMM_ERR_NOT_SUPPORTED;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (pl.pub.path == GEMM_PATH_NOOP) return GEMM_OK;
    if (pl.pub.path == GEMM_PATH_SCALE) {
        // h = beta * C + bias (rounded to C's type), then whole-row LayerNorm
        gemm_epilogue_t ep{ln->bias, ln->bias_dtype, GEMM_ACT_NONE};
        st = enqueue_scale(M, N, C, ldc, beta, dt, h->num_sms, stream, &ep);
        if (st != GEMM_OK) return st;
        return enqueue_ln_rows(M, N, C, ldc, dt, nullptr, 1, static_cast<int32_t>(N), ln,
                               h->num_sms, stream);
    }
    st = ensure_workspace(h, static_cast<size_t>(pl.pub.workspace_bytes));
    if (st != GEMM_OK) return st;
    return enqueue_plan(pl, h->encode, h->num_sms, static_cast<uint8_t*>(h->ws), h->err_dev, alpha,
                        beta, C, dt, stream, false, h->debug_flags, h->wait_limit_ns, nullptr,
                        nullptr, ln);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_run_noalloc: the same GEMM for callers that cannot allocate device
// memory.  Its scratch (packed operand copies and stream-K partial sums) lives
// in the file-scope array below instead of a handle's cudaMalloc'd workspace.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr int kNoAllocMaxDevices = 64;

// Scratch for gemm_run_noalloc.  Every GPU that loads this library holds it
// until the process exits.  In host code `g_noalloc_scratch` is only a
// stand-in symbol, never a device address: the device address comes from
// cudaGetSymbolAddress during the per-device set-up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

struct NoAllocDevice {
    std::mutex mu;
    bool ready;                // set-up succeeded (a failed one is retried by the next call)
    void* scratch;             // device address of g_noalloc_scratch on this device
    int num_sms, smem_optin;
    EncodeTiledFn encode;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Per-device set-up, with that device current; called under d.mu until it
// succeeds once.
gemm_status_t noalloc_setup(NoAllocDevice& d, int dev) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NOT_SUPPORTED;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    d.num_sms = sms;
    d.smem_optin = smem;
    d.encode = reinterpret_cast<EncodeTiledFn>(fn);
    d.scratch = ptr;
    d.ready = true;
    return GEMM_OK;
}

// gemm_run's plan, made to fit the static scratch: when its stream-K partial
// sums do not fit, the same problem is planned again with fewer stream-K
// units (CTAs or CTA pairs) -- every split tile's partial slots shrink with
// them -- and, failing that, data-parallel without stream-K.  Only when the
// packed operand copies alone exceed the scratch is the problem refused.
gemm_status_t noalloc_plan(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                           const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                           const void* C, int64_t ldc, gemm_dtypes_t dt, const NoAllocDevice& d,
                           Plan& pl) {
    const int64_t limit = static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_BYTES);
    gemm_status_t st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt,
                                 d.num_sms, d.smem_optin, pl);
    if (st != GEMM_OK || pl.pub.workspace_bytes <= limit) return st;
    int64_t units = pl.pub.grid / pl.cta_group;
    while (pl.partial_bytes > 0 && units > 1) {
        // the slots scale with the units (sk_max_seg grows by at most one
        // as the ranges lengthen): shrink in proportion, then step down
        const int64_t fixed = pl.pub.workspace_bytes - round_up(pl.partial_bytes, 256);
        const int64_t per_unit = pl.partial_bytes / units;
        int64_t fit = per_unit > 0 ? (limit - fixed) / per_unit : units - 1;
        if (fit >= units) fit = units - 1;
        if (fit < 1) break;
        units = fit;
        st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt,
                       d.num_sms, d.smem_optin, pl, true, false, kMaxKc, 3, true,
                       static_cast<int32_t>(units));
        if (st != GEMM_OK || pl.pub.workspace_bytes <= limit) return st;
        units = pl.pub.grid / pl.cta_group;
    }
    st = make_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt, d.num_sms,
                   d.smem_optin, pl, true, false, kMaxKc, 3, false);
    if (st != GEMM_OK) return st;
    // needs more scratch than the static array holds (packed operand copies)
    return pl.pub.workspace_bytes <= limit ? GEMM_OK : GEMM_ERR_INVALID_VALUE;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(char transA, char transB, int64_t M, int64_t N,
                                          int64_t K, float alpha, const void* A, int64_t lda,
                                          const void* B, int64_t ldb, float beta, void* C,
                                          int64_t ldc, gemm_dtypes_t dt, gemm_stream_t stream_) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GEMM_ERR_NOT_SUPPORTED;
    NoAllocDevice& d = g_noalloc_dev[dev];
    {
        std::lock_guard<std::mutex> lock(d.mu);
        if (!d.ready) {
            const gemm_status_t s0 = noalloc_setup(d, dev);
            if (s0 != GEMM_OK) return s0;
        }
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // The scratch address belongs to the current device: a stream of another
    // device would have the kernels use it there.  (The legacy and per-thread
    // default streams always belong to the current device.)
    if (stream != nullptr && stream != cudaStreamLegacy && stream != cudaStreamPerThread) {
        int sdev = -1;
        if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_INVALID_VALUE;
        }
        if (sdev != dev) return GEMM_ERR_INVALID_VALUE;
    }

    Plan pl;
    gemm_status_t st = noalloc_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                    dt, d, pl);
    if (st != GEMM_OK) return st;

    if (pl.pub.path == GEMM_PATH_NOOP) return GEMM_OK;
    if (pl.pub.path == GEMM_PATH_SCALE)
        return enqueue_scale(M, N, C, ldc, beta, dt, d.num_sms, stream);
    // The scratch takes the place of a handle's workspace.  Its stream-K tile
    // counters must start at zero, so they are cleared on the stream at the
    // start of every call that uses them; the packed copies and every
    // partial-sum slot are fully written before they are read within the
    // call.  No host-visible error word exists without an allocation, so
    // device timeouts are not reported.
    return enqueue_plan(pl, d.encode, d.num_sms, static_cast<uint8_t*>(d.scratch), nullptr, alpha,
                        beta, C, dt, stream, true);
}

extern "C" {

gemm_status_t conv2d_output_dims(int64_t H, int64_t W, int64_t R, int64_t S, int64_t pad_h,
                                 int64_t pad_w, int64_t stride_h, int64_t stride_w, int64_t dil_h,
                                 int64_t dil_w, int64_t* P, int64_t* Q) {
    if (P == nullptr || Q == nullptr || H < 1 || W < 1 || R < 1 || S < 1 || pad_h < 0 ||
        pad_w < 0 || stride_h < 1 || stride_w < 1 || dil_h < 1 || dil_w < 1)
        return GEMM_ERR_INVALID_VALUE;
    *P = conv_dim(H, pad_h, dil_h, R, stride_h);
    *Q = conv_dim(W, pad_w, dil_w, S, stride_w);
    return GEMM_OK;
}

gemm_status_t conv2d_plan_query(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                                int64_t S, int64_t pad_h, int64_t pad_w, int64_t stride_h,
                                int64_t stride_w, int64_t dil_h, int64_t dil_w, float alpha,
                                const void* X, const void* Wt, float beta, const void* Y,
                                gemm_dtypes_t dt, int32_t num_sms, int32_t smem_optin,
                                gemm_plan_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (num_sms < 1 || smem_optin < 64 * 1024) return GEMM_ERR_INVALID_VALUE;
    ConvDesc cd;
    Plan pl;
    gemm_status_t st = conv_plan(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, dil_h,
                                 dil_w, alpha, X, Wt, beta, Y, dt, num_sms, smem_optin, cd, pl);
    if (st == GEMM_OK) *out = pl.pub;
    return st;
}

gemm_status_t conv2d_fprop(gemm_handle_t h, int64_t N, int64_t H, int64_t W, int64_t C,
                           int64_t K, int64_t R, int64_t S, int64_t pad_h, int64_t pad_w,
                           int64_t stride_h, int64_t stride_w, int64_t dil_h, int64_t dil_w,
                           float alpha, const void* X, const void* Wt, float beta, void* Y,
                           gemm_dtypes_t dt, const gemm_epilogue_t* ep, gemm_stream_t stream_) {
    if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = take_device_error(h);
    if (st != GEMM_OK) return st;
    if (!epilogue_ok(ep)) return GEMM_ERR_INVALID_VALUE;
    ConvDesc cd;
    Plan pl;
    st = conv_plan(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, alpha, X,
                   Wt, beta, Y, dt, h->num_sms, h->smem_optin, cd, pl);
    if (st != GEMM_OK) return st;
    cd.encode_im2col = h->encode_im2col;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (pl.pub.path == GEMM_PATH_NOOP) return GEMM_OK;
    if (pl.pub.path == GEMM_PATH_SCALE)
        return enqueue_scale(cd.N * cd.P * cd.Q, K, Y, K, beta, dt, h->num_sms, stream, ep);
    st = ensure_workspace(h, static_cast<size_t>(pl.pub.workspace_bytes));
    if (st != GEMM_OK) return st;
    return enqueue_plan(pl, h->encode, h->num_sms, static_cast<uint8_t*>(h->ws), h->err_dev, alpha,
                        beta, Y, dt, stream, false, h->debug_flags, h->wait_limit_ns, ep, &cd);
}

}  // extern "C"
