// softmax.cu -- the C ABI of the row softmax (include/softmax_sm103.h):
// argument validation, the host planner that picks the work split, and the
// launch.
//
// The split follows the SGEMM tutorial page's two regimes (sections 2.3-2.4):
// a row that fits on chip is read once and kept there (registers of a warp or
// of a CTA, staged through shared memory); a longer row is read twice by one
// CTA -- a first pass folds it into a running (max, sum) by the online rule,
// a second writes y -- with the first pass's lines kept in L2, so that DRAM
// still sees the row once.  Only when the slices of all resident CTAs would
// not fit half the L2 is a row spread over a thread-block cluster whose CTAs
// merge their (max, sum) pairs through distributed shared memory (the page's
// option of splitting a long row over blocks that reduce across blocks).
// Measured on GB300: per-row cluster synchronisation cost more than the
// L2-resident second read (2048 x 65536 FP32: 298 us over a cluster of 4,
// 217 us in one CTA with two passes).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "softmax_sm103.h"
#include "softmax_launch.h"

namespace {

constexpr int64_t kWarpMaxCols = 32 * smx::kE;          // 1024
constexpr int64_t kCtaSmallCols = 256 * smx::kE;        // 8192: 256-thread CTAs
constexpr int64_t kCtaMaxCols = 512 * smx::kE;          // 16384 per CTA
constexpr int64_t kMaxCols = int64_t(1) << 30;
// Rows staged in shared memory by bulk copies: 256 B to 64 KB and at most
// 16 warps x 32 x kTmaMaxVec 16-byte vectors, one row per group of warps at a
// time (the group holds its row in registers, at most kTmaMaxVec vectors per
// thread), slots within this budget.
constexpr int64_t kStagedMinBytes = 256;
constexpr int64_t kStagedMaxBytes = 64 * 1024;
constexpr int64_t kStagedSmemBudget = 200 * 1024;
constexpr int64_t kStagedMinDepth = 6;
// Two-pass rows: the first pass's lines must still be in L2 when the second
// pass reads them, so the slices of all resident CTAs stay within half the
// 129 MB L2 of a GB300 (a cluster splits the row when one CTA per row would
// not).
constexpr int64_t kTwoPassL2Budget = int64_t(64) << 20;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
int64_t elem_bytes(int32_t dt) { return dt == GEMM_F32 ? 4 : 2; }
bool dtype_ok(int32_t dt) { return dt == GEMM_F16 || dt == GEMM_BF16 || dt == GEMM_F32; }
bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

struct Plan {
    softmax_plan_t pub;
    bool resident;
    size_t smem;          // staged path: dynamic shared memory per CTA
    int32_t bulk_elems;   // staged path: elements per row moved by the bulk copy
    int32_t row_stride;   // staged path: bytes between rows inside a slot
    int32_t contiguous;   // staged path: a slot's rows are adjacent in X (one copy)
    bool whole;           // staged path: rows fill the threads' vectors exactly, no tail
    bool long_rows;       // staged path: rows streamed twice in chunks
};

gemm_status_t check(int64_t rows, int64_t cols, const void* X, int64_t ldx, int32_t xdt,
                    const void* Y, int64_t ldy, int32_t ydt) {
    // 32-bit offsets within a row, with headroom for a chunk past its end
    if (rows < 0 || cols < 0 || cols > kMaxCols) return GEMM_ERR_INVALID_VALUE;
    if (!dtype_ok(xdt) || !dtype_ok(ydt)) return GEMM_ERR_INVALID_VALUE;
    const int64_t min_ld = cols > 1 ? cols : 1;
    if (ldx < min_ld || ldy < min_ld) return GEMM_ERR_INVALID_VALUE;
    if (rows == 0 || cols == 0) return GEMM_OK;
    if (X == nullptr || Y == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (!aligned_to(X, elem_bytes(xdt)) || !aligned_to(Y, elem_bytes(ydt)))
        return GEMM_ERR_INVALID_VALUE;
    // In place (the same matrix) is allowed; any other overlap is not.
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(X);
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(Y);
    const uintptr_t x1 = x0 + static_cast<uintptr_t>(((rows - 1) * ldx + cols) * elem_bytes(xdt));
    const uintptr_t y1 = y0 + static_cast<uintptr_t>(((rows - 1) * ldy + cols) * elem_bytes(ydt));
    const bool overlap = x0 < y1 && y0 < x1;
    const bool same = x0 == y0 && ldx == ldy && xdt == ydt;
    if (overlap && !same) return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

// ctas_per_sm <= 0: estimate from the shape (the launch path asks the
// occupancy calculator instead).
gemm_status_t make_plan(int64_t rows, int64_t cols, const void* X, int64_t ldx, int32_t xdt,
                        const void* Y, int64_t ldy, int32_t ydt, int32_t num_sms,
                        int32_t ctas_per_sm, Plan& pl) {
    gemm_status_t st = check(rows, cols, X, ldx, xdt, Y, ldy, ydt);
    if (st != GEMM_OK) return st;
    if (num_sms < 1) return GEMM_ERR_INVALID_VALUE;
    std::memset(&pl, 0, sizeof pl);
    pl.pub.cluster = 1;
    if (rows == 0 || cols == 0) {
        pl.pub.mode = SOFTMAX_MODE_NOOP;
        return GEMM_OK;
    }
    const int64_t ex = elem_bytes(xdt), ey = elem_bytes(ydt);
    pl.pub.vec = (aligned_to(X, 16) && aligned_to(Y, 16) && (ldx * ex) % 16 == 0 &&
                  (ldy * ey) % 16 == 0) ? 1 : 0;
    const int64_t row_bytes = cols * ex;
    const int64_t kvmax = smx::kTmaMaxVec;                   // vectors per thread
    const int64_t max_vec = smx::kTmaComputeWarps * 32 * kvmax;
    // a row fits one CTA's slots and registers
    const int64_t b = cols * ex;
    const bool staged = pl.pub.vec && b >= kStagedMinBytes && b <= kStagedMaxBytes &&
                        b / 16 <= max_vec;
    if (staged) {
        // staged in shared memory: one CTA of 16 warps per SM, split into
        // groups just large enough to hold a row in registers; each group a
        // pipeline of `depth` row slots
        const int64_t slice = cols;
        const int64_t nvec = slice * ex / 16;
        int64_t gw = 1, unit_rows = 1, row_stride = 0;
        bool contiguous = false;
        if (nvec <= 32 * kvmax) {
            // a warp holds a row: groups of 8 warps share slots of several
            // rows, moved by one copy of ~16 KB when the rows are adjacent
            gw = 8;
            contiguous = ldx * ex == row_bytes;
            row_stride = contiguous ? row_bytes : round_up(row_bytes, 16);
            int64_t k = 16384 / (gw * row_stride);
            k = k < 1 ? 1 : (k > 4 ? 4 : k);
            unit_rows = gw * k;
        } else {
            // the fewest warps that hold the row, doubled while a group
            // would get fewer than six slots: slots in flight beat
            // independent groups (16384 x 4096 FP32: 4 groups of 4 warps
            // with 3 slots 90.7 us, 2 groups of 8 with 6 slots 84.3 us)
            while (gw * 32 * kvmax < nvec) gw *= 2;
            while (gw < smx::kTmaComputeWarps &&
                   kStagedSmemBudget / ((smx::kTmaComputeWarps / gw) * round_up(slice * ex, 128)) <
                       kStagedMinDepth)
                gw *= 2;
        }
        // vectors per thread: the least power of two that covers the row
        const int64_t threads_per_row = unit_rows > 1 ? 32 : gw * 32;
        int64_t kv = 1;
        while (kv * threads_per_row < nvec) kv *= 2;
        const int64_t groups = smx::kTmaComputeWarps / gw;
        const int64_t slot = round_up(unit_rows == 1 ? slice * ex : unit_rows * row_stride, 128);
        int64_t depth = kStagedSmemBudget / (groups * slot);
        if (depth > smx::kTmaMaxDepth) depth = smx::kTmaMaxDepth;
        pl.pub.mode = unit_rows > 1 ? SOFTMAX_MODE_WARP : SOFTMAX_MODE_CTA;
        pl.pub.threads = smx::kTmaThreads;
        pl.pub.cluster = 1;
        pl.pub.slice = static_cast<int32_t>(round_up(slice, 8));
        pl.pub.depth = static_cast<int32_t>(depth);
        pl.pub.group_warps = static_cast<int32_t>(gw);
        pl.pub.unit_rows = static_cast<int32_t>(unit_rows);
        pl.pub.kv = static_cast<int32_t>(kv);
        pl.row_stride = static_cast<int32_t>(row_stride);
        pl.contiguous = contiguous ? 1 : 0;
        pl.resident = true;
        // a "full" and an "empty" barrier per slot, then the slots
        pl.smem = static_cast<size_t>(round_up(2 * groups * depth * 8, 128) + groups * depth * slot);
        pl.bulk_elems = static_cast<int32_t>((row_bytes / 16) * 16 / ex);
        // no 16-byte tail and every thread's kv vectors inside the row: the
        // kernel's variant without bounds checks
        pl.whole = pl.bulk_elems == cols && kv * threads_per_row * (16 / ex) == slice;
        const int64_t need = ceil_div(ceil_div(rows, unit_rows), groups);
        pl.pub.grid = static_cast<int32_t>(need < num_sms ? need : num_sms);
    } else if (cols <= kWarpMaxCols) {
        pl.pub.mode = SOFTMAX_MODE_WARP;
        pl.pub.threads = smx::kWarpCtaThreads;
        pl.pub.slice = static_cast<int32_t>(round_up(cols, 8));
        pl.resident = true;
        const int64_t per_sm = ctas_per_sm > 0 ? ctas_per_sm : 4;
        const int64_t need = ceil_div(rows, smx::kWarpCtaThreads / 32);
        const int64_t cap = per_sm * num_sms;
        pl.pub.grid = static_cast<int32_t>(need < cap ? need : cap);
    } else {
        int64_t cl = 1;
        int threads = cols <= kCtaSmallCols ? 256 : 512;
        if (cols > kCtaMaxCols) {
            // two passes: the smallest cluster whose resident slices fit the
            // L2 budget (one CTA per row unless the rows are very long)
            while (cl < smx::kMaxCluster &&
                   static_cast<int64_t>(num_sms) * ceil_div(cols, cl) * ex > kTwoPassL2Budget)
                cl *= 2;
        }
        if (pl.pub.vec && cols > kCtaMaxCols && cl <= smx::kMaxLongCluster) {
            // 16-byte aligned rows too long to stage whole: streamed twice
            // through shared memory in chunks by bulk copies
            // (softmax_long_kernel), each row split over a cluster of `cl`
            // CTAs when one CTA per row would overrun the L2 budget
            pl.pub.mode = SOFTMAX_MODE_STREAM;
            pl.pub.threads = smx::kTmaThreads;
            pl.pub.cluster = static_cast<int32_t>(cl);
            pl.pub.slice = static_cast<int32_t>(round_up(ceil_div(cols, cl), 8));
            pl.pub.depth = smx::kLongDepth;
            pl.pub.group_warps = smx::kTmaComputeWarps;
            pl.pub.unit_rows = 1;
            pl.pub.kv = smx::kLongKV;
            pl.long_rows = true;
            pl.resident = false;
            pl.smem = static_cast<size_t>(1024 + smx::kLongDepth * smx::kLongChunkBytes);
            pl.bulk_elems = static_cast<int32_t>((row_bytes / 16) * 16 / ex);
            // clusters resident at once: ctas_per_sm stands for them here
            // (the launch asks the occupancy calculator)
            int64_t groups = cl == 1 ? num_sms : (ctas_per_sm > 0 ? ctas_per_sm : num_sms / cl);
            if (groups < 1) groups = 1;
            pl.pub.grid = static_cast<int32_t>(cl * (rows < groups ? rows : groups));
            pl.pub.hbm_bytes = rows * cols * (2 * ex + ey);
            return GEMM_OK;
        }
        const int64_t slice = round_up(ceil_div(cols, cl), 8);
        pl.resident = slice <= static_cast<int64_t>(threads) * smx::kE;
        pl.pub.mode = pl.resident ? SOFTMAX_MODE_CTA : SOFTMAX_MODE_STREAM;
        pl.pub.threads = threads;
        pl.pub.cluster = static_cast<int32_t>(cl);
        pl.pub.slice = static_cast<int32_t>(slice);
        int64_t groups;
        if (cl == 1) {
            const int64_t per_sm = ctas_per_sm > 0 ? ctas_per_sm : (threads > 256 ? 1 : 2);
            groups = per_sm * num_sms;
        } else {
            // ctas_per_sm stands for resident clusters on the GPU here
            groups = ctas_per_sm > 0 ? ctas_per_sm : num_sms / cl;
            if (groups < 1) groups = 1;
        }
        pl.pub.grid = static_cast<int32_t>(cl * (rows < groups ? rows : groups));
    }
    pl.pub.hbm_bytes = rows * cols * (ex * (pl.resident ? 1 : 2) + ey);
    return GEMM_OK;
}

struct DeviceInfo {
    int sms = 0;
    bool sm103 = false;
};

bool device_info(DeviceInfo& out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool known[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> g(mu);
    if (!known[dev]) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        cache[dev].sms = sms;
        cache[dev].sm103 = (major == 10 && minor == 3);
        known[dev] = true;
    }
    out = cache[dev];
    return true;
}

cudaError_t launch(int32_t xdt, const smx::SoftmaxParams& p, int32_t ydt, bool warp_rows,
                   int threads, int grid, cudaStream_t s) {
    if (xdt == GEMM_F32) return smx::launch_softmax_f32(p, ydt, warp_rows, threads, grid, s);
    if (xdt == GEMM_F16) return smx::launch_softmax_f16(p, ydt, warp_rows, threads, grid, s);
    return smx::launch_softmax_bf16(p, ydt, warp_rows, threads, grid, s);
}

cudaError_t launch_tma(int32_t xdt, const smx::TmaSoftmaxParams& p, int32_t ydt, int grid,
                       size_t smem, cudaStream_t s) {
    if (xdt == GEMM_F32) return smx::launch_softmax_tma_f32(p, ydt, grid, smem, s);
    if (xdt == GEMM_F16) return smx::launch_softmax_tma_f16(p, ydt, grid, smem, s);
    return smx::launch_softmax_tma_bf16(p, ydt, grid, smem, s);
}

int resident(int32_t xdt, int32_t ydt, bool warp_rows, int threads, int cluster, int sms) {
    if (xdt == GEMM_F32) return smx::resident_groups_f32(ydt, warp_rows, threads, cluster, sms);
    if (xdt == GEMM_F16) return smx::resident_groups_f16(ydt, warp_rows, threads, cluster, sms);
    return smx::resident_groups_bf16(ydt, warp_rows, threads, cluster, sms);
}

// ------------------------------------------------------------------ errors

// The device error word the staged kernels set when a bounded wait runs out
// (one per device; its address is looked up with that device current).
__device__ int g_softmax_error;

std::mutex g_dbg_mu;
uint32_t g_debug_flags = 0;
uint64_t g_wait_limit_ns = 0;

int* error_word(int dev) {
    static std::mutex mu;
    static int* addr[64] = {};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return nullptr;
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_softmax_error) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev] = static_cast<int*>(p);
    }
    return addr[dev];
}

}  // namespace

extern "C" {

gemm_status_t softmax_plan_query(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                                 int32_t x_dtype, const void* Y, int64_t ldy, int32_t y_dtype,
                                 int32_t num_sms, int32_t ctas_per_sm, softmax_plan_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
    Plan pl;
    gemm_status_t st = make_plan(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, num_sms,
                                 ctas_per_sm, pl);
    if (st == GEMM_OK) *out = pl.pub;
    return st;
}

gemm_status_t softmax_rows(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                           int32_t x_dtype, void* Y, int64_t ldy, int32_t y_dtype,
                           gemm_stream_t stream) {
    gemm_status_t st = check(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype);
    if (st != GEMM_OK) return st;
    if (rows == 0 || cols == 0) return GEMM_OK;
    DeviceInfo dev;
    if (!device_info(dev)) return GEMM_ERR_LAUNCH;
    if (!dev.sm103) return GEMM_ERR_NOT_SUPPORTED;
    // the shape first (threads, cluster), then, for the register kernels, the
    // resident groups for it (the staged kernels run one CTA per SM; their
    // launch caps a cluster grid by the clusters that fit)
    Plan pl;
    st = make_plan(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, dev.sms, 0, pl);
    if (st != GEMM_OK) return st;
    const bool warp_rows = pl.pub.mode == SOFTMAX_MODE_WARP;
    if (pl.pub.depth == 0) {
        const int groups = resident(x_dtype, y_dtype, warp_rows, pl.pub.threads, pl.pub.cluster,
                                    dev.sms);
        const int per_sm_or_clusters = pl.pub.cluster > 1 ? groups : groups / dev.sms;
        st = make_plan(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, dev.sms,
                       per_sm_or_clusters > 0 ? per_sm_or_clusters : 1, pl);
        if (st != GEMM_OK) return st;
    }

    if (pl.pub.depth > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        int* err = error_word(dev);
        if (err == nullptr) return GEMM_ERR_LAUNCH;
        smx::TmaSoftmaxParams q;
        q.X = X;
        q.Y = Y;
        q.ldx = ldx;
        q.ldy = ldy;
        q.rows = rows;
        q.cols = static_cast<int32_t>(cols);
        q.bulk_elems = pl.bulk_elems;
        q.slot_bytes = static_cast<int32_t>(
            round_up(pl.pub.unit_rows == 1 ? cols * elem_bytes(x_dtype)
                                           : int64_t(pl.pub.unit_rows) * pl.row_stride, 128));
        q.depth = pl.pub.depth;
        q.group_warps = pl.pub.group_warps;
        q.unit_rows = pl.pub.unit_rows;
        q.row_stride = pl.row_stride;
        q.contiguous = pl.contiguous;
        q.kv = pl.pub.kv;
        q.whole = pl.whole ? 1 : 0;
        q.long_rows = pl.long_rows ? 1 : 0;
        q.cluster = pl.pub.cluster;
        q.slice = pl.pub.slice;
        q.err = err;
        {
            std::lock_guard<std::mutex> g(g_dbg_mu);
            q.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kDefaultWaitNs;
            q.debug_flags = g_debug_flags;
        }
        cudaError_t e = launch_tma(x_dtype, q, y_dtype, pl.pub.grid, pl.smem,
                                   reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }

    smx::SoftmaxParams p;
    p.X = X;
    p.Y = Y;
    p.ldx = ldx;
    p.ldy = ldy;
    p.rows = rows;
    p.cols = static_cast<int32_t>(cols);
    p.slice = pl.pub.slice;
    p.cluster = pl.pub.cluster;
    p.vec = pl.pub.vec;
    p.resident = pl.resident ? 1 : 0;
    cudaError_t e = launch(x_dtype, p, y_dtype, warp_rows, pl.pub.threads, pl.pub.grid,
                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // extern "C"

extern "C" {

gemm_status_t softmax_sync(gemm_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    int* err = error_word(dev);
    if (err == nullptr) return GEMM_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        cudaGetLastError();
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

gemm_status_t softmax_debug_set(uint32_t flags, uint64_t wait_limit_ns) {
    if (flags & ~SOFTMAX_DEBUG_SKIP_FIRST_LOAD) return GEMM_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> g(g_dbg_mu);
    g_debug_flags = flags;
    g_wait_limit_ns = wait_limit_ns;
    return GEMM_OK;
}

}  // extern "C"
