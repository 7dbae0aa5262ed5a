/*
 * softmax_sm103.h -- C ABI of the GB300 (sm_103a) row softmax, the
 * memory-bound kernel of the SGEMM tutorial page (section 2).
 *
 * What is computed (and where it is defined):
 *   - For every row x_0..x_{n-1} of X:  m = max_j x_j,  e_j = exp(x_j - m),
 *     s = sum_j e_j,  y_j = e_j / s  (SGEMM tutorial page, section 2.1: the
 *     maximum, the sum of exponentials of the shifted values, the division).
 *     The maximum shift keeps exp from overflowing (section 2.2).
 *   - Each element is read from HBM once and written once.  A row that fits
 *     on chip (one warp's or one CTA's registers, up to 16384 elements) is
 *     read once; a longer row is read twice by one CTA -- a first pass
 *     accumulates (m, s) chunk by chunk with the online rule m' = max(m1, m2),
 *     s' = s1 e^(m1-m') + s2 e^(m2-m') (section 2.2), a second pass writes
 *     y -- and the first pass leaves the row in L2 for the second.  Rows so
 *     long that the slices of all resident CTAs would exceed half the L2 are
 *     spread over a thread-block cluster of up to 8 CTAs whose (m, s) pairs
 *     merge by the same rule through distributed shared memory.
 *   - Arithmetic is FP32 whatever the storage type (the CATLASS page, section
 *     3.4, keeps reductions such as softmax in FP32 with 16-bit data paths);
 *     exp is the fast hardware exponential (__expf, as on the SGEMM page,
 *     section 2.5; staged rows of 16-bit inputs take 2^(t log2 e) from the
 *     hardware base-2 exponential, with results below 2^-126 flushed to
 *     zero: the same error form); y is rounded once to its type, round to
 *     nearest even.
 *   - Special values follow the formula: a row containing NaN or +inf, and a
 *     fully masked row (every entry -inf, 0/0 -- section 2.5), give NaN in
 *     every position; otherwise an entry of -inf gives exactly 0.
 *
 * Layout: row-major; element (r, j) of X is at X + r * ldx + j, of Y at
 * Y + r * ldy + j, in elements.  X and Y are DEVICE pointers owned by the
 * caller, each aligned to its element size; X is only read, Y only written
 * (the columns j >= cols of each row are never touched).  Y may be X itself
 * (same pointer, same leading dimension, same type: in place); any other
 * overlap of the two is rejected.
 *
 * Rows of 256 bytes to 64 KB (at most 16384 FP32 or 32768 16-bit elements)
 * that start on 16-byte boundaries are staged in shared memory by bulk
 * copies (TMA): one CTA of 16 warps per SM, split into
 * groups of 1-16 warps, each group a pipeline that keeps the copies of its
 * next few rows in flight while it works on one (~130-190 KB per SM in all),
 * so HBM is streamed without registers holding the loads.  Other rows are
 * held in registers (warp or CTA splits) or take the two passes above.
 *
 * Errors: returns GEMM_OK, GEMM_ERR_INVALID_VALUE (bad sizes, leading
 * dimension, type, NULL or misaligned pointer, overlap; nothing enqueued),
 * GEMM_ERR_NOT_SUPPORTED (the current device is not sm_103) or
 * GEMM_ERR_LAUNCH.  The call is asynchronous on `stream` and allocates
 * nothing.  The staged kernels wait on their own bulk copies; every such wait
 * is bounded (2 s), and one that runs out sets a per-device error word that
 * softmax_sync reports as GEMM_ERR_DEVICE_TIMEOUT (the rows of that pipeline
 * are then not written).  No kernel waits on another launch.
 */
#ifndef SOFTMAX_SM103_H_
#define SOFTMAX_SM103_H_

#include <stdint.h>

#include "gemm_sm103.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * softmax_rows: Y = softmax(X) along each of `rows` rows of `cols` elements.
 *   x_dtype, y_dtype: GEMM_F16, GEMM_BF16 or GEMM_F32 (independently).
 *   cols <= 2^30; ldx, ldy: leading dimensions in elements, >= max(1, cols).
 * rows == 0 or cols == 0 is a no-op (the pointers may then be NULL).
 */
gemm_status_t softmax_rows(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                           int32_t x_dtype, void* Y, int64_t ldy, int32_t y_dtype,
                           gemm_stream_t stream);

typedef enum {
    SOFTMAX_MODE_NOOP = 0,      /* rows == 0 or cols == 0 */
    SOFTMAX_MODE_WARP = 1,      /* one warp per row, row in registers (cols <= 1024) */
    SOFTMAX_MODE_CTA = 2,       /* one CTA per row, row in registers or staged */
    SOFTMAX_MODE_STREAM = 3     /* one CTA (or a cluster of CTAs) per row, two passes */
} softmax_mode_t;

typedef struct {
    int32_t mode;          /* softmax_mode_t */
    int32_t threads;       /* threads per CTA */
    int32_t cluster;       /* CTAs per row (1 = no cluster) */
    int32_t slice;         /* elements of a row per CTA (multiple of 8) */
    int32_t vec;           /* 1: 16-byte loads and stores (rows 16-byte aligned) */
    int32_t grid;          /* CTAs launched (persistent over rows) */
    int32_t depth;         /* > 0: rows staged in shared memory by bulk copies (TMA),
                              this many row slots per pipeline; 0: rows held in registers */
    int32_t group_warps;   /* staged: warps per pipeline (the CTA runs 16 / group_warps
                              independent pipelines, fed by one producer warp); 0 otherwise */
    int32_t unit_rows;     /* staged: rows per slot -- 1: the group's warps share a row;
                              more: each warp takes its own rows of the slot, and rows that
                              are adjacent in X arrive in one copy of the whole slot */
    int32_t kv;            /* staged: 16-byte vectors of a row per thread (1, 2, 4, 8) */
    int64_t hbm_bytes;     /* bytes this plan reads and writes (two-pass rows count X
                              twice; the second read is meant to hit L2) */
} softmax_plan_t;

/*
 * softmax_plan_query: the plan softmax_rows would use on a device with
 * `num_sms` SMs, assuming `ctas_per_sm` resident CTAs per SM of the chosen
 * shape -- or, when a row is split over a cluster, that many resident
 * clusters on the whole GPU (0: the library's estimate).  Two-pass rows
 * take the smallest cluster (1, 2, 4 or 8) whose resident slices,
 * num_sms x slice x input size, stay within 64 MB.  Pure host logic;
 * pointers are used only for their alignment and overlap.  Returns what
 * softmax_rows would return for invalid arguments.
 */
gemm_status_t softmax_plan_query(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                                 int32_t x_dtype, const void* Y, int64_t ldy, int32_t y_dtype,
                                 int32_t num_sms, int32_t ctas_per_sm, softmax_plan_t* out);

/*
 * softmax_sync: wait for `stream`, then report (and clear) a device-side
 * timeout recorded by any softmax kernel on the current device since the last
 * softmax_sync: GEMM_ERR_DEVICE_TIMEOUT, else GEMM_OK (GEMM_ERR_LAUNCH if the
 * CUDA runtime reports an error).
 */
gemm_status_t softmax_sync(gemm_stream_t stream);

/*
 * softmax_debug_set: test hook of the failure path, process-wide.
 * SOFTMAX_DEBUG_SKIP_FIRST_LOAD makes the first pipeline of the first CTA of
 * each staged launch arm its first row slot without issuing the copy, so that
 * wait runs out; wait_limit_ns replaces the 2 s bound (0 restores it).
 * flags = 0 restores normal operation.  Returns GEMM_ERR_INVALID_VALUE for
 * unknown flags.
 */
#define SOFTMAX_DEBUG_SKIP_FIRST_LOAD 1u
gemm_status_t softmax_debug_set(uint32_t flags, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif  /* SOFTMAX_SM103_H_ */
