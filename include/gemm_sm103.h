/*
 * gemm_sm103.h -- C ABI of the GB300 (sm_103a) mixed-precision dense GEMM.
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * What is computed (and where it is defined):
 *   - Each C[i][j] sums A[i][k] * B[k][j] over k (SGEMM tutorial page,
 *     section 3.1), and the formula C = A * B + C (CATLASS page, section 2.1).
 *     alpha, beta and op() are the BLAS reading of that formula; the pages
 *     name neither.
 *   - A and B are FP16 or BF16 (both the same type); products are accumulated
 *     in FP32 (DeepGEMM page, sections 1.3 and 6.2; CATLASS page, sections
 *     3.2 and 3.4).  The output C is FP32, FP16 or BF16; alpha*acc + beta*C is
 *     formed in FP32 and rounded once to the output type, round to nearest even.
 *   - A and B may also both be FP32, used as TF32 (the third format of the
 *     CATLASS page, section 3.2): they stay FP32 in memory and the tensor core
 *     keeps only the top 10 of each element's 23 mantissa bits (the low 13 are
 *     dropped, i.e. rounded toward zero); the accumulator is FP32 as above.
 *   - Storage is row-major with a leading dimension: element (m, n) of a
 *     stored matrix is at offset m * ld + n, in elements (CATLASS page,
 *     section 1.3).  op(X) = X for 'N'/'n' and X^T for 'T'/'t'.
 *       A, transA = 'N': stored M x K, lda >= max(1, K)
 *       A, transA = 'T': stored K x M, lda >= max(1, M)
 *       B, transB = 'N': stored K x N, ldb >= max(1, N)
 *       B, transB = 'T': stored N x K, ldb >= max(1, K)   ("weights N x K")
 *       C:               stored M x N, ldc >= max(1, N)
 *   - Shapes are arbitrary (M, N, K >= 0; the DeepGEMM page, section 1.3, asks
 *     for 1 to several thousand); tiles that overhang the matrix edge are
 *     zero-filled (DeepGEMM page, section 3.4).
 *   - Each of A, B and C must be aligned to its own element size (2 or 4
 *     bytes); any leading dimension and any further offset are accepted.
 *
 * Ownership and threading:
 *   - A, B and C are DEVICE pointers owned by the caller.  A and B are only
 *     read.  C is read only when beta != 0 and is always written (M x N
 *     elements; the padding columns n >= N of each row are never touched).
 *   - A handle owns a device workspace (packed copies of operands whose pitch
 *     or base address is not 16-byte aligned, split-K partial sums) and a
 *     device-visible error word.  The workspace grows on demand inside
 *     gemm_run (a cudaMalloc, which synchronises the device) and is released
 *     by gemm_destroy.
 *   - gemm_run is asynchronous with respect to the host: it enqueues work on
 *     `stream` and returns.  A handle must not be used from two host threads
 *     at once; use one handle per thread or per stream.  Calls on one handle
 *     that overlap on the GPU (different streams) may share workspace: order
 *     them on one stream.
 *
 * Errors: every entry point returns a gemm_status_t and never aborts.  Device
 * kernels never trap: every wait inside them is bounded, and a wait that runs
 * out records GEMM_ERR_DEVICE_TIMEOUT in the handle's error word, which the
 * next gemm_run or gemm_sync on that handle reports (and clears).
 */
#ifndef GEMM_SM103_H_
#define GEMM_SM103_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same layout as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* gemm_stream_t;
typedef struct gemm_ctx* gemm_handle_t;

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_F32 = 2 } gemm_dtype_t;

/* a, b: input types (must be equal: F16, BF16, or F32 computed as TF32); c:
 * output type (F32, F16 or BF16).  The accumulator is always FP32. */
typedef struct { int32_t a, b, c; } gemm_dtypes_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,   /* bad trans flag, shape, ld, pointer or dtype */
    GEMM_ERR_NOT_SUPPORTED = 2,   /* the current device is not sm_103 */
    GEMM_ERR_ALLOC = 3,           /* a workspace allocation failed */
    GEMM_ERR_LAUNCH = 4,          /* a CUDA call or kernel launch failed */
    GEMM_ERR_DEVICE_TIMEOUT = 5   /* a bounded in-kernel wait ran out */
} gemm_status_t;

/*
 * gemm_create: make a handle bound to the CURRENT CUDA device.
 *   out: receives the handle (set to NULL on failure).
 * Returns NOT_SUPPORTED if the device is not compute capability 10.3
 * (sm_103), LAUNCH if the CUDA runtime reports an error, ALLOC if the error
 * word cannot be allocated.
 */
gemm_status_t gemm_create(gemm_handle_t* out);

/*
 * gemm_run: C = alpha * op(A) * op(B) + beta * C on `stream`.
 *   transA, transB: 'N'/'n' or 'T'/'t'.
 *   M, N, K: op(A) is M x K, op(B) is K x N, C is M x N.
 *   A, lda / B, ldb / C, ldc: device pointers and leading dimensions in
 *     elements, laid out as in the table above.
 *   dt: element types (dt.a == dt.b in {F16, BF16, F32 as TF32}; dt.c in
 *     {F32, F16, BF16}).
 *   stream: the CUDA stream to enqueue on.
 * Quick returns (BLAS convention): M == 0 or N == 0 is a no-op; K == 0 or
 * alpha == 0 computes C = beta * C without reading A or B (A, B may then be
 * NULL); beta == 0 never reads C, so NaN/Inf already in C do not propagate.
 * Returns INVALID_VALUE for a bad argument (nothing is enqueued), ALLOC if the
 * workspace cannot grow, LAUNCH if a launch fails, DEVICE_TIMEOUT if an
 * earlier call on this handle recorded a device-side timeout (reported once).
 */
gemm_status_t gemm_run(gemm_handle_t h, char transA, char transB,
                       int64_t M, int64_t N, int64_t K,
                       float alpha, const void* A, int64_t lda,
                       const void* B, int64_t ldb,
                       float beta, void* C, int64_t ldc,
                       gemm_dtypes_t dt, gemm_stream_t stream);

/*
 * Fused epilogue (CATLASS page, section 5.2: an unchanged mainloop followed by
 * a replaced epilogue, read in the usual linear-layer form):
 *     C = act(alpha * op(A) * op(B) + beta * C + bias[n])
 * evaluated in FP32 before the single cast to C's type.  bias has N elements
 * (one per output column n), is read only, and may be NULL.  A residual add
 * is beta = 1 with the residual in C.
 *
 * Accuracy of the activations (x the FP32 pre-activation value):
 *   GELU -- relative error <= (x^2 / 2 + 2) 2^-21 + 3e-7 wherever the result
 *           is an FP32 normal, the negative tail included (no cancellation:
 *           it is evaluated through erfc); below about x = -13 the result
 *           leaves FP32's normal range and may be flushed to zero.  A 16-bit
 *           output is within one ulp of the correctly rounded value.
 *   SiLU -- relative error <= |x| 2^-23 + 2^-20 (the fast exponential).
 *   ReLU -- exact.
 */
typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,   /* x > 0 ? x : 0 (NaN stays NaN) */
    GEMM_ACT_GELU = 2,   /* x * Phi(x) = 0.5 x erfc(-x / sqrt 2) */
    GEMM_ACT_SILU = 3    /* x / (1 + exp(-x)) */
} gemm_activation_t;

typedef struct {
    const void* bias;    /* device pointer to N elements, or NULL */
    int32_t bias_dtype;  /* GEMM_F16, GEMM_BF16 or GEMM_F32 (ignored if bias is NULL) */
    int32_t activation;  /* gemm_activation_t */
} gemm_epilogue_t;

/*
 * gemm_run_ex: gemm_run with a fused epilogue.  ep == NULL is plain gemm_run.
 * The quick returns keep their shape: K == 0 or alpha == 0 gives
 * C = act(beta * C + bias) without reading A or B.  Returns INVALID_VALUE for
 * an unknown activation or bias type, otherwise as gemm_run.
 */
gemm_status_t gemm_run_ex(gemm_handle_t h, char transA, char transB,
                          int64_t M, int64_t N, int64_t K,
                          float alpha, const void* A, int64_t lda,
                          const void* B, int64_t ldb,
                          float beta, void* C, int64_t ldc,
                          gemm_dtypes_t dt, const gemm_epilogue_t* ep,
                          gemm_stream_t stream);

/*
 * LayerNorm after the linear layer -- the layer the CATLASS page starts from
 * (its introduction: a linear layer fused with a residual add and LayerNorm;
 * section 4.1: a normalisation is usually fused into the operator before it;
 * section 3.4: the normalisation keeps its reduction in FP32 while its data
 * path stays 16-bit):
 *     h_ij = round_C(alpha * (op(A) op(B))_ij + beta * C_ij + bias_j)
 *     C_ij <- round_C((h_ij - mean_i) / sqrt(var_i + eps) * gamma_j + shift_j)
 * where round_C rounds to C's type (h is the linear layer's output as C's type
 * holds it), mean_i and var_i are the mean and the biased variance of row i of
 * h over its N columns, and everything after the accumulation is FP32.  The
 * residual is C itself (beta = 1 adds it; beta = 0 does not read C), and C
 * receives y in place.  bias (bias_dtype) and gamma, shift (ln_dtype: F16,
 * BF16 or F32) are device vectors of N elements; NULL bias or shift reads as
 * 0, NULL gamma as 1.
 *
 * Rows of N <= 256 are normalised inside the GEMM's epilogue (the row is whole
 * in one tile): h never leaves the chip.  Wider rows: the epilogue stores h and
 * each row's per-tile (sum, M2) into the handle's workspace, then one row pass
 * combines them (mean = sum of sums / N; M2 = sum of the tiles' M2 plus
 * n_t (tile mean - mean)^2 per tile) and rewrites the row once.  K == 0 or
 * alpha == 0: h = round_C(beta * C + bias), then the row pass computes the
 * statistics itself.
 *
 * Inputs A and B: F16 or BF16 (FP32/TF32 inputs return NOT_SUPPORTED); the
 * problem is never swapped or split along K.  Returns INVALID_VALUE for
 * ln == NULL, eps not positive and finite, or an unknown bias / ln type;
 * otherwise as gemm_run.
 */
typedef struct {
    const void* bias;     /* device, N elements, or NULL */
    int32_t bias_dtype;   /* GEMM_F16, GEMM_BF16 or GEMM_F32 */
    const void* gamma;    /* device, N elements, or NULL (1) */
    const void* shift;    /* device, N elements, or NULL (0) */
    int32_t ln_dtype;     /* type of gamma and shift */
    float eps;            /* > 0 */
} gemm_layernorm_t;

gemm_status_t gemm_run_layernorm(gemm_handle_t h, char transA, char transB,
                                 int64_t M, int64_t N, int64_t K,
                                 float alpha, const void* A, int64_t lda,
                                 const void* B, int64_t ldb,
                                 float beta, void* C, int64_t ldc,
                                 gemm_dtypes_t dt, const gemm_layernorm_t* ln,
                                 gemm_stream_t stream);

/*
 * gemm_sync: wait for `stream`, then report (and clear) a device-side timeout
 * recorded by any kernel of this handle.  Returns LAUNCH if the stream itself
 * reports an error.
 */
gemm_status_t gemm_sync(gemm_handle_t h, gemm_stream_t stream);

/* gemm_destroy: synchronise the device and free the handle and its workspace.
 * NULL is accepted (no-op). */
gemm_status_t gemm_destroy(gemm_handle_t h);

/*
 * gemm_debug_set: test hook for the failure path (no counterpart on the
 * pages).  wait_limit_ns bounds every in-kernel wait of later calls on this
 * handle (0 restores the default of 2 s).  With flags =
 * GEMM_DEBUG_SKIP_FIRST_LOAD, the first CTA's producer arms its first
 * pipeline slot but issues no load into it: the MMA's bounded wait on that slot
 * runs out, the kernel records GEMM_ERR_DEVICE_TIMEOUT and winds down (no trap,
 * no fault; the CUDA context stays usable), and the next gemm_sync or gemm_run
 * on the handle reports it.  The results of such a call are undefined.
 * flags = 0 restores normal operation.  Returns INVALID_VALUE for a NULL
 * handle or an unknown flag.
 */
#define GEMM_DEBUG_SKIP_FIRST_LOAD 1u
gemm_status_t gemm_debug_set(gemm_handle_t h, uint32_t flags, uint64_t wait_limit_ns);

/* A static, human-readable name for a status code. */
const char* gemm_status_string(gemm_status_t s);

/*
 * gemm_check_args: the argument validation gemm_run performs, without a
 * handle or a device (pure host logic).  Pointers are only compared with NULL.
 */
gemm_status_t gemm_check_args(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const void* A, int64_t lda,
                              const void* B, int64_t ldb,
                              float beta, const void* C, int64_t ldc,
                              gemm_dtypes_t dt);

/* Which kernel path gemm_run takes for a problem, as decided on the host. */
typedef enum {
    GEMM_PATH_NOOP = 0,       /* M == 0 or N == 0 */
    GEMM_PATH_SCALE = 1,      /* K == 0 or alpha == 0: C = beta * C */
    GEMM_PATH_TILED_1SM = 2,  /* persistent tcgen05 kernel, one CTA per 128 x BN tile */
    GEMM_PATH_TILED_2SM = 3,  /* persistent tcgen05 kernel on 2-SM CTA pairs, 256 x BN tiles */
    GEMM_PATH_SKINNY = 4      /* memory-bound small-M path (swap A/B, split-K) */
} gemm_path_t;

typedef struct {
    int32_t path;          /* gemm_path_t */
    int32_t block_m;       /* output rows per tile (per CTA pair for 2SM) */
    int32_t block_n;       /* output columns per tile */
    int32_t block_k;       /* K elements per pipeline stage */
    int32_t stages;        /* shared-memory pipeline depth */
    int32_t split_k;       /* number of K partitions (1 = none) */
    int32_t grid;          /* CTAs launched for the main kernel */
    int32_t num_tiles;     /* output tiles (x split_k work units) */
    int32_t pack_a;        /* 1: A is copied to an aligned workspace first */
    int32_t pack_b;        /* 1: B is copied to an aligned workspace first */
                           /* (the copy is a transposition when transpose_ab says so) */
    int32_t a_mn_major;    /* 1: op(A) is read M-contiguous (transA = 'T') */
    int32_t b_mn_major;    /* 1: op(B) is read N-contiguous (transB = 'N') */
    int32_t swap_ab;       /* 1: computed as C^T = op(B)^T op(A)^T */
    int32_t c_vector;      /* 1: C rows are 16-byte aligned (vector epilogue) */
    int32_t sk_len;        /* stream-K: k-blocks per CTA (0 = data-parallel) */
    int32_t sk_max_seg;    /* stream-K: workspace slots per CTA */
    int32_t k_blocks;      /* ceil(K / block_k) */
    int32_t tiles_m;       /* tile rows (of the possibly swapped problem) */
    int32_t tiles_n;       /* tile columns */
    int32_t transpose_ab;  /* FP32 (TF32) inputs only: bit 0 (A), bit 1 (B) set when that
                              operand is stored M/N-contiguous and a pre-pass rewrites it
                              K-contiguous into the workspace (kind::tf32 reads K-major
                              operands only) */
    int32_t c_tma;         /* 1: the epilogue stages C in shared memory and stores it by TMA
                              (C rows 16-byte aligned, beta == 0, and FP32 C with K >= 2048
                              or two or more data-parallel tiles per CTA); 0: per-thread
                              row stores */
    int64_t workspace_bytes;
    int32_t conv_rows;     /* convolutions: > 0 when each tile is this many whole output rows
                              of one image, loaded as tiled boxes of the input (stride 1,
                              256-row single-CTA tiles); 0: im2col tiles (and every GEMM) */
    int32_t conv_pitch;    /* whole-row tiles: the tile's A rows per output row.  Q rounded
                              up to 8 for halo units (one box of conv_rows + (R - 1) dil_h
                              input rows per filter column and 64-channel block, the R taps
                              read at row offsets of the box: k_blocks = S ceil(C / 64));
                              Q for one box per filter tap; 0 for im2col tiles */
} gemm_plan_t;

/*
 * gemm_plan_query: the plan gemm_run would use for these arguments on a
 * device with `num_sms` SMs and `smem_optin` bytes of opt-in shared memory
 * per block (pure host logic, no device needed; pointers are used only for
 * their 16-byte alignment).  Returns INVALID_VALUE for arguments gemm_run
 * would reject.
 */
gemm_status_t gemm_plan_query(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const void* A, int64_t lda,
                              const void* B, int64_t ldb,
                              float beta, const void* C, int64_t ldc,
                              gemm_dtypes_t dt, int32_t num_sms, int32_t smem_optin,
                              gemm_plan_t* out);

/* The plan gemm_run_layernorm would use (host logic only, as gemm_plan_query);
 * *fused (if not NULL) is 1 when rows are normalised inside the epilogue. */
gemm_status_t gemm_layernorm_plan_query(char transA, char transB,
                                        int64_t M, int64_t N, int64_t K,
                                        float alpha, const void* A, int64_t lda,
                                        const void* B, int64_t ldb,
                                        float beta, const void* C, int64_t ldc,
                                        gemm_dtypes_t dt, const gemm_layernorm_t* ln,
                                        int32_t num_sms, int32_t smem_optin,
                                        gemm_plan_t* out, int32_t* fused);

/* Size of the static device scratch used by gemm_run_noalloc (32 MiB). */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * gemm_run_noalloc: gemm_run for callers that cannot allocate device memory.
 * There is no counterpart on the pages; it exists because some callers may not
 * call cudaMalloc at all -- code running inside a memory pool or allocator
 * that must not re-enter the CUDA allocator, code that has handed all device
 * memory to another owner, or code that must not trigger the implicit device
 * synchronisation a first cudaMalloc brings.  It takes no handle, calls no
 * cudaMalloc, cudaFree or other allocating routine, and computes what
 * gemm_run computes, with the same arguments, conventions and argument errors
 * (bit for bit whenever gemm_run's plan fits the scratch, below).
 *
 * Scratch: packed operand copies and split-K partial sums go to one file-scope
 * device array of GEMM_NOALLOC_SCRATCH_BYTES, which every GPU that loads this
 * library holds until the process exits.  When gemm_run's plan would need
 * more scratch than that for its split-K partial sums, the same problem is
 * planned with fewer split-K units (and, if that is not enough, without
 * split-K); the result then obeys the same accuracy bound as gemm_run's but
 * may differ from it in the last bits (another summation split).  A problem
 * whose packed operand copies alone exceed the array is rejected with
 * GEMM_ERR_INVALID_VALUE and nothing is enqueued.  All calls on a device
 * share the array and it keeps the last call's contents; the part that must
 * start at zero (split-K tile counters) is cleared on the stream by each call
 * that uses it.  Calls that overlap on the GPU -- on different streams, or
 * from different host threads without ordering -- race on it, so order them
 * on one stream.
 *
 * Set-up: the first call on each device (with that device current) resolves
 * the array's device address and loads the kernels; make that first call
 * before any stream capture.  A set-up that fails (LAUNCH or NOT_SUPPORTED
 * returned) is tried again by the next call on that device.  `stream` must
 * belong to the current device (GEMM_ERR_INVALID_VALUE otherwise: the
 * array's address is the current device's).  Device-side timeouts still wind
 * the kernel down cleanly but are not reported, since there is no handle
 * error word.  Returns NOT_SUPPORTED off sm_103 and LAUNCH if a CUDA call
 * fails.
 */
gemm_status_t gemm_run_noalloc(char transA, char transB,
                               int64_t M, int64_t N, int64_t K,
                               float alpha, const void* A, int64_t lda,
                               const void* B, int64_t ldb,
                               float beta, void* C, int64_t ldc,
                               gemm_dtypes_t dt, gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_SM103_H_ */
