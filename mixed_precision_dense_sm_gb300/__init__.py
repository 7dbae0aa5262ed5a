"""Python binding for libgemm_sm103.so, the GB300 mixed-precision GEMM and
row softmax.

Argument marshalling only: every step of C = alpha*op(A)*op(B) + beta*C runs in
the library's CUDA kernels.  PyTorch is used for device memory and streams.
If the compiled library is missing, importing this package raises -- there is
no fallback implementation.

The entry points mirror include/gemm_sm103.h one to one:
``gemm_create``, ``gemm_run``, ``gemm_sync``, ``gemm_destroy``,
``gemm_status_string``, ``gemm_check_args``, ``gemm_plan_query``,
``gemm_run_ex`` (fused bias/activation epilogue), ``gemm_run_layernorm``
and ``gemm_layernorm_plan_query`` (LayerNorm after the linear layer),
``gemm_debug_set`` and ``gemm_run_noalloc``; and include/softmax_sm103.h: ``softmax_rows``,
``softmax_plan_query``, ``softmax_sync``, ``softmax_debug_set``; and
include/conv_sm103.h: ``conv2d_fprop``, ``conv2d_plan_query``,
``conv2d_output_dims``.
``Gemm`` wraps a handle and adds ``__call__`` for torch tensors; ``softmax``
does the same for the row softmax.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgemm_sm103.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "gemm_sm103.h")
HEADERS = [HEADER, os.path.join(os.path.dirname(HERE), "include", "softmax_sm103.h"),
           os.path.join(os.path.dirname(HERE), "include", "conv_sm103.h")]

GEMM_F16, GEMM_BF16, GEMM_F32 = 0, 1, 2
STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_VALUE", 2: "GEMM_ERR_NOT_SUPPORTED",
          3: "GEMM_ERR_ALLOC", 4: "GEMM_ERR_LAUNCH", 5: "GEMM_ERR_DEVICE_TIMEOUT"}
PATHS = {0: "noop", 1: "scale", 2: "tiled_1sm", 3: "tiled_2sm", 4: "skinny"}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class Dtypes(ctypes.Structure):
    _fields_ = [("a", ctypes.c_int32), ("b", ctypes.c_int32), ("c", ctypes.c_int32)]


class Epilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int32),
                ("activation", ctypes.c_int32)]


class LayerNorm(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int32),
                ("gamma", ctypes.c_void_p), ("shift", ctypes.c_void_p),
                ("ln_dtype", ctypes.c_int32), ("eps", ctypes.c_float)]


ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3
ACTIVATIONS = {None: ACT_NONE, "none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU,
               "silu": ACT_SILU}


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "path", "block_m", "block_n", "block_k", "stages", "split_k", "grid", "num_tiles",
        "pack_a", "pack_b", "a_mn_major", "b_mn_major", "swap_ab", "c_vector", "sk_len",
        "sk_max_seg", "k_blocks", "tiles_m", "tiles_n", "transpose_ab", "c_tma")] + \
        [("workspace_bytes", ctypes.c_int64), ("conv_rows", ctypes.c_int32),
         ("conv_pitch", ctypes.c_int32)]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["path_name"] = PATHS.get(self.path, "?")
        return d


SOFTMAX_MODES = {0: "noop", 1: "warp", 2: "cta", 3: "stream"}


class SoftmaxPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "mode", "threads", "cluster", "slice", "vec", "grid", "depth", "group_warps", "unit_rows",
        "kv")] + \
        [("hbm_bytes", ctypes.c_int64)]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["mode_name"] = SOFTMAX_MODES.get(self.mode, "?")
        return d


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, c = ctypes.c_int64, ctypes.c_void_p, ctypes.c_char
    run_args = [c, c, i64, i64, i64, ctypes.c_float, vp, i64, vp, i64, ctypes.c_float, vp, i64,
                Dtypes]
    lib.gemm_create.restype = ctypes.c_int
    lib.gemm_create.argtypes = [ctypes.POINTER(vp)]
    lib.gemm_run.restype = ctypes.c_int
    lib.gemm_run.argtypes = [vp] + run_args + [vp]
    lib.gemm_run_ex.restype = ctypes.c_int
    lib.gemm_run_ex.argtypes = [vp] + run_args + [ctypes.POINTER(Epilogue), vp]
    lib.gemm_run_layernorm.restype = ctypes.c_int
    lib.gemm_run_layernorm.argtypes = [vp] + run_args + [ctypes.POINTER(LayerNorm), vp]
    lib.gemm_layernorm_plan_query.restype = ctypes.c_int
    lib.gemm_layernorm_plan_query.argtypes = run_args + [
        ctypes.POINTER(LayerNorm), ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Plan),
        ctypes.POINTER(ctypes.c_int32)]
    lib.gemm_run_noalloc.restype = ctypes.c_int
    lib.gemm_run_noalloc.argtypes = run_args + [vp]
    lib.gemm_debug_set.restype = ctypes.c_int
    lib.gemm_debug_set.argtypes = [vp, ctypes.c_uint32, ctypes.c_uint64]
    lib.gemm_sync.restype = ctypes.c_int
    lib.gemm_sync.argtypes = [vp, vp]
    lib.gemm_destroy.restype = ctypes.c_int
    lib.gemm_destroy.argtypes = [vp]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_check_args.restype = ctypes.c_int
    lib.gemm_check_args.argtypes = run_args
    lib.gemm_plan_query.restype = ctypes.c_int
    lib.gemm_plan_query.argtypes = run_args + [ctypes.c_int32, ctypes.c_int32,
                                               ctypes.POINTER(Plan)]
    i32 = ctypes.c_int32
    smx_args = [i64, i64, vp, i64, i32, vp, i64, i32]
    lib.softmax_rows.restype = ctypes.c_int
    lib.softmax_rows.argtypes = smx_args + [vp]
    lib.softmax_plan_query.restype = ctypes.c_int
    lib.softmax_plan_query.argtypes = smx_args + [i32, i32, ctypes.POINTER(SoftmaxPlan)]
    conv_geo = [i64] * 13
    lib.conv2d_output_dims.restype = ctypes.c_int
    lib.conv2d_output_dims.argtypes = [i64] * 10 + [ctypes.POINTER(i64)] * 2
    lib.conv2d_fprop.restype = ctypes.c_int
    lib.conv2d_fprop.argtypes = [vp] + conv_geo + [ctypes.c_float, vp, vp, ctypes.c_float, vp,
                                                   Dtypes, ctypes.POINTER(Epilogue), vp]
    lib.conv2d_plan_query.restype = ctypes.c_int
    lib.conv2d_plan_query.argtypes = conv_geo + [ctypes.c_float, vp, vp, ctypes.c_float, vp,
                                                 Dtypes, i32, i32, ctypes.POINTER(Plan)]
    lib.softmax_sync.restype = ctypes.c_int
    lib.softmax_sync.argtypes = [vp]
    lib.softmax_debug_set.restype = ctypes.c_int
    lib.softmax_debug_set.argtypes = [ctypes.c_uint32, ctypes.c_uint64]
    return lib


lib = _load()


def _tr(t: str) -> bytes:
    return t.encode() if isinstance(t, str) else bytes(t)


def gemm_status_string(status: int) -> str:
    return lib.gemm_status_string(status).decode()


def gemm_create() -> int:
    h = ctypes.c_void_p()
    st = lib.gemm_create(ctypes.byref(h))
    if st != 0:
        raise GemmError(st, "gemm_create")
    return h.value


def gemm_destroy(h) -> int:
    return lib.gemm_destroy(h)


GEMM_DEBUG_SKIP_FIRST_LOAD = 1


def gemm_debug_set(h, flags: int, wait_limit_ns: int = 0) -> int:
    """Test hook of the failure path (see include/gemm_sm103.h)."""
    return lib.gemm_debug_set(h, flags, wait_limit_ns)


def gemm_sync(h, stream=0) -> int:
    return lib.gemm_sync(h, stream)


def gemm_run(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
             dtypes, stream=0) -> int:
    """Raw C-ABI call: A, B, C are device addresses (ints), dtypes a
    (a, b, c) tuple of GEMM_F16/GEMM_BF16/GEMM_F32, stream a cudaStream_t
    value.  Returns the gemm_status_t code."""
    return lib.gemm_run(h, _tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B, ldb,
                        float(beta), C, ldc, Dtypes(*dtypes), stream)


def gemm_run_ex(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtypes,
                bias=0, bias_dtype=GEMM_F32, act=ACT_NONE, stream=0) -> int:
    """Raw C-ABI call with a fused epilogue: act(alpha*AB + beta*C + bias[n]).
    bias is a device address (0 for none)."""
    ep = Epilogue(bias or None, bias_dtype, act)
    return lib.gemm_run_ex(h, _tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B, ldb,
                           float(beta), C, ldc, Dtypes(*dtypes), ctypes.byref(ep), stream)


def gemm_run_layernorm(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtypes,
                       bias=0, bias_dtype=GEMM_F32, gamma=0, shift=0, ln_dtype=GEMM_F32,
                       eps=1e-5, stream=0) -> int:
    """Raw C-ABI call of LayerNorm after the linear layer: C <- LayerNorm(
    round_C(alpha*AB + beta*C + bias)) * gamma + shift along each row of C.
    bias, gamma, shift are device addresses (0 for none)."""
    ln = LayerNorm(bias or None, bias_dtype, gamma or None, shift or None, ln_dtype, eps)
    return lib.gemm_run_layernorm(h, _tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B,
                                  ldb, float(beta), C, ldc, Dtypes(*dtypes), ctypes.byref(ln),
                                  stream)


def gemm_layernorm_plan_query(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              dtypes, bias=0, bias_dtype=GEMM_F32, gamma=0, shift=0,
                              ln_dtype=GEMM_F32, eps=1e-5, num_sms=152, smem_optin=232448):
    """(status, plan dict with "ln_fused") gemm_run_layernorm would use
    (host logic only)."""
    ln = LayerNorm(bias or None, bias_dtype, gamma or None, shift or None, ln_dtype, eps)
    plan = Plan()
    fused = ctypes.c_int32(-1)
    st = lib.gemm_layernorm_plan_query(_tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B,
                                       ldb, float(beta), C, ldc, Dtypes(*dtypes), ctypes.byref(ln),
                                       num_sms, smem_optin, ctypes.byref(plan),
                                       ctypes.byref(fused))
    if st != 0:
        return st, None
    d = plan.as_dict()
    d["ln_fused"] = fused.value
    return st, d


def gemm_run_noalloc(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     dtypes, stream=0) -> int:
    """Raw C-ABI call of the entry point that allocates nothing (no handle):
    for callers that cannot call cudaMalloc.  Same arguments as gemm_run
    without the handle; returns the gemm_status_t code."""
    return lib.gemm_run_noalloc(_tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B, ldb,
                                float(beta), C, ldc, Dtypes(*dtypes), stream)


def gemm_check_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtypes) -> int:
    return lib.gemm_check_args(_tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B, ldb,
                               float(beta), C, ldc, Dtypes(*dtypes))


def gemm_plan_query(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtypes,
                    num_sms=152, smem_optin=232448):
    """(status, plan dict) of the path gemm_run would take (host logic only)."""
    plan = Plan()
    st = lib.gemm_plan_query(_tr(transA), _tr(transB), M, N, K, float(alpha), A, lda, B, ldb,
                             float(beta), C, ldc, Dtypes(*dtypes), num_sms, smem_optin,
                             ctypes.byref(plan))
    return st, (plan.as_dict() if st == 0 else None)


def declared_symbols():
    """Function names declared in include/gemm_sm103.h and softmax_sm103.h."""
    import re
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names |= set(re.findall(r"^\s*(?:gemm_status_t|const char\*)\s+((?:gemm|softmax|conv2d)_\w+)\s*\(",
                                text, flags=re.M))
    return sorted(names)


def softmax_rows(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, stream=0) -> int:
    """Raw C-ABI call: Y = softmax(X) along each row.  X, Y are device
    addresses (ints); dtypes GEMM_F16/GEMM_BF16/GEMM_F32; stream a
    cudaStream_t value.  Returns the gemm_status_t code."""
    return lib.softmax_rows(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, stream)


SOFTMAX_DEBUG_SKIP_FIRST_LOAD = 1


def conv2d_output_dims(H, W, R, S, pad=(0, 0), stride=(1, 1), dilation=(1, 1)):
    """(P, Q) of a forward convolution (raises on bad geometry)."""
    P, Q = ctypes.c_int64(), ctypes.c_int64()
    st = lib.conv2d_output_dims(H, W, R, S, pad[0], pad[1], stride[0], stride[1], dilation[0],
                                dilation[1], ctypes.byref(P), ctypes.byref(Q))
    if st != 0:
        raise GemmError(st, "conv2d_output_dims")
    return P.value, Q.value


def conv2d_fprop(h, N, H, W, C, K, R, S, pad, stride, dilation, alpha, X, Wt, beta, Y, dtypes,
                 bias=0, bias_dtype=GEMM_F32, act=ACT_NONE, stream=0) -> int:
    """Raw C-ABI call (include/conv_sm103.h): X (NHWC), Wt (KRSC), Y (NPQK)
    device addresses; pad/stride/dilation (h, w) pairs; dtypes (x, w, y).
    Returns the gemm_status_t code."""
    ep = Epilogue(bias or None, bias_dtype, act)
    return lib.conv2d_fprop(h, N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1],
                            dilation[0], dilation[1], float(alpha), X, Wt, float(beta), Y,
                            Dtypes(*dtypes), ctypes.byref(ep), stream)


def conv2d_plan_query(N, H, W, C, K, R, S, pad, stride, dilation, alpha, X, Wt, beta, Y, dtypes,
                      num_sms=152, smem_optin=232448):
    """(status, GEMM plan dict) conv2d_fprop would use (host logic only)."""
    plan = Plan()
    st = lib.conv2d_plan_query(N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1],
                               dilation[0], dilation[1], float(alpha), X, Wt, float(beta), Y,
                               Dtypes(*dtypes), num_sms, smem_optin, ctypes.byref(plan))
    return st, (plan.as_dict() if st == 0 else None)


def softmax_sync(stream=0) -> int:
    """Wait for the stream; GEMM_ERR_DEVICE_TIMEOUT (5) if a softmax kernel
    recorded a bounded wait that ran out (then cleared)."""
    return lib.softmax_sync(stream)


def softmax_debug_set(flags: int, wait_limit_ns: int = 0) -> int:
    """Test hook of the softmax failure path (see include/softmax_sm103.h)."""
    return lib.softmax_debug_set(flags, wait_limit_ns)


def softmax_plan_query(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, num_sms=152,
                       ctas_per_sm=0):
    """(status, plan dict) of the work split softmax_rows would use (host logic)."""
    plan = SoftmaxPlan()
    st = lib.softmax_plan_query(rows, cols, X, ldx, x_dtype, Y, ldy, y_dtype, num_sms,
                                ctas_per_sm, ctypes.byref(plan))
    return st, (plan.as_dict() if st == 0 else None)


def softmax(X, Y=None, rows=None, cols=None, stream=None):
    """Row softmax of a 2-D torch tensor on the GPU (unit inner stride, row
    pitch = stride(0)) into Y (a new tensor of X's type and shape if None;
    Y may be X for in place).  Returns Y."""
    import torch
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be 2-D with unit inner stride")
    if Y is None:
        Y = torch.empty_like(X)
    if Y.dim() != 2 or Y.stride(1) != 1:
        raise ValueError("Y must be 2-D with unit inner stride")
    rows = X.shape[0] if rows is None else rows
    cols = X.shape[1] if cols is None else cols
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    st = softmax_rows(rows, cols, X.data_ptr(), X.stride(0), dtype_code(X.dtype), Y.data_ptr(),
                      Y.stride(0), dtype_code(Y.dtype), stream)
    if st != 0:
        raise GemmError(st, "softmax_rows")
    return Y


_TORCH_CODE = None


def dtype_code(t) -> int:
    global _TORCH_CODE
    if _TORCH_CODE is None:
        import torch
        _TORCH_CODE = {torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16,
                       torch.float32: GEMM_F32}
    return _TORCH_CODE[t]


class Gemm:
    """A library handle bound to the current CUDA device.

    ``g(A, B, C, transA, transB, alpha, beta, M=, N=, K=)`` marshals torch
    tensors (device, 2-D, unit inner stride, row pitch = stride(0)) into one
    gemm_run call on the current torch stream.  The logical sizes default to
    what the stored shapes imply."""

    def __init__(self):
        self.h = gemm_create()

    def close(self):
        if self.h:
            gemm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __call__(self, A, B, C, transA="N", transB="N", alpha=1.0, beta=0.0,
                 M=None, N=None, K=None, stream=None, bias=None, act=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        for t in (A, B, C):
            if t is not None and (t.dim() != 2 or t.stride(1) != 1):
                raise ValueError("operands must be 2-D with unit inner stride")
        if M is None:
            M = C.shape[0]
        if N is None:
            N = C.shape[1]
        if K is None:
            K = A.shape[1] if transA in "Nn" else A.shape[0]
        dts = (dtype_code(A.dtype), dtype_code(B.dtype), dtype_code(C.dtype))
        if bias is None and act is None:
            st = gemm_run(self.h, transA, transB, M, N, K, alpha, A.data_ptr(), A.stride(0),
                          B.data_ptr(), B.stride(0), beta, C.data_ptr(), C.stride(0), dts, stream)
        else:
            st = gemm_run_ex(self.h, transA, transB, M, N, K, alpha, A.data_ptr(), A.stride(0),
                             B.data_ptr(), B.stride(0), beta, C.data_ptr(), C.stride(0), dts,
                             bias.data_ptr() if bias is not None else 0,
                             dtype_code(bias.dtype) if bias is not None else GEMM_F32,
                             ACTIVATIONS[act] if not isinstance(act, int) else act, stream)
        if st != 0:
            raise GemmError(st, "gemm_run")
        return C

    def layernorm(self, A, B, C, transA="N", transB="N", alpha=1.0, beta=1.0, bias=None,
                  gamma=None, shift=None, eps=1e-5, M=None, N=None, K=None, stream=None):
        """LayerNorm after the linear layer, in place on C (the residual when
        beta != 0): C <- (h - mean) / sqrt(var + eps) * gamma + shift per row,
        h = round_C(alpha*op(A)op(B) + beta*C + bias).  gamma and shift share
        one dtype."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        for t in (A, B, C):
            if t is not None and (t.dim() != 2 or t.stride(1) != 1):
                raise ValueError("operands must be 2-D with unit inner stride")
        if gamma is not None and shift is not None and gamma.dtype != shift.dtype:
            raise ValueError("gamma and shift must share a dtype")
        M = C.shape[0] if M is None else M
        N = C.shape[1] if N is None else N
        if K is None:
            K = A.shape[1] if transA in "Nn" else A.shape[0]
        ln_t = gamma if gamma is not None else shift
        dts = (dtype_code(A.dtype), dtype_code(B.dtype), dtype_code(C.dtype))
        st = gemm_run_layernorm(
            self.h, transA, transB, M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(),
            B.stride(0), beta, C.data_ptr(), C.stride(0), dts,
            bias.data_ptr() if bias is not None else 0,
            dtype_code(bias.dtype) if bias is not None else GEMM_F32,
            gamma.data_ptr() if gamma is not None else 0,
            shift.data_ptr() if shift is not None else 0,
            dtype_code(ln_t.dtype) if ln_t is not None else GEMM_F32, eps, stream)
        if st != 0:
            raise GemmError(st, "gemm_run_layernorm")
        return C

    def sync(self, stream=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        st = gemm_sync(self.h, stream)
        if st != 0:
            raise GemmError(st, "gemm_sync")
