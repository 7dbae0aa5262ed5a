"""gemm_run_noalloc: the entry point for callers that cannot allocate.

Some callers of this library may not call cudaMalloc (code inside a memory
pool or allocator, code that has given all device memory to another owner, or
code that must not trigger the device synchronisation of a first allocation).
gemm_run_noalloc serves them: no handle, no allocation, its scratch in a static
device array.  These tests call it through the C ABI and check its output
against gemm_run's on the same inputs, within the tolerance the parity tests
use, on two calls in a row.  The file is named so pytest collects it last.
"""
import numpy as np
import pytest
import torch

import checks
import gpu_cases as gc
import workloads
from workloads import DT_BF16, DT_F16, DT_F32

pytestmark = pytest.mark.gpu


def _run(entry, w, inp, lib, handle=None):
    A, B = inp.A.cuda(), inp.B.cuda()
    cdt = workloads.TORCH_DTYPE[w.c_dtype]
    C = torch.full((w.M, inp.ldc), gc.CANARY, dtype=cdt)
    if inp.C is not None:
        C[:, :w.N] = inp.C[:, :w.N]
    C = C.cuda()
    s = torch.cuda.current_stream().cuda_stream
    args = (w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(), inp.lda, B.data_ptr(),
            inp.ldb, w.beta, C.data_ptr(), inp.ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype), s)
    st = lib.gemm_run(handle, *args) if entry == "run" else lib.gemm_run_noalloc(*args)
    assert st == 0, lib.gemm_status_string(st)
    torch.cuda.synchronize()
    return C


def _close(orc, w, inp, got, ref):
    """got (no-alloc) against ref (gemm_run), with the parity tests' bound."""
    A, B = workloads.as_codes(inp.A), workloads.as_codes(inp.B)
    Cc = None if inp.C is None else workloads.as_codes(inp.C)
    _, S = orc.gemm(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, inp.lda, B, inp.ldb, w.beta,
                    Cc, inp.ldc, w.ab_dtype, w.c_dtype)
    gv, gcodes = checks.gpu_values(got, w.M, w.N)
    rv, rcodes = checks.gpu_values(ref, w.M, w.N)
    cin = gc.cin_values(w, inp)
    stats, bad = checks.compare(gv, gcodes, rv, S, cin, w.alpha, w.beta, w.c_dtype, rcodes)
    assert stats["fail"] == 0, stats
    gc.check_canary(w, got)


CASES = ["skinny_64x16384x8192_f16", "ragged1000x1023x777_bf16_beta1",
         "square1024_f16_nt_f16out",
         # FP32 C: the epilogue stages C in shared memory and stores it by TMA
         workloads.Workload("noalloc_tma_store_1000x1000x2048", 1000, 1000, 2048, "N", "T",
                            DT_BF16, DT_F32, 1.0, 0.0, "N1", "N1")]


def test_noalloc_matches_gemm_run_twice(orc):
    """Two calls in a row per workload (scratch reused, stream-K partial sums
    and packed operands, C stored by TMA), each checked against gemm_run."""
    import mixed_precision_dense_sm_gb300 as lib
    g = lib.Gemm()
    try:
        for name in CASES:
            w = workloads.WORKLOADS[name] if isinstance(name, str) else name
            if not isinstance(name, str):
                lda, ldb, ldc = w.lds()
                st, plan = lib.gemm_plan_query(w.transA, w.transB, w.M, w.N, w.K, 1.0, 256, lda,
                                               256, ldb, 0.0, 256, ldc,
                                               (w.ab_dtype, w.ab_dtype, w.c_dtype))
                assert st == 0 and plan["c_tma"] == 1, plan
            inp = workloads.make_inputs(w)
            ref = _run("run", w, inp, lib, g.h)
            for _ in range(2):
                got = _run("noalloc", w, inp, lib)
                _close(orc, w, inp, got, ref)
    finally:
        g.close()


def test_noalloc_rejects_scratch_beyond_maximum():
    """A problem whose scratch exceeds the static array is refused up front
    and nothing is written."""
    import mixed_precision_dense_sm_gb300 as lib
    M, N, K = 8192, 256, 8191           # lda = 8191: A (128 MB) would need a packed copy
    st, plan = lib.gemm_plan_query("N", "N", M, N, K, 1.0, 256, K, 256, N, 0.0, 256, N,
                                   (DT_F16, DT_F16, DT_F32))
    assert st == 0 and plan["workspace_bytes"] > (32 << 20)
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 5.0, device="cuda")
    st = lib.gemm_run_noalloc("N", "N", M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                              C.data_ptr(), N, (DT_F16, DT_F16, DT_F32),
                              torch.cuda.current_stream().cuda_stream)
    assert st == 1
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)
