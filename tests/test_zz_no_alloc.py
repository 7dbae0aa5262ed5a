"""gemm_run_noalloc: the entry point for callers that cannot allocate.

Some callers of this library may not call cudaMalloc (code inside a memory
pool or allocator, code that has given all device memory to another owner, or
code that must not trigger the device synchronisation of a first allocation).
gemm_run_noalloc serves them: no handle, no allocation, its scratch in a static
device array.  These tests call it through the C ABI, twice in a row per
problem, and check every output element against the CPU oracle with the
parity tests' bound; where gemm_run's own plan fits the static scratch the two
entry points run the same plan, so their outputs must also be bitwise equal.
The file is named so pytest collects it last.
"""
import numpy as np
import pytest
import torch

import checks
import gpu_cases as gc
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, Workload

pytestmark = pytest.mark.gpu

SCRATCH = 32 << 20          # GEMM_NOALLOC_SCRATCH_BYTES


def _run(entry, w, inp, lib, handle=None):
    A = None if inp.A is None else inp.A.cuda()
    B = None if inp.B is None else inp.B.cuda()
    cdt = workloads.TORCH_DTYPE[w.c_dtype]
    C = torch.full((w.M, inp.ldc), gc.CANARY, dtype=cdt)
    if inp.C is not None:
        C[:, :w.N] = inp.C[:, :w.N]
    else:
        C[:, :w.N] = float("nan")          # beta == 0: C must not be read
    C = C.cuda()
    s = torch.cuda.current_stream().cuda_stream
    args = (w.transA, w.transB, w.M, w.N, w.K, w.alpha, 0 if A is None else A.data_ptr(),
            inp.lda, 0 if B is None else B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc,
            (w.ab_dtype, w.ab_dtype, w.c_dtype), s)
    st = lib.gemm_run(handle, *args) if entry == "run" else lib.gemm_run_noalloc(*args)
    assert st == 0, lib.gemm_status_string(st)
    torch.cuda.synchronize()
    return C


def _oracle(orc, w, inp):
    A = None if inp.A is None else workloads.as_codes(inp.A)
    B = None if inp.B is None else workloads.as_codes(inp.B)
    Cc = None if inp.C is None else workloads.as_codes(inp.C)
    return orc.gemm(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, inp.lda, B, inp.ldb, w.beta,
                    Cc, inp.ldc, w.ab_dtype, w.c_dtype)


def _check_oracle(orc, w, inp, got, R, S):
    """Every element of the no-alloc output against the oracle's result."""
    gv, gcodes = checks.gpu_values(got, w.M, w.N)
    ocodes = None if w.c_dtype == DT_F32 else orc.round_output(R, w.c_dtype)
    stats, bad = checks.compare(gv, gcodes, R, S, gc.cin_values(w, inp), w.alpha, w.beta,
                                w.c_dtype, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{w.name}: {stats}; first bad ({i},{j}) gpu={gv[i, j]!r} "
                             f"oracle={R[i, j]!r}")
    gc.check_canary(w, got)


def _plan(lib, w, inp):
    st, plan = lib.gemm_plan_query(w.transA, w.transB, w.M, w.N, w.K, w.alpha, 256, inp.lda,
                                   256, inp.ldb, w.beta, 256, inp.ldc,
                                   (w.ab_dtype, w.ab_dtype, w.c_dtype),
                                   num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0
    return plan


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def _k0_inputs(w):
    gen = torch.Generator().manual_seed(7)
    C = torch.randn((w.M, w.N), generator=gen).to(workloads.TORCH_DTYPE[w.c_dtype])
    return workloads.Inputs(None, None, C, 1, w.N, w.N)


# (workload, what it covers, the path gemm_run's plan takes)
CASES = [
    ("skinny_64x16384x8192_f16", "swapped skinny stream-K", "skinny"),
    ("ragged1000x1023x777_bf16_beta1", "packed ragged operands, beta = 1", None),
    ("square1024_f16_nt_f16out", "single-CTA tiles", "tiled_1sm"),
    (Workload("noalloc_tma_store_1000x1000x2048", 1000, 1000, 2048, "N", "T", DT_BF16, DT_F32,
              1.0, 0.0, "N1", "N1"), "C stored by TMA", None),
    (Workload("noalloc_pair_sk_512x3072x4096", 512, 3072, 4096, "N", "T", DT_BF16, DT_F32,
              1.0, 0.0, "N1", "N002"), "stream-K over CTA pairs", "tiled_2sm"),
    (Workload("noalloc_tf32_nt_300x520x1000", 300, 520, 1000, "N", "T", DT_F32, DT_F32,
              1.0, 0.0, "N1", "N1"), "FP32 inputs as TF32", None),
    (Workload("noalloc_tf32_nn_300x520x1000", 300, 520, 1000, "N", "N", DT_F32, DT_BF16,
              1.0, 0.0, "N1", "N1"), "TF32 with the transposing pre-pass", None),
    (Workload("noalloc_k0_beta_200x300", 200, 300, 0, "N", "N", DT_F16, DT_F32,
              1.0, 0.5, "N1", "N1", "N1"), "K = 0: C = beta C", "scale"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[1] for c in CASES])
def test_noalloc_matches_oracle_and_gemm_run_twice(orc, case):
    """Two calls in a row (the scratch reused) against the oracle, and
    bitwise against gemm_run, whose plan fits the scratch in every case."""
    import mixed_precision_dense_sm_gb300 as lib
    name, _, path = case
    w = workloads.WORKLOADS[name] if isinstance(name, str) else name
    inp = _k0_inputs(w) if w.K == 0 else workloads.make_inputs(w)
    plan = _plan(lib, w, inp)
    assert plan["workspace_bytes"] <= SCRATCH, plan
    if path is not None:
        assert plan["path_name"] == path, plan
    if w.name == "noalloc_tma_store_1000x1000x2048":
        assert plan["c_tma"] == 1, plan
    if w.name == "noalloc_pair_sk_512x3072x4096":
        assert plan["split_k"] > 1, plan
    if w.name == "noalloc_tf32_nn_300x520x1000":
        assert plan["transpose_ab"] == 2, plan
    R, S = _oracle(orc, w, inp)
    g = lib.Gemm()
    try:
        ref = _run("run", w, inp, lib, g.h)
    finally:
        g.close()
    for _ in range(2):
        got = _run("noalloc", w, inp, lib)
        _check_oracle(orc, w, inp, got, R, S)
        assert torch.equal(_bits(got), _bits(ref)), f"{w.name}: differs from gemm_run"


def test_noalloc_replans_split_k_to_fit(orc):
    """A problem whose gemm_run plan keeps more stream-K partial sums than the
    static scratch holds (6272 x 512 x 4608 on CTA pairs: about 37.5 MiB) is
    planned again with fewer stream-K units, not refused: the result obeys
    the oracle bound on two calls in a row."""
    import mixed_precision_dense_sm_gb300 as lib
    w = Workload("noalloc_replan_6272x512x4608", 6272, 512, 4608, "N", "T", DT_BF16, DT_F32,
                 1.0, 0.0, "N1", "N002")
    inp = workloads.make_inputs(w)
    plan = _plan(lib, w, inp)
    assert plan["workspace_bytes"] > SCRATCH and plan["split_k"] > 1, plan
    R, S = _oracle(orc, w, inp)
    for _ in range(2):
        got = _run("noalloc", w, inp, lib)
        _check_oracle(orc, w, inp, got, R, S)


def test_noalloc_rejects_scratch_beyond_maximum():
    """A problem whose packed operand copy alone exceeds the static array is
    refused up front and nothing is written."""
    import mixed_precision_dense_sm_gb300 as lib
    M, N, K = 8192, 256, 8191           # lda = 8191: A (128 MB) would need a packed copy
    st, plan = lib.gemm_plan_query("N", "N", M, N, K, 1.0, 256, K, 256, N, 0.0, 256, N,
                                   (DT_F16, DT_F16, DT_F32))
    assert st == 0 and plan["pack_a"] == 1 and plan["workspace_bytes"] > SCRATCH
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 5.0, device="cuda")
    st = lib.gemm_run_noalloc("N", "N", M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                              C.data_ptr(), N, (DT_F16, DT_F16, DT_F32),
                              torch.cuda.current_stream().cuda_stream)
    assert st == 1
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)
