"""GPU parity of LayerNorm after the linear layer (gemm_run_layernorm)
against the oracle: rows normalised inside the GEMM epilogue (N <= 256, one
tile per row; single-CTA and CTA-pair tiles) and rows spread over several
tiles (per-tile statistics merged by the row pass), the quick returns
(K == 0, alpha == 0), exact integer inputs, and the canary columns of C."""
import numpy as np
import pytest
import torch

import checks
import gpu_cases as gc
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, TORCH_DTYPE, Workload

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module")
def g():
    import mixed_precision_dense_sm_gb300 as lib
    h = lib.Gemm()
    yield h
    h.close()


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _vectors(N, bias_dt, ln_dt, seed, integer=False):
    """bias ~ N(0, 1); gamma = 1 + 0.1 N(0, 1), shift = 0.1 N(0, 1) (the usual
    LayerNorm initialisation, perturbed); integer: small integers / halves."""
    gen = torch.Generator().manual_seed(seed + 11)
    if integer:
        bias = torch.randint(-4, 5, (N,), generator=gen).float()
        gamma = torch.randint(1, 5, (N,), generator=gen).float() * 0.5
        shift = torch.randint(-4, 5, (N,), generator=gen).float() * 0.25
    else:
        bias = torch.randn(N, generator=gen)
        gamma = 1.0 + 0.1 * torch.randn(N, generator=gen)
        shift = 0.1 * torch.randn(N, generator=gen)
    bias = None if bias_dt is None else bias.to(TORCH_DTYPE[bias_dt])
    if ln_dt is None:
        return bias, None, None
    return bias, gamma.to(TORCH_DTYPE[ln_dt]), shift.to(TORCH_DTYPE[ln_dt])


def _codes(t):
    return None if t is None else workloads.as_codes(t)


def _vals(t):
    return None if t is None else t.to(torch.float64).numpy()


def _run(g, orc, w, inp, bias, gamma, shift, rows=None, expect=None, exact_h=False,
         calls=1):
    """One (or `calls`) gemm_run_layernorm through the C ABI on the seeded
    inputs; compares the rows `rows` (all when None) with the oracle."""
    import mixed_precision_dense_sm_gb300 as lib
    M, N, K = w.M, w.N, w.K
    ln_dt = DT_F32 if gamma is None else workloads.DT_OF[gamma.dtype]
    bias_dt = DT_F32 if bias is None else workloads.DT_OF[bias.dtype]
    if expect is not None:
        st, plan = lib.gemm_layernorm_plan_query(
            w.transA, w.transB, M, N, K, w.alpha, 256, inp.lda, 256, inp.ldb, w.beta, 256,
            inp.ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype), bias=256 if bias is not None else 0,
            bias_dtype=bias_dt, gamma=256 if gamma is not None else 0,
            shift=256 if shift is not None else 0, ln_dtype=ln_dt, eps=EPS, num_sms=_num_sms())
        assert st == 0, st
        got = (plan["path_name"], plan["ln_fused"])
        assert got == expect, (w.name, got, plan)
    A, B = inp.A.cuda(), inp.B.cuda()
    cdt = TORCH_DTYPE[w.c_dtype]
    C0 = torch.full((M, inp.ldc), gc.CANARY, dtype=cdt)
    C0[:, :N] = inp.C[:, :N] if inp.C is not None else float("nan")   # beta == 0: unread
    dev = [t.cuda() if t is not None else None for t in (bias, gamma, shift)]
    for _ in range(calls):
        C = C0.cuda()
        g.layernorm(A, B, C, w.transA, w.transB, w.alpha, w.beta, bias=dev[0], gamma=dev[1],
                    shift=dev[2], eps=EPS, M=M, N=N, K=K)
        g.sync()
    Y, H, S = orc.gemm_layernorm(
        w.transA, w.transB, M, N, K, w.alpha, workloads.as_codes(inp.A), inp.lda,
        workloads.as_codes(inp.B), inp.ldb, w.beta,
        None if inp.C is None else workloads.as_codes(inp.C), inp.ldc, w.ab_dtype, w.c_dtype,
        _codes(bias), bias_dt, _codes(gamma), _codes(shift), ln_dt, EPS, row_ids=rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    blk = C[:M, :N].cpu()[sel]
    vals = blk.to(torch.float64).numpy()
    codes = None if w.c_dtype == DT_F32 else blk.contiguous().view(torch.int16).numpy().view(np.uint16)
    cin = None
    if w.beta != 0 and inp.C is not None:
        cin = inp.C[:, :N].to(torch.float64).numpy()
        cin = cin if rows is None else cin[rows]
    bound = checks.layernorm_bound(H, S, cin, None if bias is None else _vals(bias)[None, :],
                                   _vals(gamma), _vals(shift), w.alpha, w.beta, w.c_dtype, EPS,
                                   exact_h=exact_h)
    ocodes = None if w.c_dtype == DT_F32 else orc.round_output(Y, w.c_dtype)
    stats, bad = checks.compare_layernorm(vals, codes, Y, bound, w.c_dtype, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{w.name}: {stats}; first bad ({i},{j}) gpu={vals[i, j]!r} "
                             f"oracle={Y[i, j]!r} bound={bound[i, j]!r}")
    gc.check_canary(w, C)
    return stats


def _rows(M, n=96, seed=0):
    rng = np.random.default_rng(seed)
    r = np.unique(np.concatenate([rng.integers(0, M, n), [0, 1, M // 2, M - 2, M - 1]]))
    return r.astype(np.int64)


# (M, N, K, transA, transB, ab, c, beta, bias dtype, ln dtype, (path, fused), sampled rows)
CASES = [
    (300, 100, 200, "N", "T", DT_BF16, DT_BF16, 1.0, DT_BF16, DT_F32, ("tiled_1sm", 1), False),
    (517, 256, 333, "N", "N", DT_F16, DT_F16, 0.0, DT_F32, DT_F16, ("tiled_1sm", 1), False),
    (700, 200, 1000, "T", "N", DT_BF16, DT_F32, 1.0, None, DT_BF16, ("tiled_1sm", 1), False),
    (333, 1000, 500, "N", "T", DT_F16, DT_F32, 0.0, DT_F16, DT_BF16, ("tiled_1sm", 0), False),
    (40, 3000, 700, "N", "T", DT_BF16, DT_BF16, 1.0, DT_BF16, DT_BF16, ("tiled_1sm", 0), False),
    (129, 513, 64, "T", "T", DT_F16, DT_F16, 1.0, None, None, ("tiled_1sm", 0), False),
    (20000, 256, 192, "N", "T", DT_BF16, DT_BF16, 1.0, DT_F32, DT_F32, ("tiled_2sm", 1), True),
    (8192, 1024, 320, "N", "T", DT_BF16, DT_BF16, 1.0, DT_BF16, DT_BF16, ("tiled_2sm", 0), True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_{c[10][0]}_{'fused' if c[10][1] else 'rows'}"
                                             for c in CASES])
def test_layernorm_paths(g, orc, case):
    M, N, K, ta, tb, ab, c, beta, bias_dt, ln_dt, expect, sampled = case
    w = Workload(f"ln_{M}x{N}x{K}", M, N, K, ta, tb, ab, c, 1.0, beta, "N1", "N002",
                 "N1" if beta != 0 else None, seed=M + N + K)
    inp = workloads.make_inputs(w)
    bias, gamma, shift = _vectors(N, bias_dt, ln_dt, w.seed)
    _run(g, orc, w, inp, bias, gamma, shift, rows=_rows(M) if sampled else None, expect=expect)


@pytest.mark.parametrize("M,N,K,expect", [
    (250, 200, 96, ("tiled_1sm", 1)),
    (300, 777, 130, ("tiled_1sm", 0)),
    (8192, 600, 64, ("tiled_2sm", 0)),
    (20000, 256, 64, ("tiled_2sm", 1)),
    (20000, 160, 64, ("tiled_1sm", 1)),
])
def test_layernorm_exact_h(g, orc, M, N, K, expect):
    """Integer inputs in [-8, 8], integer bias and residual: every FP32 sum is
    exact, so h equals the oracle's and only the FP32 normalisation differs
    (a wrong mean, variance or merge fails the tight bound)."""
    w = Workload(f"ln_int_{M}x{N}x{K}", M, N, K, "N", "T", DT_BF16, DT_F32, 1.0, 1.0, "N1",
                 "N1", "N1", seed=M * 7 + N)
    inp = gc.integer_inputs(w)
    bias, gamma, shift = _vectors(N, DT_F32, DT_F32, w.seed, integer=True)
    sampled = _rows(M) if M > 2000 else None
    _run(g, orc, w, inp, bias, gamma, shift, rows=sampled, expect=expect, exact_h=True)


def test_layernorm_repeat_calls(g, orc):
    """Two calls in a row reuse the handle's workspace (per-tile statistics)."""
    w = Workload("ln_repeat_1000x1023x777", 1000, 1023, 777, "N", "N", DT_BF16, DT_F32, 1.0,
                 1.0, "N1", "N1", "N1", seed=5)
    inp = workloads.make_inputs(w)
    bias, gamma, shift = _vectors(w.N, DT_BF16, DT_F32, w.seed)
    _run(g, orc, w, inp, bias, gamma, shift, calls=2, expect=("tiled_1sm", 0))


@pytest.mark.parametrize("K,alpha,N", [(0, 1.0, 300), (64, 0.0, 100)])
def test_layernorm_quick_returns(g, orc, K, alpha, N):
    """K == 0 or alpha == 0: h = round_C(beta * C + bias), then the row pass
    computes the statistics itself."""
    w = Workload(f"ln_quick_K{K}", 77, N, K, "N", "N", DT_F16, DT_F16, alpha, 1.0, "N1", "N1",
                 "N1", seed=9)
    inp = workloads.make_inputs(w)
    bias, gamma, shift = _vectors(N, DT_F16, DT_BF16, w.seed)
    _run(g, orc, w, inp, bias, gamma, shift)


def test_layernorm_single_column(g, orc):
    """N == 1: zero deviation, every output equals shift."""
    w = Workload("ln_n1", 300, 1, 40, "N", "N", DT_BF16, DT_F32, 1.0, 0.0, "N1", "N1", None,
                 seed=3)
    inp = workloads.make_inputs(w)
    bias, gamma, shift = _vectors(1, None, DT_F32, w.seed)
    _run(g, orc, w, inp, bias, gamma, shift)


def test_layernorm_errors(g):
    import mixed_precision_dense_sm_gb300 as lib
    A = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    args = ("N", "N", 64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64, 0.0, C.data_ptr(), 64)
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.gemm_run_layernorm(g.h, *args, (0, 0, 0), eps=eps) == 1
    assert lib.gemm_run_layernorm(g.h, *args, (0, 0, 0), gamma=A.data_ptr(), ln_dtype=9) == 1
    assert lib.gemm_run_layernorm(g.h, *args, (0, 0, 0), bias=A.data_ptr(), bias_dtype=9) == 1
    assert lib.lib.gemm_run_layernorm(g.h, b"N", b"N", 64, 64, 64, 1.0, A.data_ptr(), 64,
                                      A.data_ptr(), 64, 0.0, C.data_ptr(), 64,
                                      lib.Dtypes(0, 0, 0), None, 0) == 1
    Af = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    Cf = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    st = lib.gemm_run_layernorm(g.h, "N", "N", 64, 64, 64, 1.0, Af.data_ptr(), 64, Af.data_ptr(),
                                64, 0.0, Cf.data_ptr(), 64, (2, 2, 2))
    assert st == 2
    # M == 0: no-op, C untouched
    st = lib.gemm_run_layernorm(g.h, "N", "N", 0, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64,
                                0.0, C.data_ptr(), 64, (0, 0, 0))
    assert st == 0
    g.sync()
    assert bool((C == 0).all())
