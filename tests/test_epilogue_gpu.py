"""GPU parity of the fused epilogue act(alpha*op(A)*op(B) + beta*C + bias[n])
against the oracle, on every kernel path."""
import itertools

import numpy as np
import pytest
import torch

import checks
import gpu_cases as gc
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, TORCH_DTYPE, Workload

pytestmark = pytest.mark.gpu

ACTS = [0, 1, 2, 3]          # none, ReLU, GELU, SiLU


@pytest.fixture(scope="module")
def g():
    import mixed_precision_dense_sm_gb300 as lib
    h = lib.Gemm()
    yield h
    h.close()


def _case(g, orc, M, N, K, ta, tb, ab, c, act, bias_dt, beta, seed, path=None):
    import mixed_precision_dense_sm_gb300 as lib
    w = Workload(f"ep_{M}x{N}x{K}", M, N, K, ta, tb, ab, c, 0.75, beta, "N1", "N1",
                 "N1" if beta != 0 else None, seed=seed)
    inp = workloads.make_inputs(w)
    gen = torch.Generator().manual_seed(seed + 7)
    bias = None if bias_dt is None else torch.randn(N, generator=gen).to(TORCH_DTYPE[bias_dt])
    if path is not None:
        lda, ldb, ldc = w.lds()
        st, plan = lib.gemm_plan_query(ta, tb, M, N, K, w.alpha, 256, lda, 256, ldb, beta, 256,
                                       ldc, (ab, ab, c),
                                       num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert st == 0 and plan["path_name"] == path[0] and bool(plan["sk_len"]) == path[1], plan
    A, B = inp.A.cuda(), inp.B.cuda()
    C = torch.full((M, inp.ldc), gc.CANARY, dtype=TORCH_DTYPE[c])
    C[:, :N] = inp.C[:, :N] if inp.C is not None else float("nan")
    C = C.cuda()
    g(A, B, C, ta, tb, w.alpha, beta, M=M, N=N, K=K,
      bias=None if bias is None else bias.cuda(), act=act)
    g.sync()
    bias_codes = None if bias is None else workloads.as_codes(bias)
    R, S = orc.gemm_ex(ta, tb, M, N, K, w.alpha, workloads.as_codes(inp.A), inp.lda,
                       workloads.as_codes(inp.B), inp.ldb, beta,
                       None if inp.C is None else workloads.as_codes(inp.C), inp.ldc, ab, c,
                       bias_codes, DT_F32 if bias_dt is None else bias_dt, act)
    vals, codes = checks.gpu_values(C, M, N)
    ocodes = None if c == DT_F32 else orc.round_output(R, c)
    bias_vals = None if bias is None else bias.to(torch.float64).numpy()[None, :]
    stats, bad = checks.compare_epilogue(vals, codes, R, S, gc.cin_values(w, inp), bias_vals,
                                         w.alpha, beta, c, ocodes)
    if stats["fail"]:
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{w.name} act={act} bias={bias_dt}: {stats}; ({i},{j}) "
                             f"gpu={vals[i, j]!r} oracle={R[i, j]!r}")
    gc.check_canary(w, C)


PATHS = [
    # (M, N, K, transA, transB, (path, stream-K))
    (1900, 4736, 200, "N", "T", ("tiled_2sm", False)),
    (300, 520, 1000, "N", "N", ("tiled_1sm", False)),
    (257, 129, 4096, "T", "T", ("tiled_1sm", True)),
    (40, 1000, 3000, "N", "T", ("skinny", True)),
]


@pytest.mark.parametrize("M,N,K,ta,tb,path", PATHS, ids=[p[-1][0] + ("_sk" if p[-1][1] else "")
                                                        for p in PATHS])
def test_fused_epilogue_paths(g, orc, M, N, K, ta, tb, path):
    for n, act in enumerate(ACTS):
        c = (DT_BF16, DT_F32, DT_F16, DT_F32)[n]
        bias_dt = (DT_F32, DT_BF16, None, DT_F16)[n]
        beta = (0.0, 1.0)[n % 2]
        _case(g, orc, M, N, K, ta, tb, DT_BF16 if n % 2 else DT_F16, c, act, bias_dt, beta,
              seed=M + n, path=path if n == 0 else None)


def test_fused_epilogue_pair_stream_k(g, orc):
    """Stream-K on CTA pairs: 20 pair tiles of 256 x 256, each split in two,
    so the finishing pair adds its partner's partial sums before the fused
    bias, residual and GELU."""
    _case(g, orc, 512, 2432, 4096, "N", "T", DT_BF16, DT_BF16, 2, DT_F32, 1.0, seed=11,
          path=("tiled_2sm", True))


def test_fused_epilogue_quick_return(g, orc):
    """K == 0: C = act(beta * C + bias)."""
    for act, beta in itertools.product(ACTS, (0.0, 1.5)):
        _case(g, orc, 70, 90, 0, "N", "N", DT_F16, DT_F32, act, DT_BF16, beta, seed=act)


def test_fused_epilogue_rejects_bad_arguments(g):
    import mixed_precision_dense_sm_gb300 as lib
    A = torch.ones((8, 8), dtype=torch.float16, device="cuda")
    C = torch.full((8, 8), 2.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for bias_dt, act in [(DT_F32, 9), (7, 0), (DT_F32, -1)]:
        st = lib.gemm_run_ex(g.h, "N", "N", 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0,
                             C.data_ptr(), 8, (DT_F16, DT_F16, DT_F32), C.data_ptr(), bias_dt,
                             act, s)
        assert st == 1
    g.sync()
    assert torch.all(C == 2.0)


def test_gelu_and_silu_evaluation_error(g, orc):
    """A K = 1 GEMM with A = x (a dense grid of exactly representable values)
    and B = 1 makes the accumulator exactly x, so the output isolates the
    activation's evaluation.  GELU = x Phi(x) through erfc (Numerical Recipes'
    erfcc, fractional error < 1.2e-7) in the form without cancellation, its
    reciprocal approximate and its exponential the fast 2^(x log2 e), whose
    error grows like the argument |u^2| 2^-23 (u = |x| / sqrt 2), plus the
    FP32 rounding of u^2 itself: relative error <= (u^2 + 2) 2^-21 + 3e-7
    (twice the analysis, for the fast exponential).  SiLU = x / (1 + exp(-x))
    with the fast exponential: bound |silu(x)| (|x| 2^-23 + 16 * 2^-24).
    Results below FP32's normal range may flush to zero (1e-30 floor)."""
    xs = np.arange(-2048, 2049, dtype=np.float64) / 128.0          # [-16, 16], exact in FP16
    M, N, K = xs.size, 8, 1
    A = torch.tensor(xs, dtype=torch.float16).view(M, 1)
    B = torch.ones((1, N), dtype=torch.float16)
    for act in (2, 3):
        C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        g(A.cuda(), B.cuda(), C, "N", "N", 1.0, 0.0, act=act)
        g.sync()
        got = C[:, 0].cpu().double().numpy()
        want = np.array([orc.activation(act, x) for x in xs])
        if act == 2:
            bound = np.abs(want) * ((xs * xs / 2 + 2) * 2.0 ** -21 + 3e-7) + 1e-30
        else:
            bound = np.abs(want) * (np.abs(xs) * 2.0 ** -23 + 16 * 2.0 ** -24) + 1e-30
        err = np.abs(got - want)
        assert (err <= bound).all(), (act, xs[np.argmax(err / bound)], float(np.max(err / bound)))


@pytest.mark.parametrize("c_dtype", [DT_F16, DT_BF16], ids=["f16", "bf16"])
def test_gelu_16bit_output_within_one_ulp(g, orc, c_dtype):
    """GELU into a 16-bit output on [-12, 16], its negative tail included
    (GELU(-5) is about -1.4e-6, an FP16 subnormal; GELU(-12) about -2e-32, a
    BF16 normal; below about -13 GELU leaves FP32's normal range, where the
    fast exponential flushes it to zero): with no cancellation in the kernel's
    form, every output is within one ulp of the oracle's correctly rounded
    value."""
    xs = np.arange(-1536, 2049, dtype=np.float64) / 128.0
    M, N, K = xs.size, 8, 1
    A = torch.tensor(xs, dtype=torch.float16).view(M, 1)
    B = torch.ones((1, N), dtype=torch.float16)
    C = torch.zeros((M, N), dtype=workloads.TORCH_DTYPE[c_dtype], device="cuda")
    g(A.cuda(), B.cuda(), C, "N", "N", 1.0, 0.0, act=2)
    g.sync()
    got = C[:, 0].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    want = orc.round_output(np.array([orc.activation(2, x) for x in xs]), c_dtype)

    def ordered(c):
        c = c.astype(np.int64)
        return np.where(c & 0x8000, -(c & 0x7FFF), c)
    dist = np.abs(ordered(got) - ordered(want))
    assert dist.max() <= 1, (xs[np.argmax(dist)], int(dist.max()))
