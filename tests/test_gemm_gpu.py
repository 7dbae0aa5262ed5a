"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle."""
import dataclasses
import itertools

import numpy as np
import pytest
import torch

import gpu_cases as gc
import workloads
from workloads import DT_BF16, DT_F16, DT_F32, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import mixed_precision_dense_sm_gb300 as lib
    h = lib.Gemm()
    yield h
    h.close()


def W(M, N, K, ta="N", tb="N", ab=DT_F16, c=DT_F32, alpha=1.0, beta=0.0, lda=None, ldb=None,
      ldc=None, dist="N1", seed=0, name=None):
    return Workload(name or f"{M}x{N}x{K}_{ta}{tb}", M, N, K, ta, tb, ab, c, alpha, beta,
                    dist, dist, dist if beta != 0 else None, lda, ldb, ldc, seed)


def test_layout_4x4_block(g, orc):
    """A 4 x 4 block first (DeepGEMM page, section 4.4): distinct small integers
    in every position, every transpose pair, both input types, exact."""
    for ta, tb, ab in itertools.product("NT", "NT", (DT_F16, DT_BF16)):
        w = W(4, 4, 4, ta, tb, ab, DT_F32)
        A = torch.arange(16, dtype=torch.float32).view(4, 4) - 7
        B = (torch.arange(16, dtype=torch.float32).view(4, 4) * 3) % 11 - 5
        t = workloads.TORCH_DTYPE[ab]
        inp = workloads.Inputs(A.to(t), B.to(t), None, 4, 4, 4)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


SIZES = [1, 2, 3, 15, 16, 17, 63, 64, 65, 127, 128, 129]


def _tiny_cases():
    rng = np.random.default_rng(5)
    cases = []
    for n in range(72):
        M, N, K = (int(rng.choice(SIZES)) for _ in range(3))
        ta, tb = "NT"[n % 2], "NT"[(n // 2) % 2]
        ab = (DT_F16, DT_BF16)[(n // 4) % 2]
        c = (DT_F32, DT_F16, DT_BF16)[n % 3]
        cases.append((M, N, K, ta, tb, ab, c))
    return cases


@pytest.mark.parametrize("integer", [True, False], ids=["integer_exact", "random_tol"])
def test_tiny_shapes(g, orc, integer):
    """Tiny ragged shapes across every transpose pair and type combination.
    Integer inputs keep every FP32 partial sum exact, so the result must be
    bit-identical to the oracle's correctly rounded value."""
    for (M, N, K, ta, tb, ab, c) in _tiny_cases():
        beta = 0.0 if (M + N) % 2 else 1.0
        w = W(M, N, K, ta, tb, ab, c, alpha=1.0 if integer else 0.75, beta=beta, seed=M * N + K)
        inp = gc.integer_inputs(w) if integer else workloads.make_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=integer)


MEDIUM = [
    (300, 520, 1000), (257, 129, 4096), (129, 300, 777), (1000, 1023, 777),
    (5, 300, 700), (64, 1000, 513), (33, 128, 2048), (640, 768, 320),
]


@pytest.mark.parametrize("M,N,K", MEDIUM, ids=[f"{m}x{n}x{k}" for m, n, k in MEDIUM])
def test_medium_integer_exact(g, orc, M, N, K):
    """Several tiles with ragged tails (data-parallel, stream-K and skinny
    paths); integer inputs, bit-exact against the oracle."""
    for ta, tb in itertools.product("NT", "NT"):
        c = (DT_F32, DT_BF16, DT_F16)[(M + N + K) % 3]
        w = W(M, N, K, ta, tb, DT_BF16 if K % 2 else DT_F16, c, beta=1.0 if K % 3 == 0 else 0.0)
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


# The strict one-ulp rate that FP32 accumulation in the tensor core permits
# for 16-bit outputs.  Rounding the FP32 sum once more can leave the correctly
# rounded value by one ulp, and by more only where the accumulation error
# exceeds an output ulp, i.e. for outputs far below their S = sum |a b|.  The
# tensor core does not add in round-to-nearest FP32: its multi-term adder
# aligns every term of an MMA step to the largest one and truncates the bits
# below (M. Fasi, N. J. Higham, M. Mikaitis, S. Pranesh, "Numerical behavior
# of NVIDIA tensor cores", PeerJ Computer Science, 2021), so the error grows
# faster with K than a round-to-nearest sum.  A simulation of that model on
# each workload's value distributions (0 to 3 extra bits) predicts
# 0.9995-0.9998 for the 1024^3 FP16 case, 0.9965-0.999 for the skinny FP16
# case (K = 8192, values N(0,1) x N(0,0.02)) and 0.9998-1.0 for the BF16
# layer GEMMs; the floors sit below those ranges.  The measured rates, and
# cuBLAS's on the same inputs for context, are printed.
STRICT_FLOOR = {"square1024_f16_nt_f16out": 0.999, "skinny_64x16384x8192_f16": 0.995,
                "linear_8192x4096x4096_bf16": 0.999, "linear_8192x14336x4096_bf16": 0.999,
                "linear_8192x4096x14336_bf16": 0.999}

FULL = ["square256_f16_f32out", "square1024_f16_nt_f16out", "ragged1000x1023x777_bf16_beta1",
        "skinny_64x16384x8192_f16", "linear_8192x4096x4096_bf16", "linear_8192x14336x4096_bf16",
        "linear_8192x4096x14336_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full(g, orc, name):
    """The named workloads at full size -- including the three transformer-layer
    GEMMs in the launch configuration bench.py times -- every output element
    checked against the oracle; 16-bit outputs also keep the strict one-ulp
    rate above its floor."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    C = gc.run_gpu(g, w, inp)
    keep = {}
    stats = gc.check_full(orc, w, inp, C, keep=keep)
    if w.c_dtype != DT_F32:
        stats["cublas_strict_1ulp_frac"] = gc.cublas_strict_frac(w, inp, keep["codes"])
    print(name, stats)
    if w.c_dtype != DT_F32:
        assert stats["strict_1ulp_frac"] >= STRICT_FLOOR[name], stats


@pytest.mark.parametrize("M", [96, 128])
@pytest.mark.parametrize("N,K", [(14336, 4096), (16384, 8192)], ids=["swapped", "tiled"])
def test_decode_batch_up_to_128_rows(g, orc, M, N, K):
    """Decode batches of 96 and 128 tokens (FP16, weights N x K, FP16 out) on
    both plans the planner picks between for 64 < M <= 128: swapped stream-K
    (14336 x 4096) and unswapped one-row tiles (16384 x 8192); every output
    element against the oracle, and integer inputs bit-exact."""
    import mixed_precision_dense_sm_gb300 as lib
    w = W(M, N, K, "N", "T", DT_F16, DT_F16, name=f"decode_{M}x{N}x{K}")
    w = dataclasses.replace(w, b_dist="N002")
    st, p = lib.gemm_plan_query("N", "T", M, N, K, 1.0, 256, K, 256, K, 0.0, 256, N,
                                (DT_F16, DT_F16, DT_F16),
                                num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and p["swap_ab"] == (1 if N == 14336 else 0), p
    inp = workloads.make_inputs(w)
    C = gc.run_gpu(g, w, inp)
    stats = gc.check_full(orc, w, inp, C)
    assert stats["strict_1ulp_frac"] >= 0.995, stats
    inp = gc.integer_inputs(w, -4, 4)
    C = gc.run_gpu(g, w, inp)
    gc.check_full(orc, w, inp, C, exact=True)


@pytest.mark.parametrize("name", ["linear_8192x4096x14336_bf16", "linear_8192x14336x4096_bf16"])
def test_workload_integer_exact(g, orc, name):
    """A transformer-layer GEMM at full size with integer inputs in [-8, 8]:
    every FP32 partial sum is an integer below 2^24 (at most K * 64), so the
    BF16 output must equal the oracle's correctly rounded value bit for bit
    on every element (wave boundaries, raster and the TMA-store epilogue
    included)."""
    w = workloads.WORKLOADS[name]
    inp = gc.integer_inputs(w)
    C = gc.run_gpu(g, w, inp)
    gc.check_full(orc, w, inp, C, exact=True)


def test_padded_leading_dimensions(g, orc):
    """lda/ldb/ldc larger than the rows: NaN in the operand padding must not be
    read, the C padding (canary) must not be written."""
    for ta, tb in itertools.product("NT", "NT"):
        for (M, N, K) in [(200, 300, 150), (64, 256, 96)]:
            a_cols = K if ta == "N" else M
            b_cols = N if tb == "N" else K
            w = W(M, N, K, ta, tb, DT_BF16, DT_BF16, beta=1.0, lda=a_cols + 8,
                  ldb=b_cols + 16, ldc=N + 8)
            inp = workloads.make_inputs(w)
            C = gc.run_gpu(g, w, inp)
            gc.check_full(orc, w, inp, C)


def test_unaligned_pitch_and_base(g, orc):
    """Leading dimensions that are not a multiple of 8 elements and base
    addresses that are not 16-byte aligned go through the pack pre-pass."""
    for ta, tb in itertools.product("NT", "NT"):
        M, N, K = 150, 201, 333
        a_cols = K if ta == "N" else M
        b_cols = N if tb == "N" else K
        w = W(M, N, K, ta, tb, DT_F16, DT_F32, beta=1.0, lda=a_cols + 1, ldb=b_cols + 3,
              ldc=N + 1)
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp, misalign=True)
        gc.check_full(orc, w, inp, C, exact=True)


def test_quick_returns(g, orc):
    import mixed_precision_dense_sm_gb300 as lib
    # M == 0 / N == 0: nothing touched
    C = torch.full((4, 4), 7.0, device="cuda")
    A = torch.ones((4, 4), dtype=torch.float16, device="cuda")
    g(A, A, C, M=0, N=4, K=4)
    g(A, A, C, M=4, N=0, K=4)
    g.sync()
    assert torch.all(C == 7.0)
    # K == 0: C = beta * C, A and B not read (NULL allowed)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.gemm_run(g.h, "N", "N", 4, 4, 0, 1.0, 0, 1, 0, 4, 0.5, C.data_ptr(), 4,
                      (DT_F16, DT_F16, DT_F32), s)
    assert st == 0
    g.sync()
    assert torch.all(C == 3.5)
    # alpha == 0, beta == 0: zeros even when C held NaN
    C.fill_(float("nan"))
    st = lib.gemm_run(g.h, "N", "N", 4, 4, 4, 0.0, 0, 4, 0, 4, 0.0, C.data_ptr(), 4,
                      (DT_F16, DT_F16, DT_F32), s)
    assert st == 0
    g.sync()
    assert torch.all(C == 0.0)


def test_invalid_arguments_enqueue_nothing(g):
    import mixed_precision_dense_sm_gb300 as lib
    C = torch.full((8, 8), 3.0, device="cuda")
    A = torch.ones((8, 8), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    bad = [
        dict(ta="X"), dict(M=-1), dict(lda=7), dict(ldb=7), dict(ldc=7),
        dict(dts=(DT_F16, DT_BF16, DT_F32)), dict(dts=(DT_F32, DT_F16, DT_F32)),
        dict(dts=(DT_F16, DT_F16, 9)), dict(a=0), dict(c=0),
        dict(a=A.data_ptr() + 1), dict(c=C.data_ptr() + 2),
    ]
    for b in bad:
        kw = dict(ta="N", M=8, lda=8, ldb=8, ldc=8, dts=(DT_F16, DT_F16, DT_F32),
                  a=A.data_ptr(), c=C.data_ptr())
        kw.update(b)
        st = lib.gemm_run(g.h, kw["ta"], "N", kw["M"], 8, 8, 1.0, kw["a"], kw["lda"],
                          A.data_ptr(), kw["ldb"], 0.0, kw["c"], kw["ldc"], kw["dts"], s)
        assert st == 1, (b, st)
    g.sync()
    assert torch.all(C == 3.0)


def test_deterministic_and_stream(g, orc):
    """Bitwise-identical results on repeated calls (the stream-K fixup adds
    partial sums in a fixed order), on a non-default stream."""
    w = W(1000, 1023, 777, "N", "N", DT_BF16, DT_F32, beta=1.0)
    inp = workloads.make_inputs(w)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(5):
        with torch.cuda.stream(s):
            outs.append(gc.run_gpu(g, w, inp, stream=s.cuda_stream).cpu())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    gc.check_full(orc, w, inp, outs[0].cuda())


PAIR_SHAPES = [(1900, 4736, 200), (2048, 4864, 136), (4096, 4096, 64)]


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in PAIR_SHAPES])
def test_cta_pair_tiles_integer_exact(g, orc, M, N, K):
    """Shapes large enough for 256 x 256 CTA-pair tiles, every transpose pair,
    bit-exact with integer inputs.  1900 x 4736 puts the odd CTA's half of the
    last tile row (rows 1920+) and of the last tile column (columns 4736+)
    wholly outside the matrix."""
    import mixed_precision_dense_sm_gb300 as lib
    for ta, tb in itertools.product("NT", "NT"):
        c = (DT_BF16, DT_F32, DT_F16, DT_BF16)["NT".index(ta) * 2 + "NT".index(tb)]
        w = W(M, N, K, ta, tb, DT_BF16 if ta == tb else DT_F16, c,
              beta=1.0 if ta == "T" else 0.0)
        lda, ldb, ldc = w.lds()
        st, plan = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, 256, lda, 256, ldb, w.beta, 256, ldc,
                                       (w.ab_dtype, w.ab_dtype, w.c_dtype),
                                       num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert st == 0 and plan["path_name"] == "tiled_2sm", plan
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


TMA_STORE_CASES = [
    # (M, N, K, transA, transB, input, output, path, ldc): ragged M and N, each output type
    (777, 1000, 2048, "N", "N", DT_F16, DT_F32, "tiled_2sm", None),   # CTA pairs (stream-K,
                                                                       # no split), FP32 C
    (5000, 1800, 96, "T", "N", DT_BF16, DT_BF16, "tiled_2sm", 1808),  # pairs; the last pair's odd
                                                                       # CTA (rows 5120+) stores
                                                                       # nothing; C pitch > N
    (200, 40008, 64, "N", "T", DT_F16, DT_F16, "tiled_1sm", None),    # 256-wide tiles, 2+ per SM
    (1000, 1000, 2048, "N", "T", DT_F32, DT_F32, "tiled_1sm", None),  # TF32 inputs
]


@pytest.mark.parametrize("M,N,K,ta,tb,ab,c,path,ldc", TMA_STORE_CASES,
                         ids=[f"{m}x{n}x{k}" for m, n, k, *_ in TMA_STORE_CASES])
def test_tma_store_epilogue_integer_exact(g, orc, M, N, K, ta, tb, ab, c, path, ldc):
    """C staged in shared memory (128-byte swizzle) and written by TMA stores of
    128-row boxes, the boxes clipped at M and N: bit-exact with integer inputs,
    and the canary columns between N and the C pitch untouched."""
    import mixed_precision_dense_sm_gb300 as lib
    w = W(M, N, K, ta, tb, ab, c, ldc=ldc)
    lda, ldb, ldc = w.lds()
    st, plan = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, 256, lda, 256, ldb, 0.0, 256, ldc,
                                   (ab, ab, c),
                                   num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == 0 and plan["c_tma"] == 1 and plan["path_name"] == path, plan
    inp = gc.integer_inputs(w)
    C = gc.run_gpu(g, w, inp)
    gc.check_full(orc, w, inp, C, exact=True)


BALANCE_SHAPES = [(2560, 1000, 4096, "tiled_2sm", 256), (20480, 256, 2048, "tiled_2sm", 256),
                  (200, 3072, 4096, "tiled_1sm", 256), (2048, 256, 4096, "tiled_1sm", 128)]


@pytest.mark.parametrize("M,N,K,path,bn", BALANCE_SHAPES,
                         ids=[f"{m}x{n}x{k}" for m, n, k, _, _ in BALANCE_SHAPES])
def test_wave_balancing_stream_k_integer_exact(g, orc, M, N, K, path, bn):
    """Shapes whose data-parallel schedule would leave most SMs idle run
    stream-K: over 256 x 256 CTA-pair tiles when M has 256 rows -- 2560 x 1000
    with fewer tiles than pairs (tiles split up to three ways, each CTA of the
    finishing pair summing its own half), 20480 x 256 with more (each pair's
    range then spans whole tiles as well as split ones) -- else over
    single-CTA tiles.  Bit-exact with integer inputs."""
    import mixed_precision_dense_sm_gb300 as lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ta, tb in (("N", "T"), ("T", "N")):
        w = W(M, N, K, ta, tb, DT_BF16, DT_F32 if ta == "N" else DT_BF16,
              beta=1.0 if ta == "T" else 0.0)
        lda, ldb, ldc = w.lds()
        st, plan = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, 256, lda, 256, ldb, w.beta, 256, ldc,
                                       (w.ab_dtype, w.ab_dtype, w.c_dtype), num_sms=sms)
        assert st == 0 and plan["sk_len"] > 0, plan
        assert (plan["path_name"], plan["block_n"]) == (path, bn), plan
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)
