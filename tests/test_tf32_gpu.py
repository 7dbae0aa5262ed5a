"""GPU parity for FP32 inputs computed as TF32 (the third input format of the
CATLASS page, section 3.2): the CUDA path through the C ABI against the
oracle, which cuts every FP32 input to TF32's 10-bit mantissa."""
import itertools
import struct

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


def W(M, N, K, ta="N", tb="N", c=DT_F32, alpha=1.0, beta=0.0, lda=None, ldb=None, ldc=None,
      dist="N1", seed=0):
    return Workload(f"tf32_{M}x{N}x{K}_{ta}{tb}", M, N, K, ta, tb, DT_F32, c, alpha, beta,
                    dist, dist, dist if beta != 0 else None, lda, ldb, ldc, seed)


def f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_low_mantissa_bits_are_dropped(g, orc):
    """Inputs that differ from a TF32 value only below TF32's 10-bit mantissa.
    Truncation (the oracle's reading) and round-to-nearest give different,
    exactly representable sums here, so the result tells them apart:
      1 + 3*2^-12 -> 1 (nearest would give 1 + 2^-10),
      1 + 2^-10 + 2^-11 + 2^-13 -> 1 + 2^-10 (nearest: 1 + 2^-9),
      -(2 - 2^-23) -> -(2 - 2^-10) (nearest: -2)."""
    vals = [f32(0x3F801800), f32(0x3F80_0000 | (1 << 13) | (1 << 12) | (1 << 10)),
            f32(0xBFFFFFFF), 3.0]
    K = len(vals)
    for ta, tb in itertools.product("NT", "NT"):
        w = W(1, 1, K, ta, tb)
        A = torch.tensor(vals, dtype=torch.float32).view(1, K)
        if ta == "T":
            A = A.view(K, 1).contiguous()
        B = torch.ones((K, 1) if tb == "N" else (1, K), dtype=torch.float32)
        inp = workloads.Inputs(A, B, None, A.shape[1], B.shape[1], 1)
        C = gc.run_gpu(g, w, inp)
        got = float(C[0, 0])
        want = 1.0 + (1.0 + 2.0 ** -10) - (2.0 - 2.0 ** -10) + 3.0
        assert got == want, (ta, tb, got, want)
        gc.check_full(orc, w, inp, C, exact=True)


def test_layout_4x4_block(g, orc):
    """Distinct small integers in every position, every transpose pair,
    every output type, exact (DeepGEMM page, section 4.4)."""
    for ta, tb, c in itertools.product("NT", "NT", (DT_F32, DT_F16, DT_BF16)):
        w = W(4, 4, 4, ta, tb, c)
        A = torch.arange(16, dtype=torch.float32).view(4, 4) - 7
        B = (torch.arange(16, dtype=torch.float32).view(4, 4) * 3) % 11 - 5
        inp = workloads.Inputs(A, B, None, 4, 4, 4)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


SHAPES = [(1, 1, 1), (3, 17, 33), (17, 3, 31), (64, 128, 64), (129, 65, 100),
          (300, 520, 1000), (257, 129, 4096), (1000, 1023, 777), (5, 300, 700),
          (64, 1000, 513), (33, 128, 2048), (640, 768, 320)]


@pytest.mark.parametrize("M,N,K", SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SHAPES])
def test_integer_exact(g, orc, M, N, K):
    """Tiny to medium ragged shapes on every planner path (single-CTA tiles
    of each width, stream-K, the swapped skinny path), every transpose pair;
    integer inputs are exact in TF32, so the result is bit-exact."""
    for ta, tb in itertools.product("NT", "NT"):
        c = (DT_F32, DT_BF16, DT_F16)[(M + N + K) % 3]
        w = W(M, N, K, ta, tb, c, beta=1.0 if K % 3 == 0 else 0.0, seed=M + N + K)
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


@pytest.mark.parametrize("M,N,K", [(300, 520, 1000), (1000, 1023, 777), (64, 4096, 2048),
                                   (2048, 4864, 200)])
def test_random_full(g, orc, M, N, K):
    """Normal inputs with all 23 mantissa bits in use: every output element
    against the oracle's TF32 result (FP32 accumulation bound)."""
    for ta, tb in itertools.product("NT", "NT"):
        w = W(M, N, K, ta, tb, beta=0.5 if ta == tb else 0.0, alpha=0.75, seed=K)
        inp = workloads.make_inputs(w)
        C = gc.run_gpu(g, w, inp)
        stats = gc.check_full(orc, w, inp, C)
        print(M, N, K, ta, tb, stats)


def test_cta_pair_tiles(g, orc):
    """Large enough for 256 x 256 CTA-pair tiles; ragged in M and N."""
    import mixed_precision_dense_sm_gb300 as lib
    M, N, K = 1900, 4736, 200
    for ta, tb in itertools.product("NT", "NT"):
        w = W(M, N, K, ta, tb, DT_F32, beta=1.0 if ta == "T" else 0.0)
        lda, ldb, ldc = w.lds()
        st, plan = lib.gemm_plan_query(ta, tb, M, N, K, 1.0, 256, lda, 256, ldb, w.beta, 256, ldc,
                                       (DT_F32, DT_F32, DT_F32),
                                       num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert st == 0 and plan["path_name"] == "tiled_2sm", plan
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C, exact=True)


def test_padded_and_unaligned(g, orc):
    """Pitches that are not a multiple of 4 elements and bases that are not
    16-byte aligned (the pack pre-pass); NaN padding must not be read and
    C's padding must survive."""
    for ta, tb in itertools.product("NT", "NT"):
        M, N, K = 150, 201, 333
        a_cols = K if ta == "N" else M
        b_cols = N if tb == "N" else K
        w = W(M, N, K, ta, tb, DT_F32, beta=1.0, lda=a_cols + 1, ldb=b_cols + 3, ldc=N + 1)
        inp = gc.integer_inputs(w)
        C = gc.run_gpu(g, w, inp, misalign=True)
        gc.check_full(orc, w, inp, C, exact=True)
        w = W(M, N, K, ta, tb, DT_BF16, beta=0.0, lda=a_cols + 4, ldb=b_cols + 8, ldc=N + 8)
        inp = workloads.make_inputs(w)
        C = gc.run_gpu(g, w, inp)
        gc.check_full(orc, w, inp, C)


def test_workload_full(g, orc):
    """The TF32 linear layer at full size, every output element checked."""
    w = workloads.WORKLOADS["tf32_linear_8192x4096x4096_f32out"]
    inp = workloads.make_inputs(w)
    C = gc.run_gpu(g, w, inp)
    stats = gc.check_full(orc, w, inp, C)
    print(w.name, stats)
