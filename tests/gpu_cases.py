"""Shared helpers for the GPU parity tests: build seeded inputs, run the CUDA
path through the C ABI, run the oracle on the same bit patterns, compare."""
from __future__ import annotations

import numpy as np
import torch

import checks
import workloads
from workloads import DT_F16, DT_BF16, DT_F32, TORCH_DTYPE

CANARY = 1234.5   # written into C's padding columns; must survive every call


def integer_inputs(w: workloads.Workload, lo=-8, hi=8):
    """Like workloads.make_inputs, but entries are integers in [lo, hi]."""
    gen = torch.Generator().manual_seed(w.seed + 1000)
    lda, ldb, ldc = w.lds()

    def mk(shape, ld, dt):
        v = torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)
        buf = torch.full((shape[0], ld), float("nan"), dtype=dt)
        buf[:, :shape[1]] = v.to(dt)
        return buf

    ab = TORCH_DTYPE[w.ab_dtype]
    A = mk(w.a_shape(), lda, ab)
    B = mk(w.b_shape(), ldb, ab)
    C = mk((w.M, w.N), ldc, TORCH_DTYPE[w.c_dtype]) if w.c_dist is not None else None
    return workloads.Inputs(A, B, C, lda, ldb, ldc)


def to_device(t: torch.Tensor, misalign: bool = False) -> torch.Tensor:
    """Copy a stored (rows x ld) CPU tensor to the GPU; with misalign the view
    starts one element into its allocation (base address not 16-byte aligned)."""
    if not misalign:
        return t.cuda()
    rows, ld = t.shape
    flat = torch.empty(rows * ld + 8, dtype=t.dtype, device="cuda")
    view = flat[1:1 + rows * ld].view(rows, ld)
    view.copy_(t)
    return view


def run_gpu(g, w: workloads.Workload, inp: workloads.Inputs, misalign=False, stream=None):
    """One gemm_run through the C ABI.  Returns the device C (stored M x ldc)."""
    A = to_device(inp.A, misalign)
    B = to_device(inp.B, misalign)
    cdt = TORCH_DTYPE[w.c_dtype]
    C = torch.full((w.M, inp.ldc), CANARY, dtype=cdt)
    if inp.C is not None:
        C[:, :w.N] = inp.C[:, :w.N]
    else:
        C[:, :w.N] = float("nan")        # beta == 0: C must not be read
    C = to_device(C, misalign)
    g(A, B, C, w.transA, w.transB, w.alpha, w.beta, M=w.M, N=w.N, K=w.K, stream=stream)
    g.sync(stream)
    return C


def oracle_full(orc, w, inp):
    A = workloads.as_codes(inp.A)
    B = workloads.as_codes(inp.B)
    C = None if inp.C is None else workloads.as_codes(inp.C)
    R, S = orc.gemm(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, inp.lda, B, inp.ldb,
                    w.beta, C, inp.ldc, w.ab_dtype, w.c_dtype)
    return R, S


def cin_values(w, inp):
    if inp.C is None:
        return None
    return inp.C[:, :w.N].to(torch.float64).numpy()


def check_full(orc, w, inp, Cdev, exact=False, keep=None):
    """Compare every output element with the oracle; returns the stats dict.
    With a dict `keep`, the oracle's output codes (16-bit C) are left in
    keep["codes"]."""
    R, S = oracle_full(orc, w, inp)
    vals, codes = checks.gpu_values(Cdev, w.M, w.N)
    ocodes = None if w.c_dtype == DT_F32 else orc.round_output(R, w.c_dtype)
    if keep is not None:
        keep["codes"] = ocodes
    if exact:
        if w.c_dtype == DT_F32:
            want = orc.round_output(R, DT_F32).astype(np.float64)
            bad = ~((vals == want) | (np.isnan(vals) & np.isnan(want)))
        else:
            bad = codes != ocodes
        assert not bad.any(), f"{w.name}: {int(bad.sum())} elements differ from the exact result"
        stats = {"n": int(bad.size), "fail": 0, "exact": True}
    else:
        stats, bad = checks.compare(vals, codes, R, S, cin_values(w, inp), w.alpha, w.beta,
                                    w.c_dtype, ocodes)
        if stats["fail"]:
            i, j = np.argwhere(bad)[0]
            raise AssertionError(f"{w.name}: {stats}; first bad ({i},{j}) gpu={vals[i, j]!r} "
                                 f"oracle={R[i, j]!r} S={S[i, j]!r}")
    check_canary(w, Cdev)
    return stats


def check_sampled(orc, w, inp, Cdev, nsamp=4096, seed=0):
    """Compare sampled outputs (random + first/last rows and columns)."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, w.M, nsamp))
    cols = list(rng.integers(0, w.N, nsamp))
    for j in rng.integers(0, w.N, 64):
        rows += [0, w.M - 1]
        cols += [int(j), int(j)]
    for i in rng.integers(0, w.M, 64):
        rows += [int(i), int(i)]
        cols += [0, w.N - 1]
    rows += [w.M - 1]
    cols += [w.N - 1]
    rows = np.array(rows, dtype=np.int64)
    cols = np.array(cols, dtype=np.int64)
    A = workloads.as_codes(inp.A)
    B = workloads.as_codes(inp.B)
    C = None if inp.C is None else workloads.as_codes(inp.C)
    R, S = orc.gemm_sampled(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, inp.lda, B, inp.ldb,
                            w.beta, C, inp.ldc, w.ab_dtype, w.c_dtype, rows, cols)
    blk = Cdev[torch.as_tensor(rows, device=Cdev.device), torch.as_tensor(cols, device=Cdev.device)]
    blk = blk.cpu()
    vals = blk.to(torch.float64).numpy()
    codes = None
    if blk.dtype != torch.float32:
        codes = blk.contiguous().view(torch.int16).numpy().view(np.uint16)
    ocodes = None if w.c_dtype == DT_F32 else orc.round_output(R, w.c_dtype)
    cin = None if inp.C is None else inp.C[rows, cols].to(torch.float64).numpy()
    stats, bad = checks.compare(vals, codes, R, S, cin, w.alpha, w.beta, w.c_dtype, ocodes)
    if stats["fail"]:
        k = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{w.name}: {stats}; first bad ({rows[k]},{cols[k]}) "
                             f"gpu={vals[k]!r} oracle={R[k]!r}")
    return stats


def check_canary(w, Cdev):
    ldc = Cdev.shape[1]
    if ldc > w.N:
        pad = Cdev[:, w.N:].float().cpu()
        want = torch.tensor(CANARY, dtype=Cdev.dtype).float()
        assert torch.all(pad == want), f"{w.name}: C padding columns were written"


def cublas_strict_frac(w, inp, want):
    """Context for the accuracy record: the strict one-ulp rate of cuBLAS
    (torch.matmul, FP32 accumulation, reduced-precision reductions off) on
    the same inputs against the oracle's codes `want`, for alpha = 1,
    beta = 0 problems (else None)."""
    if w.alpha != 1.0 or w.beta != 0.0:
        return None
    A, B = inp.A[:, :w.a_shape()[1]].cuda(), inp.B[:, :w.b_shape()[1]].cuda()
    opA = A if w.transA in "Nn" else A.t()
    opB = B if w.transB in "Nn" else B.t()
    m = torch.backends.cuda.matmul
    keep = (m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction)
    try:
        m.allow_fp16_reduced_precision_reduction = False
        m.allow_bf16_reduced_precision_reduction = False
        C = torch.matmul(opA, opB).to(TORCH_DTYPE[w.c_dtype])
    finally:
        m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction = keep
    torch.cuda.synchronize()
    got = C.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def ordered(c):
        c = c.astype(np.int64)
        return np.where(c & 0x8000, -(c & 0x7FFF), c)
    return float((np.abs(ordered(got) - ordered(want)) <= 1).mean())
