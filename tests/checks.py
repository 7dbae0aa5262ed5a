"""Acceptance rules for comparing a GPU result with the oracle (tests only).

FP32 output (absolute/relative bound on the FP32 accumulation):
    |C_gpu - r| <= 1e-5 * (|alpha| * S + |beta * c|) + 1e-6
FP16/BF16 output: pass when C_gpu is within 1 ulp of the correctly rounded
r (ordered-code distance <= 1), or when
    |C_gpu - r| <= ulp_out(r) + 1e-5 * (|alpha| * S + |beta * c|) + 1e-6,
the second clause covering FP32 accumulation noise that exceeds one output
ulp near zero.  r is the oracle's binary64 result and S = sum_k |a_ik b_kj|.
The strict one-ulp pass fraction is reported alongside.
"""
from __future__ import annotations

import numpy as np
import torch

F16, BF16, F32 = 0, 1, 2
REL, ABS = 1e-5, 1e-6


def gpu_values(C: torch.Tensor, M: int, N: int):
    """(float64 values, uint16 codes or None) of the logical M x N block."""
    block = C[:M, :N].detach().cpu()
    vals = block.to(torch.float64).numpy()
    codes = None
    if block.dtype in (torch.float16, torch.bfloat16):
        codes = block.contiguous().view(torch.int16).numpy().view(np.uint16)
    return vals, codes


def _ordered(codes: np.ndarray) -> np.ndarray:
    """Map sign-magnitude 16-bit codes to integers ordered like the values."""
    c = codes.astype(np.int64)
    return np.where(c & 0x8000, -(c & 0x7FFF), c)


def ulp_of(vals: np.ndarray, dtype: int) -> np.ndarray:
    """Spacing of the output format at |vals| (the ulp used by the loose rule)."""
    a = np.abs(vals)
    if dtype == F16:
        mbits, emin = 10, -14
    else:
        mbits, emin = 7, -126
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - mbits).astype(np.int64))


def compare(gpu_vals, gpu_codes, R, S, Cin_vals, alpha, beta, c_dtype, oracle_codes=None):
    """Returns a dict of statistics and a boolean mask of failing elements."""
    scale = abs(alpha) * S
    if beta != 0 and Cin_vals is not None:
        scale = scale + np.abs(beta * Cin_vals)
    bound = REL * scale + ABS
    err = np.abs(gpu_vals - R)
    nan_ok = np.isnan(gpu_vals) & np.isnan(R)
    if c_dtype == F32:
        ok = (err <= bound) | nan_ok
        inf_ok = np.isinf(gpu_vals) & np.isinf(R) & (np.sign(gpu_vals) == np.sign(R))
        ok |= inf_ok
        stats = {"max_err_over_S": float(np.max(err / np.maximum(scale, 1e-300))) if err.size else 0.0}
    else:
        assert oracle_codes is not None
        dist = np.abs(_ordered(gpu_codes) - _ordered(oracle_codes))
        strict = dist <= 1
        loose = err <= ulp_of(R, c_dtype) + bound
        ok = strict | loose | nan_ok
        stats = {"strict_1ulp_frac": float(strict.mean()) if strict.size else 1.0,
                 "max_ulp": int(dist.max()) if dist.size else 0}
    stats["n"] = int(ok.size)
    stats["fail"] = int((~ok).sum())
    return stats, ~ok


def compare_epilogue(gpu_vals, gpu_codes, R, S, Cin_vals, bias_vals, alpha, beta, c_dtype,
                     oracle_codes=None, slope=1.2, rel=2e-6):
    """Acceptance for act(alpha*AB + beta*C + bias): the pre-activation bound
    (the same FP32 rule, with |bias| added to the scale) times the largest
    slope of the activations (ReLU 1, SiLU ~1.1, GELU ~1.13), plus a relative
    term for the FP32 evaluation of erf/exp and the extra roundings."""
    scale = abs(alpha) * S
    if beta != 0 and Cin_vals is not None:
        scale = scale + np.abs(beta * Cin_vals)
    if bias_vals is not None:
        scale = scale + np.abs(bias_vals)
    bound = slope * (REL * scale + ABS) + rel * np.abs(R)
    err = np.abs(gpu_vals - R)
    nan_ok = np.isnan(gpu_vals) & np.isnan(R)
    if c_dtype == F32:
        ok = (err <= bound) | nan_ok
        stats = {}
    else:
        dist = np.abs(_ordered(gpu_codes) - _ordered(oracle_codes))
        strict = dist <= 1
        ok = strict | (err <= ulp_of(R, c_dtype) + bound) | nan_ok
        stats = {"strict_1ulp_frac": float(strict.mean()) if strict.size else 1.0}
    stats["n"] = int(ok.size)
    stats["fail"] = int((~ok).sum())
    return stats, ~ok
