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


def softmax_bound(X, R, levels=16):
    """Per-element bound on |y_gpu - r| for the FP32 softmax with __expf.

    With t = x - max(x) per row: the kernel's exp(t) is within
    (2 + 1.16|t|) ulp of exp for __expf (CUDA's documented bound) plus the
    rounding of t itself (|t| 2^-24): eps_exp(t) <= (2 + 1.7|t|) 2^-23.  The
    row sum s inherits the exps' errors weighted by their share,
    W = sum_j e_j eps_exp(t_j) / s, once per merge level of the reduction tree
    (every partial's rescale exp(m_p - m) has |m_p - m| <= |t_j| for all its
    elements), plus at most `levels` FP32 additions and rescalings of
    2^-24 each and 32 more for a thread's own running sum.  The output adds
    one reciprocal and one product.  Values below FLT_MIN may flush to 0.
    X: float64 inputs (n, cols); R: the oracle's float64 result."""
    X = np.asarray(X, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        m = np.max(np.where(np.isnan(X), -np.inf, X), axis=1, keepdims=True)
        t = X - m
        e = np.exp(t)
        e = np.where(np.isfinite(e), e, 0.0)
        a = np.abs(np.where(np.isfinite(t), t, 0.0))
        eps_exp = np.where(e > 0, (2.0 + 1.7 * a) * 2.0 ** -23, 0.0)
        s = e.sum(axis=1, keepdims=True)
        W = np.where(s > 0, (e * eps_exp).sum(axis=1, keepdims=True) / np.where(s > 0, s, 1.0), 0.0)
    eps_s = (levels + 1) * W + (2 * levels + 32) * 2.0 ** -24
    return np.abs(R) * (eps_exp + eps_s + 3 * 2.0 ** -24) + 2.0 ** -126


def compare_softmax(gpu_vals, gpu_codes, R, X, y_dtype, oracle_codes=None):
    """FP32 output: within softmax_bound.  FP16/BF16 output: within one ulp
    of the correctly rounded oracle value, or within softmax_bound plus one
    output ulp.  NaN exactly where the oracle has NaN."""
    bound = softmax_bound(X, R)
    nan_r, nan_g = np.isnan(R), np.isnan(gpu_vals)
    err = np.abs(gpu_vals - R)
    with np.errstate(invalid="ignore"):
        if y_dtype == F32:
            ok = err <= bound
        else:
            dist = np.abs(_ordered(gpu_codes) - _ordered(oracle_codes))
            ok = (dist <= 1) | (err <= ulp_of(np.where(nan_r, 0.0, R), y_dtype) + bound)
    ok = np.where(nan_r | nan_g, nan_r & nan_g, ok)
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(nan_r | (R == 0), 0.0, err / np.abs(R))
    stats = {"n": int(ok.size), "fail": int((~ok).sum()),
             "max_rel_err": float(np.max(rel)) if rel.size else 0.0}
    return stats, ~ok


U32 = 2.0 ** -24          # unit roundoff of binary32


def layernorm_bound(H, S, Cin_vals, bias_vals, gamma_vals, shift_vals, alpha, beta, c_dtype,
                    eps, exact_h=False):
    """Per-element bound on |y_gpu - y| for LayerNorm after the linear layer,
    before the output's own rounding.  H, S: the oracle's h (as C's type holds
    it) and |product| sums, one row of N per selected row.

    1. h on the GPU is round_C(v) with |v - h_exact| <= a = the GEMM's FP32
       rule 1e-5 * (|alpha| S + |beta c| + |bias|) + 1e-6, so
       |h_gpu - H| <= e = a + ulp_C(|H| + a)  (0 for exact_h: integer inputs
       whose FP32 sums are exact).
    2. Through the row statistics: mean moves by at most mean(e); the biased
       variance by dv = (2/N) sum |h - mu| e + (1/N) sum e^2; sigma by at most
       dv / (sigma + sigma_lo), sigma_lo = sqrt(max(var - dv, 0) + eps).
       y - shift = gamma (h - mu) / sigma moves by
       |gamma| ((e + mean(e)) / sigma_lo + |h - mu| dv / (sigma sigma_lo (sigma + sigma_lo))).
    3. The FP32 evaluation on the GPU (with the GEMM rule for an FP32 sum of
       n terms: 1e-5 of the sum of magnitudes): mean off by
       dm = 1e-5 mean|h| + 1e-6, M2 relatively by 1e-5 + (dm/sigma)^2, then
       1/sqrt and three products, 3 roundings each:
       |gamma| (dm / sigma + |z| (0.5e-5 + (dm/sigma)^2 + 4u)) + 3u (|gamma z| + |shift|).
    """
    H = np.asarray(H, dtype=np.float64)
    n = H.shape[1]
    a = REL * (abs(alpha) * S) + ABS
    if beta != 0 and Cin_vals is not None:
        a = a + REL * np.abs(beta * Cin_vals)
    if bias_vals is not None:
        a = a + REL * np.abs(bias_vals)
    if exact_h:
        e = np.zeros_like(H)
    elif c_dtype == F32:
        e = a + U32 * 2 * (np.abs(H) + a)
    else:
        e = a + ulp_of(np.abs(H) + a, c_dtype)
    mu = H.mean(axis=1, keepdims=True)
    dev = np.abs(H - mu)
    var = (dev * dev).mean(axis=1, keepdims=True)
    sigma = np.sqrt(var + eps)
    ebar = e.mean(axis=1, keepdims=True)
    dv = 2.0 * (dev * e).mean(axis=1, keepdims=True) + (e * e).mean(axis=1, keepdims=True)
    sigma_lo = np.sqrt(np.maximum(var - dv, 0.0) + eps)
    g = np.ones_like(H) if gamma_vals is None else np.abs(np.asarray(gamma_vals))[None, :n]
    t = np.zeros_like(H) if shift_vals is None else np.abs(np.asarray(shift_vals))[None, :n]
    prop = g * ((e + ebar) / sigma_lo + dev * dv / (sigma * sigma_lo * (sigma + sigma_lo)))
    dm = REL * np.abs(H).mean(axis=1, keepdims=True) + ABS
    z = dev / sigma
    rm = (dm / sigma) ** 2
    arith = g * (dm / sigma + z * (0.5 * REL + rm + 4 * U32)) + 3 * U32 * (g * z + t)
    return prop + arith


def compare_layernorm(gpu_vals, gpu_codes, Y, bound, y_dtype, oracle_codes=None):
    """FP32 output: |y_gpu - y| <= bound.  FP16/BF16 output: within one ulp
    of the correctly rounded oracle value, or |y_gpu - y| <= bound plus one
    output ulp at |y| + bound."""
    err = np.abs(gpu_vals - Y)
    if y_dtype == F32:
        ok = err <= bound + U32 * np.abs(Y)
        stats = {}
    else:
        dist = np.abs(_ordered(gpu_codes) - _ordered(oracle_codes))
        strict = dist <= 1
        ok = strict | (err <= bound + ulp_of(np.abs(Y) + bound, y_dtype))
        stats = {"strict_1ulp_frac": float(strict.mean()) if strict.size else 1.0,
                 "max_ulp": int(dist.max()) if dist.size else 0}
    ok &= np.isfinite(gpu_vals)
    stats["n"] = int(ok.size)
    stats["fail"] = int((~ok).sum())
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / bound, 0.0)
    stats["max_err_over_bound"] = float(np.max(r)) if r.size else 0.0
    return stats, ~ok
