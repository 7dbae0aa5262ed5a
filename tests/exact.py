"""Exact-arithmetic helpers for pinning the oracle (tests only).

Everything here is an independent restatement of the definitions, written
differently from oracle.c: values are exact rationals (fractions.Fraction),
decoding goes through the library's own FP16/BF16 -> float64 conversion, and
round-to-nearest-even picks between the two neighbouring codes of a sorted
table of every representable value instead of scaling onto a grid.
"""
from __future__ import annotations

import bisect
from fractions import Fraction

import numpy as np
import torch

F16, BF16, F32 = 0, 1, 2


def codes_to_float64(codes, dtype: int) -> np.ndarray:
    """Library decode (torch) of uint16 codes to float64."""
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint16).astype(np.int16).copy())
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    return t.view(tdt).to(torch.float64).numpy()


class _Table:
    """All non-negative finite codes of a format in increasing order, plus the
    infinity code treated as the value 2^(emax+1) (what RNE with an unbounded
    exponent range would produce on overflow)."""

    def __init__(self, dtype: int):
        if dtype == F16:
            inf_code, past_max = 0x7C00, Fraction(2) ** 16
        else:
            inf_code, past_max = 0x7F80, Fraction(2) ** 128
        codes = np.arange(0, inf_code, dtype=np.uint32).astype(np.uint16)
        vals = codes_to_float64(codes, dtype)
        self.codes = [int(c) for c in codes] + [inf_code]
        self.vals = [Fraction(float(v)) for v in vals] + [past_max]
        self.inf_code = inf_code


_TABLES = {}


def table(dtype: int) -> _Table:
    if dtype not in _TABLES:
        _TABLES[dtype] = _Table(dtype)
    return _TABLES[dtype]


def exact_round(x: Fraction, dtype: int) -> int:
    """Round-to-nearest-even of an exact rational to an FP16/BF16 code."""
    tb = table(dtype)
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a >= tb.vals[-1]:
        return sign | tb.inf_code
    hi = bisect.bisect_left(tb.vals, a)
    if tb.vals[hi] == a:
        return sign | tb.codes[hi]
    lo = hi - 1
    dlo, dhi = a - tb.vals[lo], tb.vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:                                   # tie: the code with an even last bit
        pick = lo if tb.codes[lo] % 2 == 0 else hi
    return sign | tb.codes[pick]


def op_matrix(stored: np.ndarray, rows: int, cols: int, trans: str) -> np.ndarray:
    """op(X) from the stored (rows x ld) buffer: the logical rows x cols block,
    transposed for 'T' (numpy slicing and .T, no index arithmetic)."""
    block = stored[:rows, :cols]
    return block.T if trans in "Tt" else block


def exact_gemm(opA: np.ndarray, opB: np.ndarray, alpha: float, beta: float, C):
    """r_ij = alpha * sum_k opA_ik opB_kj + beta * C_ij in exact rationals.
    opA, opB, C hold float64 values (exact decodes).  Returns (r, S) as
    nested lists of Fractions."""
    M, K = opA.shape
    K2, N = opB.shape
    assert K == K2
    al, be = Fraction(float(np.float32(alpha))), Fraction(float(np.float32(beta)))
    Af = [[Fraction(float(v)) for v in row] for row in opA]
    Bf = [[Fraction(float(v)) for v in row] for row in opB]
    r, S = [], []
    for i in range(M):
        rr, ss = [], []
        for j in range(N):
            prods = [Af[i][k] * Bf[k][j] for k in range(K)]
            acc = sum(prods, Fraction(0))
            v = al * acc if (K > 0 and al != 0) else Fraction(0)
            if be != 0:
                v += be * Fraction(float(C[i][j]))
            rr.append(v)
            ss.append(sum((abs(p) for p in prods), Fraction(0)))
        r.append(rr)
        S.append(ss)
    return r, S
