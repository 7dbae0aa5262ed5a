"""The battery of checks that pins the CPU oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages, the IEEE-754 format definitions
or plain mathematics fix.  ``test_oracle_pins.py`` runs every pin against the
real oracle (all must pass); ``test_oracle_mutants.py`` runs the battery against
builds of oracle.c with one planted mistake each (at least one pin must fail).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import exact
from exact import F16, BF16, F32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _to_codes(values, dtype):
    """float64 values that are exactly representable -> uint16 codes (torch)."""
    import torch
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    t = torch.tensor(np.asarray(values, dtype=np.float64)).to(tdt)
    back = t.to(torch.float64).numpy()
    ok = (back == np.asarray(values)) | (np.isnan(back) & np.isnan(values))
    assert ok.all(), "test input not representable"
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _random_codes(rng, shape, dtype, scale=1.0):
    import torch
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    v = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale).to(tdt)
    return v.view(torch.int16).numpy().view(np.uint16).copy()


def _stored(rng, rows, cols, ld, dtype, maker):
    """A rows x ld buffer with the logical block from `maker` and NaN padding."""
    buf = np.full((rows, ld), 0x7E00 if dtype == F16 else 0x7FC0, dtype=np.uint16)
    buf[:, :cols] = maker(rows, cols)
    return buf


# ----------------------------------------------------------------- formats

def pin_decode_exhaustive(o):
    """Every one of the 65536 FP16 and BF16 codes decodes to the value the
    library's own conversion gives (NaN codes to NaN)."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in (F16, BF16):
        mine = o.decode(codes, dt)
        lib = exact.codes_to_float64(codes, dt)
        same = (mine == lib) | (np.isnan(mine) & np.isnan(lib))
        assert same.all(), f"decode mismatch dtype={dt} at codes {np.flatnonzero(~same)[:5]}"
        # signed zeros keep their sign
        assert math.copysign(1.0, o.decode_scalar(0x8000, dt)) == -1.0


def pin_page_format_limits(o):
    """The printed format limits (CATLASS page, section 3.2)."""
    path = os.path.join(GOLDEN, "format_limits.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 5
    for fmt, qty, printed, code, tol in rows:
        dt = F16 if fmt == "f16" else BF16
        v = o.decode_scalar(int(code, 16), dt)
        assert abs(v - float(printed)) <= float(tol) * float(printed), (fmt, qty, v)
        if qty == "max":
            # the next code up is infinity: values past the maximum overflow
            assert math.isinf(o.decode_scalar(int(code, 16) + 1, dt))
            assert o.round_scalar(v, dt) == int(code, 16)
    # FP16: 65504 is the largest finite value; rounding past it goes to infinity
    assert o.round_scalar(65504.0, F16) == 0x7BFF
    assert o.round_scalar(1e6, F16) == 0x7C00


def pin_round_ieee_table(o):
    """Round-to-nearest-even facts that follow from the binary16/bfloat16
    definitions (ties go to the code with an even last bit)."""
    cases = [
        (65504.0, F16, 0x7BFF),
        (65519.99, F16, 0x7BFF),            # below the overflow midpoint
        (65520.0, F16, 0x7C00),             # the midpoint 65504..65536 ties to even -> inf
        (-65520.0, F16, 0xFC00),
        (2.0 ** -25, F16, 0x0000),          # half of the smallest subnormal ties to 0
        (3 * 2.0 ** -25, F16, 0x0002),      # 1.5 subnormal ulps ties up to 2 (even)
        (2.0 ** -24, F16, 0x0001),
        (1.0 + 2.0 ** -11, F16, 0x3C00),    # tie between 1 and 1+2^-10 -> 1 (even)
        (1.0 + 3 * 2.0 ** -11, F16, 0x3C02),
        (1.0, BF16, 0x3F80),
        (1.0 + 2.0 ** -8, BF16, 0x3F80),    # tie -> 1 (even)
        (1.0 + 3 * 2.0 ** -8, BF16, 0x3F82),  # tie -> 1 + 2^-6 (even)
        (-0.0, F16, 0x8000),
        (float("inf"), BF16, 0x7F80),
        (3.3961775292304455e38, BF16, 0x7F7F),  # bf16 max
        (3.4e38, BF16, 0x7F80),             # past max + half ulp -> inf
        (2.0 ** -133, BF16, 0x0001),        # smallest bf16 subnormal
        (2.0 ** -134, BF16, 0x0000),        # tie -> 0
    ]
    for x, dt, want in cases:
        got = o.round_scalar(x, dt)
        assert got == want, f"round({x!r}, {dt}) = {got:#06x}, want {want:#06x}"
    for dt in (F16, BF16):
        assert (o.round_scalar(float("nan"), dt) & 0x7FFF) > (0x7C00 if dt == F16 else 0x7F80)


def pin_round_roundtrip_exhaustive(o):
    """Every finite code, decoded by the library, rounds back to itself."""
    for dt in (F16, BF16):
        codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        vals = exact.codes_to_float64(codes, dt)
        fin = np.isfinite(vals)
        out = o.round_output(vals[fin], dt)
        # -0 and +0 both exist; the round trip keeps the sign bit
        assert (out == codes[fin]).all(), f"roundtrip mismatch dtype={dt}"


def pin_round_midpoints(o):
    """Exhaustive over adjacent positive codes: the exact midpoint ties to the
    even code, one double below it rounds down, one above rounds up."""
    for dt in (F16, BF16):
        tb = exact.table(dt)
        vals = [float(v) for v in tb.vals]
        lo = np.array(vals[:-1])
        hi = np.array(vals[1:])
        mid = (lo + hi) / 2.0          # exact: both are on a grid far coarser than binary64
        below = np.nextafter(mid, 0.0)
        above = np.nextafter(mid, np.inf)
        codes_lo = np.array(tb.codes[:-1], dtype=np.uint16)
        codes_hi = np.array(tb.codes[1:], dtype=np.uint16)
        even = np.where(codes_lo % 2 == 0, codes_lo, codes_hi)
        assert (o.round_output(mid, dt) == even).all(), f"midpoint ties dtype={dt}"
        assert (o.round_output(below, dt) == codes_lo).all(), f"below-midpoint dtype={dt}"
        assert (o.round_output(above, dt) == codes_hi).all(), f"above-midpoint dtype={dt}"
        assert (o.round_output(-above, dt) == (codes_hi | 0x8000)).all()


def pin_round_random_exact(o):
    """Random doubles over the whole range vs exact rational round-to-nearest-even."""
    rng = _rng(7)
    for dt, lo_e, hi_e in ((F16, -30, 18), (BF16, -140, 130)):
        e = rng.integers(lo_e, hi_e, 1500)
        x = rng.uniform(1.0, 2.0, 1500) * np.ldexp(1.0, e) * rng.choice([-1.0, 1.0], 1500)
        got = o.round_output(x, dt)
        want = np.array([exact.exact_round(Fraction(float(v)), dt) for v in x], dtype=np.uint16)
        assert (got == want).all(), f"random rounding dtype={dt}"


def pin_f32_output(o):
    """FP32 output is the IEEE double -> float conversion (numpy's cast)."""
    rng = _rng(8)
    x = rng.standard_normal(4000) * np.ldexp(1.0, rng.integers(-160, 140, 4000))
    x = np.concatenate([x, [3.5e38, -3.5e38, 1e-46, np.nan]])
    got = o.round_output(x, F32)
    want = x.astype(np.float32)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same.all()


# -------------------------------------------------------------------- GEMM

def _gemm_case(o, rng, M, N, K, ta, tb, dt, cdt, alpha, beta, pad, integer, sampled=False):
    a_rows, a_cols = (M, K) if ta == "N" else (K, M)
    b_rows, b_cols = (K, N) if tb == "N" else (N, K)
    lda, ldb, ldc = max(a_cols, 1) + pad, max(b_cols, 1) + pad, max(N, 1) + pad

    if integer:
        mk = lambda r, c: _to_codes(rng.integers(-8, 9, (r, c)).astype(np.float64), dt)
    else:
        mk = lambda r, c: _random_codes(rng, (r, c), dt)
    A = _stored(rng, a_rows, a_cols, lda, dt, mk)
    B = _stored(rng, b_rows, b_cols, ldb, dt, mk)
    C = None
    if beta != 0:
        if cdt == F32:
            C = np.full((M, ldc), np.nan, dtype=np.float32)
            cv = rng.integers(-8, 9, (M, N)) if integer else rng.standard_normal((M, N))
            C[:, :N] = cv.astype(np.float32)
        else:
            C = _stored(rng, M, N, ldc, cdt, mk)

    opA = exact.op_matrix(exact.codes_to_float64(A, dt), a_rows, a_cols, ta)
    opB = exact.op_matrix(exact.codes_to_float64(B, dt), b_rows, b_cols, tb)
    if C is None:
        Cv = np.zeros((M, N))
    elif cdt == F32:
        Cv = C[:, :N].astype(np.float64)
    else:
        Cv = exact.codes_to_float64(C, cdt)[:, :N]
    r_ex, s_ex = exact.exact_gemm(opA, opB, alpha, beta, Cv)

    if sampled:
        rows = np.array([i for i in range(M) for _ in range(N)], dtype=np.int64)
        cols = np.array([j for _ in range(M) for j in range(N)], dtype=np.int64)
        R, S = o.gemm_sampled(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              dt, cdt, rows, cols)
        R, S = R.reshape(M, N), S.reshape(M, N)
    else:
        R, S = o.gemm(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dt, cdt)

    for i in range(M):
        for j in range(N):
            ex, sx = r_ex[i][j], s_ex[i][j]
            scale = abs(Fraction(float(np.float32(alpha)))) * sx + \
                abs(Fraction(float(np.float32(beta))) * Fraction(float(Cv[i][j])))
            err = abs(Fraction(float(R[i, j])) - ex)
            if integer:
                assert err == 0, (i, j, float(ex), R[i, j])
            else:
                assert err <= Fraction(2) ** -48 * scale + Fraction(1, 2 ** 1000), \
                    (M, N, K, ta, tb, i, j, float(ex), R[i, j])
            assert abs(Fraction(float(S[i, j])) - sx) <= Fraction(2) ** -48 * sx, (i, j)
    if integer and cdt != F32:
        got = o.round_output(R, cdt)
        want = np.array([[exact.exact_round(r_ex[i][j], cdt) for j in range(N)]
                         for i in range(M)], dtype=np.uint16).reshape(M, N)
        assert (got == want).all()


def pin_gemm_bruteforce(o):
    """Tiny shapes against exact rational arithmetic: every transpose pair,
    both input formats, all output formats, alpha/beta, padded leading
    dimensions, full and sampled entry points."""
    rng = _rng(11)
    shapes = [(1, 1, 1), (2, 3, 5), (3, 2, 4), (5, 7, 3), (8, 8, 8), (4, 1, 7), (1, 6, 2)]
    n = 0
    for (M, N, K) in shapes:
        for ta in "NT":
            for tb in "NT":
                dt = (F16, BF16)[n % 2]
                cdt = (F32, F16, BF16)[n % 3]
                alpha = (1.0, -0.5, 3.0, 0.3)[n % 4]
                beta = (0.0, 1.0, -2.0, 0.7)[(n // 2) % 4]
                pad = (0, 3)[(n // 3) % 2]
                _gemm_case(o, rng, M, N, K, ta, tb, dt, cdt, alpha, beta, pad,
                           integer=False, sampled=(n % 5 == 4))
                n += 1


def pin_gemm_integer_exact(o):
    """Integer inputs make every sum exact: the oracle must equal the exact
    rational result bit for bit, and its FP16/BF16 outputs must be the exact
    round-to-nearest-even of it."""
    rng = _rng(12)
    n = 0
    for (M, N, K) in [(3, 4, 5), (6, 5, 8), (2, 9, 1)]:
        for ta in "NT":
            for tb in "NT":
                cdt = (F16, BF16, F32)[n % 3]
                _gemm_case(o, rng, M, N, K, ta, tb, (F16, BF16)[n % 2], cdt,
                           (1.0, 2.0, -1.0)[n % 3], (0.0, 1.0, -3.0)[(n + 1) % 3],
                           (0, 2)[n % 2], integer=True, sampled=(n % 4 == 1))
                n += 1


def pin_identity_and_permutation(o):
    """A * I = A and I * B = B exactly; A * P permutes columns exactly."""
    rng = _rng(13)
    for dt in (F16, BF16):
        M, K = 9, 12
        A = _random_codes(rng, (M, K), dt)
        Av = exact.codes_to_float64(A, dt)
        I = _to_codes(np.eye(K), dt)
        for tb in "NT":
            R, _ = o.gemm("N", tb, M, K, K, 1.0, A, K, I, K, 0.0, None, K, dt, dt)
            assert (R == Av).all()
            out = o.round_output(R, dt)
            assert (exact.codes_to_float64(out, dt) == Av).all()
        R, _ = o.gemm("N", "N", K, M, K, 1.0, I, K, A.T.copy(), M, 0.0, None, M, dt, dt)
        assert (R == Av.T).all()
        perm = rng.permutation(K)
        P = np.zeros((K, K))
        P[perm, np.arange(K)] = 1.0           # (A P)[:, j] = A[:, perm[j]]
        R, _ = o.gemm("N", "N", M, K, K, 1.0, A, K, _to_codes(P, dt), K, 0.0, None, K, dt, F32)
        assert (R == Av[:, perm]).all()


def pin_all_ones(o):
    """All-ones inputs: every entry equals K (and S equals K)."""
    for dt in (F16, BF16):
        for (M, N, K) in [(5, 7, 1), (4, 3, 257), (2, 2, 1000)]:
            A = _to_codes(np.ones((M, K)), dt)
            B = _to_codes(np.ones((N, K)), dt)
            R, S = o.gemm("N", "T", M, N, K, 1.0, A, K, B, K, 0.0, None, N, dt, F32)
            assert (R == K).all() and (S == K).all()


def pin_rank1_closed_form(o):
    """A_ik = x_i y_k, B_kj = y'_k z_j gives C_ij = x_i z_j sum_k y_k y'_k."""
    rng = _rng(14)
    vals = np.array([1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 4.0, 0.25])
    for dt in (F16, BF16):
        M, N, K = 6, 5, 33
        x, z = rng.choice(vals, M), rng.choice(vals, N)
        y, yp = rng.choice(vals, K), rng.choice(vals, K)
        A = _to_codes(np.outer(x, y), dt)
        B = _to_codes(np.outer(yp, z), dt)
        dot = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(y, yp))
        R, _ = o.gemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, dt, F32)
        want = np.array([[float(Fraction(float(xi)) * Fraction(float(zj)) * dot)
                          for zj in z] for xi in x])
        assert (R == want).all()


def pin_linearity(o):
    """A (B1 + B2) = A B1 + A B2 with integer entries (all sums exact)."""
    rng = _rng(15)
    for dt in (F16, BF16):
        M, N, K = 7, 6, 40
        A = _to_codes(rng.integers(-16, 17, (M, K)).astype(np.float64), dt)
        b1 = rng.integers(-16, 17, (K, N)).astype(np.float64)
        b2 = rng.integers(-16, 17, (K, N)).astype(np.float64)
        R1, _ = o.gemm("N", "N", M, N, K, 1.0, A, K, _to_codes(b1, dt), N, 0.0, None, N, dt, F32)
        R2, _ = o.gemm("N", "N", M, N, K, 1.0, A, K, _to_codes(b2, dt), N, 0.0, None, N, dt, F32)
        R12, _ = o.gemm("N", "N", M, N, K, 1.0, A, K, _to_codes(b1 + b2, dt), N, 0.0, None, N,
                        dt, F32)
        assert (R12 == R1 + R2).all()
        assert not (R1 == 0).all()


def pin_quick_returns(o):
    """K == 0 or alpha == 0 gives beta*C without reading A or B; beta == 0 never
    reads C (NaN in C does not propagate); M == 0 / N == 0 is a no-op."""
    rng = _rng(16)
    M, N = 4, 5
    C = rng.standard_normal((M, N)).astype(np.float32)
    R, S = o.gemm("N", "N", M, N, 0, 1.0, None, 1, None, N, 2.0, C, N, F16, F32)
    assert (R == 2.0 * C.astype(np.float64)).all() and (S == 0).all()
    A = _random_codes(rng, (M, 3), F16)
    B = _random_codes(rng, (3, N), F16)
    R, _ = o.gemm("N", "N", M, N, 3, 0.0, None, 3, None, N, -1.0, C, N, F16, F32)
    assert (R == -C.astype(np.float64)).all()
    Cnan = np.full((M, N), np.nan, dtype=np.float32)
    R, _ = o.gemm("N", "N", M, N, 3, 1.0, A, 3, B, N, 0.0, Cnan, N, F16, F32)
    assert np.isfinite(R).all()
    R, _ = o.gemm("N", "N", 0, N, 3, 1.0, A, 3, B, N, 0.0, None, N, F16, F32)
    assert R.shape == (0, N)


def pin_bad_arguments(o):
    """Invalid arguments are rejected, not computed."""
    A = np.zeros((4, 4), dtype=np.uint16)
    bad = [
        dict(ta="X"), dict(M=-1), dict(lda=3), dict(ldb=3), dict(ldc=3),
        dict(dt=5), dict(cdt=7),
    ]
    for b in bad:
        kw = dict(ta="N", tb="N", M=4, N=4, K=4, lda=4, ldb=4, ldc=4, dt=F16, cdt=F32)
        kw.update(b)
        try:
            o.gemm(kw["ta"], kw["tb"], kw["M"], kw["N"], kw["K"], 1.0, A, kw["lda"], A,
                   kw["ldb"], 0.0, None, kw["ldc"], kw["dt"], kw["cdt"])
        except ValueError:
            continue
        raise AssertionError(f"accepted bad arguments {b}")


def pin_threads_deterministic(o):
    """The result does not depend on the number of host threads."""
    rng = _rng(17)
    M, N, K = 37, 29, 65
    A = _random_codes(rng, (M, K), BF16)
    B = _random_codes(rng, (K, N), BF16)
    R1, S1 = o.gemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, BF16, F32, nthreads=1)
    R4, S4 = o.gemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, BF16, F32, nthreads=4)
    assert (R1 == R4).all() and (S1 == S4).all()


# ----------------------------------------------------------- fused epilogue

ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3


def pin_activation_values(o):
    """GELU = x * Phi(x) and SiLU = x * sigmoid(x) against scipy's own normal
    CDF and logistic routines; ReLU exactly; the odd-part identities
    act(x) - act(-x) = x that both GELU and SiLU satisfy."""
    from scipy.special import expit, ndtr
    rng = _rng(21)
    xs = np.concatenate([rng.standard_normal(500) * 4.0, [0.0, 1.0, -1.0, 8.0, -8.0, 30.0, -30.0]])
    for x in xs:
        g = o.activation(ACT_GELU, x)
        assert abs(g - x * ndtr(x)) <= 1e-14 * max(1.0, abs(x)), x
        s = o.activation(ACT_SILU, x)
        assert abs(s - x * expit(x)) <= 1e-14 * max(1.0, abs(x)), x
        assert abs((o.activation(ACT_GELU, x) - o.activation(ACT_GELU, -x)) - x) <= 1e-14 * max(1.0, abs(x))
        assert abs((o.activation(ACT_SILU, x) - o.activation(ACT_SILU, -x)) - x) <= 1e-14 * max(1.0, abs(x))
        assert o.activation(ACT_RELU, x) == (x if x > 0 else 0.0)
        assert o.activation(ACT_NONE, x) == x
    assert math.isnan(o.activation(ACT_RELU, float("nan")))
    assert o.activation(ACT_GELU, 0.0) == 0.0 and o.activation(ACT_SILU, 0.0) == 0.0
    # GELU's negative tail to full relative precision: x Phi(x) is tiny there
    # (about 1e-13 at x = -7.5, 1e-300 near x = -37), and a 16-bit output
    # rounds it relative to its own size, so the oracle must not lose it to
    # cancellation.  scipy's ndtr is accurate in the tail (via erfc).
    for x in np.concatenate([-np.linspace(1.0, 37.0, 400), [-5.0, -10.0, -20.0]]):
        want = x * ndtr(x)
        assert abs(o.activation(ACT_GELU, x) - want) <= 1e-12 * abs(want), x


def pin_epilogue_bruteforce(o):
    """act(alpha*AB + beta*C + bias) on tiny shapes: the GEMM part in exact
    rationals, the activation by scipy, every transpose pair."""
    from scipy.special import expit, ndtr
    ref_act = {ACT_NONE: lambda x: x, ACT_RELU: lambda x: max(x, 0.0),
               ACT_GELU: lambda x: x * ndtr(x), ACT_SILU: lambda x: x * expit(x)}
    rng = _rng(22)
    n = 0
    for (M, N, K) in [(3, 5, 4), (6, 2, 7), (1, 8, 3)]:
        for ta in "NT":
            for tb in "NT":
                dt = (F16, BF16)[n % 2]
                act = n % 4
                a_rows, a_cols = (M, K) if ta == "N" else (K, M)
                b_rows, b_cols = (K, N) if tb == "N" else (N, K)
                A = _random_codes(rng, (a_rows, a_cols), dt)
                B = _random_codes(rng, (b_rows, b_cols), dt)
                C = rng.standard_normal((M, N)).astype(np.float32)
                bias = _random_codes(rng, (N,), BF16)
                alpha, beta = (1.0, -0.5)[n % 2], (0.0, 1.0)[(n // 2) % 2]
                R, _ = o.gemm_ex(ta, tb, M, N, K, alpha, A, a_cols, B, b_cols, beta, C, N, dt,
                                 F32, bias, BF16, act)
                opA = exact.op_matrix(exact.codes_to_float64(A, dt), a_rows, a_cols, ta)
                opB = exact.op_matrix(exact.codes_to_float64(B, dt), b_rows, b_cols, tb)
                r_ex, _ = exact.exact_gemm(opA, opB, alpha, beta, C.astype(np.float64))
                bv = exact.codes_to_float64(bias, BF16)
                for i in range(M):
                    for j in range(N):
                        x = float(r_ex[i][j] + Fraction(float(bv[j])))
                        want = ref_act[act](x)
                        assert abs(R[i, j] - want) <= 1e-12 * max(1.0, abs(want)), (i, j, act)
                n += 1


def pin_epilogue_exact_and_sampled(o):
    """Integer inputs and bias with ReLU are exact; the sampled entry point
    agrees with the full one element by element; a NULL bias is no bias."""
    rng = _rng(23)
    M, N, K = 9, 11, 13
    A = _to_codes(rng.integers(-4, 5, (M, K)).astype(np.float64), F16)
    B = _to_codes(rng.integers(-4, 5, (K, N)).astype(np.float64), F16)
    bias = rng.integers(-20, 21, N).astype(np.float32)
    R, _ = o.gemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, F16, F32, bias, F32,
                     ACT_RELU)
    plain, _ = o.gemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, F16, F32)
    assert (R == np.maximum(plain + bias[None, :].astype(np.float64), 0.0)).all()
    R0, _ = o.gemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, F16, F32, None, F32,
                      ACT_NONE)
    assert (R0 == plain).all()
    rows = rng.integers(0, M, 40)
    cols = rng.integers(0, N, 40)
    for act in range(4):
        Rf, _ = o.gemm_ex("N", "N", M, N, K, 0.5, A, K, B, N, 0.0, None, N, F16, F32, bias, F32,
                          act)
        Rs, _ = o.gemm_sampled_ex("N", "N", M, N, K, 0.5, A, K, B, N, 0.0, None, N, F16, F32,
                                  rows, cols, bias, F32, act)
        assert (Rs == Rf[rows, cols]).all()
    try:
        o.gemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, F16, F32, bias, F32, 9)
    except ValueError:
        pass
    else:
        raise AssertionError("unknown activation accepted")


# -------------------------------------------------------------------- TF32

def _tf32_numpy(x32):
    """TF32 value of float32 inputs by a numpy bit mask (independent of C)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    special = ((u >> 23) & 0xFF) == 0xFF
    t = np.where(special, u, u & np.uint32(0xFFFFE000)).astype(np.uint32)
    return t.view(np.float32).astype(np.float64)


def pin_tf32_truncation(o):
    """FP32 used as TF32 keeps 10 mantissa bits, dropping the rest toward zero
    (CATLASS page, section 3.2): page facts and random bit patterns."""
    import struct
    bits = lambda f: struct.unpack("<I", struct.pack("<f", f))[0]
    facts = [(1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10), (1.0 + 2.0 ** -11, 1.0),
             (1.0 + 2.0 ** -10 + 2.0 ** -11, 1.0 + 2.0 ** -10), (-(1.0 + 3 * 2.0 ** -12), -1.0),
             (3.0e38, float(_tf32_numpy(np.float32([3.0e38]))[0])), (0.0, 0.0)]
    for x, want in facts:
        assert o.decode_tf32(bits(x)) == want, (x, o.decode_tf32(bits(x)), want)
    assert math.isinf(o.decode_tf32(bits(float("inf"))))
    assert math.isnan(o.decode_tf32(0x7FC00001))
    rng = _rng(31)
    u = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    mine = np.array([o.decode_tf32(int(v)) for v in u])
    lib = _tf32_numpy(x)
    same = (mine == lib) | (np.isnan(mine) & np.isnan(lib))
    assert same.all()
    fin = np.isfinite(lib) & (lib != 0)
    assert (np.abs(lib[fin]) <= np.abs(x[fin].astype(np.float64))).all()     # toward zero


def pin_gemm_tf32_bruteforce(o):
    """FP32 inputs as TF32 against exact rationals (every transpose pair), and
    integer inputs exactly."""
    rng = _rng(32)
    n = 0
    for (M, N, K) in [(3, 4, 5), (5, 2, 7), (1, 6, 3)]:
        for ta in "NT":
            for tb in "NT":
                a_rows, a_cols = (M, K) if ta == "N" else (K, M)
                b_rows, b_cols = (K, N) if tb == "N" else (N, K)
                A = rng.standard_normal((a_rows, a_cols)).astype(np.float32)
                B = rng.standard_normal((b_rows, b_cols)).astype(np.float32)
                alpha = (1.0, 0.5)[n % 2]
                R, S = o.gemm(ta, tb, M, N, K, alpha, A.view(np.uint32), a_cols,
                              B.view(np.uint32), b_cols, 0.0, None, N, F32, F32)
                opA = exact.op_matrix(_tf32_numpy(A), a_rows, a_cols, ta)
                opB = exact.op_matrix(_tf32_numpy(B), b_rows, b_cols, tb)
                r_ex, s_ex = exact.exact_gemm(opA, opB, alpha, 0.0, np.zeros((M, N)))
                for i in range(M):
                    for j in range(N):
                        assert abs(Fraction(float(R[i, j])) - r_ex[i][j]) <= \
                            Fraction(2) ** -48 * s_ex[i][j] + Fraction(1, 2 ** 1000)
                n += 1
    Ai = rng.integers(-1000, 1001, (6, 9)).astype(np.float32)
    Bi = rng.integers(-1000, 1001, (9, 7)).astype(np.float32)
    R, _ = o.gemm("N", "N", 6, 7, 9, 1.0, Ai.view(np.uint32), 9, Bi.view(np.uint32), 7, 0.0,
                  None, 7, F32, F32)
    assert (R == Ai.astype(np.float64) @ Bi.astype(np.float64)).all()   # 10-bit integers are exact


# ----------------------------------------------------------------- softmax

def _softmax_rows(o, X, dt, ldx=None, row_ids=None):
    """X: float64 values that are exact in dt -> the oracle's softmax of them."""
    rows, cols = X.shape
    ldx = ldx or max(cols, 1)
    if dt == F32:
        buf = np.full((rows, ldx), np.nan, dtype=np.float32)
        buf[:, :cols] = X.astype(np.float32)
        assert (buf[:, :cols].astype(np.float64) == X)[np.isfinite(X)].all()
    else:
        buf = np.full((rows, ldx), 0x7E00 if dt == F16 else 0x7FC0, dtype=np.uint16)
        buf[:, :cols] = _to_codes(X, dt) if X.size else buf[:, :cols]
    return o.softmax(buf, rows, cols, ldx, dt, row_ids=row_ids)


def pin_softmax_closed_forms(o):
    """Constant rows give exactly 1/n; two-point rows the logistic closed form;
    a row far above exp's range (1000, 999, 998) gives the shifted result,
    which only the maximum subtraction reaches (SGEMM page, section 2.2:
    the shift keeps exp from overflowing); a single entry gives 1."""
    for dt in (F16, BF16, F32):
        for n in (1, 2, 3, 7, 64, 1000):
            for c in (0.0, -3.0, 40.0):
                R = _softmax_rows(o, np.full((1, n), c), dt)
                assert (R == 1.0 / n).all(), (dt, n, c)
    for t in (0.5, -1.25, 3.0, 11.0, -20.0):
        R = _softmax_rows(o, np.array([[0.0, t]]), F32)
        want = [1.0 / (1.0 + math.exp(t)), 1.0 / (1.0 + math.exp(-t))]
        assert np.allclose(R[0], want, rtol=4e-16, atol=0), (t, R, want)
    R = _softmax_rows(o, np.array([[1000.0, 999.0, 998.0]]), F32)
    e = np.array([1.0, math.exp(-1.0), math.exp(-2.0)])
    assert np.allclose(R[0], e / e.sum(), rtol=4e-16, atol=0)
    R = _softmax_rows(o, np.array([[60000.0, 0.0]]), F16)
    assert R[0, 0] == 1.0 and R[0, 1] == 0.0


def pin_softmax_library_and_invariants(o):
    """Random rows of every input type against scipy.special.softmax; rows
    sum to 1; integer rows are bitwise invariant under an integer shift;
    permuting a row permutes its result; padding (NaN) is never read; the
    selected-rows entry point matches the full one."""
    from scipy.special import softmax as sp_softmax
    rng = _rng(41)
    for dt in (F16, BF16, F32):
        X = rng.standard_normal((9, 37)) * 3.0
        X = X.astype(np.float32).astype(np.float64)
        if dt != F32:
            X = exact.codes_to_float64(_to_codes_round(X, dt), dt).reshape(X.shape)
        R = _softmax_rows(o, X, dt, ldx=45)
        ref = sp_softmax(X, axis=1)
        assert np.allclose(R, ref, rtol=1e-14, atol=0), dt
        assert np.allclose(R.sum(axis=1), 1.0, rtol=0, atol=64 * 2.0 ** -52)
        perm = rng.permutation(37)
        Rp = _softmax_rows(o, X[:, perm], dt)
        assert np.allclose(Rp, R[:, perm], rtol=1e-15, atol=0)
        ids = np.array([8, 0, 3, 3])
        Rs = _softmax_rows(o, X, dt, ldx=40, row_ids=ids)
        assert (Rs == R[ids]).all()
    Xi = rng.integers(-20, 21, (5, 50)).astype(np.float64)
    R0 = _softmax_rows(o, Xi, F32)
    R1 = _softmax_rows(o, Xi + 64.0, F32)
    assert (R0 == R1).all()
    # exp(x - m) for integers is e^-k: check the values themselves
    m = Xi.max(axis=1, keepdims=True)
    e = np.exp(Xi - m)
    assert np.allclose(R0, e / e.sum(axis=1, keepdims=True), rtol=1e-15, atol=0)


def pin_softmax_special_values(o):
    """The formula's own values at the edges: NaN or +inf anywhere makes the
    row NaN; a fully masked row (all -inf) is 0/0 = NaN (SGEMM page, section
    2.5); a single -inf entry is exactly 0; empty inputs are no-ops; bad
    arguments are rejected."""
    inf, nan = math.inf, math.nan
    X = np.array([[1.0, nan, 2.0], [1.0, inf, 2.0], [-inf, -inf, -inf], [0.0, -inf, 0.0],
                  [-inf, 5.0, -inf]])
    for dt in (F16, BF16, F32):
        R = _softmax_rows(o, X, dt)
        assert np.isnan(R[0]).all() and np.isnan(R[1]).all() and np.isnan(R[2]).all(), dt
        assert (R[3] == [0.5, 0.0, 0.5]).all() and (R[4] == [0.0, 1.0, 0.0]).all(), dt
    assert o.softmax(np.zeros((0, 4), np.float32), 0, 4, 4, F32).shape == (0, 4)
    assert o.softmax(np.zeros((3, 1), np.float32), 3, 0, 1, F32).shape == (3, 0)
    for bad in [dict(ldx=3), dict(dt=7), dict(ids=[5])]:
        try:
            o.softmax(np.zeros((4, 4), np.float32), 4, 4, bad.get("ldx", 4), bad.get("dt", F32),
                      row_ids=bad.get("ids"))
        except ValueError:
            continue
        raise AssertionError(f"accepted {bad}")


# --------------------------------------------------------------- convolution

def _conv_case(rng, N, H, W, C, K, R, S, dt, integer=False):
    if integer:
        x = rng.integers(-3, 4, (N, H, W, C)).astype(np.float64)
        w = rng.integers(-3, 4, (K, R, S, C)).astype(np.float64)
        return _to_codes(x, dt), _to_codes(w, dt), x, w
    xc = _random_codes(rng, (N, H, W, C), dt)
    wc = _random_codes(rng, (K, R, S, C), dt)
    return xc, wc, exact.codes_to_float64(xc, dt).reshape(N, H, W, C), \
        exact.codes_to_float64(wc, dt).reshape(K, R, S, C)


CONV_SHAPES = [
    # N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w
    (2, 5, 6, 3, 4, 3, 3, 1, 1, 1, 1, 1, 1),
    (1, 7, 9, 2, 3, 3, 2, 0, 1, 2, 3, 2, 1),
    (3, 4, 4, 5, 2, 1, 1, 0, 0, 1, 1, 1, 1),
    (1, 8, 5, 4, 5, 5, 3, 2, 0, 1, 2, 1, 2),
    (2, 3, 3, 1, 1, 3, 3, 2, 2, 1, 1, 1, 1),
    (1, 8, 9, 2, 3, 3, 3, 1, 1, 2, 2, 1, 1),     # a stride that does not divide the span
]


def pin_conv_vs_torch(o):
    """Against torch.nn.functional.conv2d in float64 (a cross-correlation with
    zero padding, stride and dilation) on exactly decoded random inputs, both
    input types, alpha and beta."""
    import torch
    rng = _rng(51)
    for i, (N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw) in enumerate(CONV_SHAPES):
        dt = (F16, BF16)[i % 2]
        xc, wc, x, w = _conv_case(rng, N, H, W, C, K, R, S, dt)
        P, Q = o.conv2d_dims(H, W, R, S, ph, pw, sh, sw, dh, dw)
        yin = rng.standard_normal((N * P * Q, K)).astype(np.float32)
        alpha, beta = (1.0, 0.0) if i % 2 else (0.5, -2.0)
        Rr, Sr = o.conv2d(N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw, alpha, xc, wc, beta,
                          yin if beta else None, dt, F32)
        ref = torch.nn.functional.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2),
                                         torch.from_numpy(w).permute(0, 3, 1, 2),
                                         stride=(sh, sw), padding=(ph, pw), dilation=(dh, dw))
        ref = ref.permute(0, 2, 3, 1).reshape(N * P * Q, K).numpy()
        assert ref.shape == Rr.shape
        want = alpha * ref + beta * yin.astype(np.float64)
        assert np.all(np.abs(Rr - want) <= 1e-13 * (np.abs(alpha) * Sr + np.abs(beta * yin)) + 1e-300), i


def pin_conv_exact_bruteforce(o):
    """Tiny shapes against a direct evaluation of the definition in exact
    rationals (the products of 16-bit inputs are exact in binary64)."""
    rng = _rng(52)
    for i, (N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw) in enumerate(CONV_SHAPES[:4]):
        dt = (BF16, F16)[i % 2]
        xc, wc, x, w = _conv_case(rng, N, H, W, C, K, R, S, dt)
        P, Q = o.conv2d_dims(H, W, R, S, ph, pw, sh, sw, dh, dw)
        Rr, Sr = o.conv2d(N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw, 1.0, xc, wc, 0.0, None, dt, F32)
        for n in range(N):
            for p_ in range(P):
                for q in range(Q):
                    for k in range(K):
                        acc = Fraction(0)
                        for r in range(R):
                            h = p_ * sh - ph + r * dh
                            if not 0 <= h < H:
                                continue
                            for s_ in range(S):
                                ww = q * sw - pw + s_ * dw
                                if not 0 <= ww < W:
                                    continue
                                for c in range(C):
                                    acc += Fraction(float(x[n, h, ww, c])) * Fraction(float(w[k, r, s_, c]))
                        m = (n * P + p_) * Q + q
                        assert abs(Fraction(float(Rr[m, k])) - acc) <= Fraction(2) ** -50 * Fraction(float(Sr[m, k]))


def pin_conv_closed_forms(o):
    """A 1 x 1 convolution is the matrix product X (NHW x C) W^T; a delta
    filter copies the input shifted by its tap; all-ones inputs count the
    taps that fall inside the image.  Integer inputs: exact."""
    rng = _rng(53)
    # 1 x 1, stride 1, no padding: a matrix product
    xc, wc, x, w = _conv_case(rng, 2, 5, 7, 6, 4, 1, 1, BF16, integer=True)
    Rr, _ = o.conv2d(2, 5, 7, 6, 4, 1, 1, 0, 0, 1, 1, 1, 1, 1.0, xc, wc, 0.0, None, BF16, F32)
    assert (Rr == x.reshape(-1, 6) @ w.reshape(4, 6).T).all()
    # delta filter at tap (r0, s0), K = C: output = input at the tapped position
    N, H, W, C, R, S, ph, pw, sh, sw, dh, dw = 2, 6, 7, 3, 3, 3, 1, 2, 2, 1, 1, 2
    x = rng.integers(-50, 50, (N, H, W, C)).astype(np.float64)
    for r0, s0 in [(0, 0), (2, 1), (1, 2)]:
        w = np.zeros((C, R, S, C))
        for c in range(C):
            w[c, r0, s0, c] = 1.0
        P, Q = o.conv2d_dims(H, W, R, S, ph, pw, sh, sw, dh, dw)
        Rr, _ = o.conv2d(N, H, W, C, C, R, S, ph, pw, sh, sw, dh, dw, 1.0, _to_codes(x, F16),
                         _to_codes(w, F16), 0.0, None, F16, F32)
        for n in range(N):
            for p_ in range(P):
                for q in range(Q):
                    h, ww = p_ * sh - ph + r0 * dh, q * sw - pw + s0 * dw
                    want = x[n, h, ww] if (0 <= h < H and 0 <= ww < W) else np.zeros(C)
                    assert (Rr[(n * P + p_) * Q + q] == want).all()
    # all ones: C times the number of taps inside the image
    N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw = 1, 5, 4, 3, 2, 3, 3, 2, 1, 2, 1, 1, 2
    ones = _to_codes(np.ones(N * H * W * C), F16)
    wones = _to_codes(np.ones(K * R * S * C), F16)
    P, Q = o.conv2d_dims(H, W, R, S, ph, pw, sh, sw, dh, dw)
    Rr, _ = o.conv2d(N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw, 1.0, ones, wones, 0.0, None, F16, F32)
    for p_ in range(P):
        for q in range(Q):
            taps = sum(1 for r in range(R) for s_ in range(S)
                       if 0 <= p_ * sh - ph + r * dh < H and 0 <= q * sw - pw + s_ * dw < W)
            assert (Rr[p_ * Q + q] == C * taps).all()
    # the sampled entry point agrees with the full one, row by row
    N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw = CONV_SHAPES[1]
    xc, wc, _, _ = _conv_case(rng, N, H, W, C, K, R, S, F16)
    P, Q = o.conv2d_dims(H, W, R, S, ph, pw, sh, sw, dh, dw)
    yin = rng.standard_normal((N * P * Q, K)).astype(np.float32)
    Rf, Sf = o.conv2d(N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw, 0.5, xc, wc, 2.0, yin, F16, F32)
    ids = np.array([N * P * Q - 1, 0, 3, 3])
    Rs, Ss = o.conv2d_sampled(N, H, W, C, K, R, S, ph, pw, sh, sw, dh, dw, 0.5, xc, wc, 2.0, yin,
                              F16, F32, ids)
    assert (Rs == Rf[ids]).all() and (Ss == Sf[ids]).all()
    # argument checks and empty outputs
    assert o.conv2d_dims(3, 3, 5, 1, 0, 0, 1, 1, 1, 1) == (0, 3)
    for bad in [dict(C=0), dict(st=0), dict(dil=0), dict(pad=-1), dict(dt=F32)]:
        try:
            o.conv2d(1, 4, 4, bad.get("C", 2), 2, 3, 3, bad.get("pad", 1), 1, bad.get("st", 1), 1,
                     bad.get("dil", 1), 1, 1.0, np.zeros(64, np.uint16), np.zeros(64, np.uint16),
                     0.0, None, bad.get("dt", F16), F32)
        except ValueError:
            continue
        raise AssertionError(f"accepted {bad}")


# ------------------------------------------------- LayerNorm after linear

def _ln_call(o, M, N, K, A, B, C, c_dtype, beta=0.0, bias=None, bias_dtype=F32, gamma=None,
             shift=None, ln_dtype=F32, eps=1e-5, row_ids=None, dt=F16, alpha=1.0):
    return o.gemm_layernorm("N", "N", M, N, K, alpha, A, K, B, N, beta, C, N, dt, c_dtype,
                            bias, bias_dtype, gamma, shift, ln_dtype, eps, row_ids)


def pin_layernorm_closed_forms(o):
    """Rows of two values have a closed form: h = (a, b) gives
    y = +-(a - b)/2 / sqrt(((a - b)/2)^2 + eps), then gamma and shift per
    column; a constant row gives y = shift; with eps = 0 every row of y has
    mean 0 and mean square 1 (the biased variance)."""
    A = _to_codes([1.0, 2.0, -1.0], F16).reshape(3, 1)
    B = _to_codes([3.0, 1.0], F16).reshape(1, 2)
    gamma = np.array([2.0, 3.0], dtype=np.float32)
    shift = np.array([0.5, -1.0], dtype=np.float32)
    eps = 0.25
    Y, H, _ = _ln_call(o, 3, 2, 1, A, B, None, F32, gamma=gamma, shift=shift, eps=eps)
    assert (H == np.array([[3.0, 1.0], [6.0, 2.0], [-3.0, -1.0]])).all()
    for i, (a, b) in enumerate(H):
        d = (a - b) / 2.0
        u = d / np.sqrt(d * d + eps)
        want = np.array([u * 2.0 + 0.5, -u * 3.0 - 1.0])
        assert np.allclose(Y[i], want, rtol=1e-15, atol=1e-15), (i, Y[i], want)
    # constant rows: zero deviation, y = shift
    A1 = _to_codes([1.0, -2.0], F16).reshape(2, 1)
    B1 = _to_codes([1.5] * 5, F16).reshape(1, 5)
    sh = np.array([0.25, -1.0, 3.0, 0.0, 7.5], dtype=np.float32)
    Y, _, _ = _ln_call(o, 2, 5, 1, A1, B1, None, F32, gamma=np.full(5, 4.0, np.float32),
                       shift=sh, eps=1e-3)
    assert (Y == sh[None, :].astype(np.float64)).all()
    # eps = 0: standardised rows
    rng = _rng(61)
    M, N, K = 7, 33, 19
    A = _random_codes(rng, (M, K), BF16)
    B = _random_codes(rng, (K, N), BF16)
    Y, _, _ = _ln_call(o, M, N, K, A, B, None, F32, eps=0.0, dt=BF16)
    assert np.abs(Y.mean(axis=1)).max() < 1e-13
    assert np.abs((Y * Y).mean(axis=1) - 1.0).max() < 1e-13


def pin_layernorm_vs_library(o):
    """h is the fused-epilogue oracle's result rounded to C's type; y is
    torch's layer_norm (binary64) of h with gamma and shift; selected rows
    equal the full evaluation's; NULL gamma / shift are ones / zeros."""
    import torch
    rng = _rng(62)
    for (M, N, K, cdt, ldt, dt) in [(5, 40, 24, BF16, F32, BF16), (4, 17, 9, F16, BF16, F16),
                                    (3, 64, 50, F32, F16, BF16)]:
        A = _random_codes(rng, (M, K), dt)
        B = _random_codes(rng, (K, N), dt)
        if cdt == F32:
            C = rng.standard_normal((M, N)).astype(np.float32)
        else:
            C = _random_codes(rng, (M, N), cdt)
        bias = _random_codes(rng, (N,), BF16, 0.5)
        if ldt == F32:
            gamma = (1.0 + 0.1 * rng.standard_normal(N)).astype(np.float32)
            shift = (0.1 * rng.standard_normal(N)).astype(np.float32)
            g64, t64 = gamma.astype(np.float64), shift.astype(np.float64)
        else:
            gamma = _random_codes(rng, (N,), ldt, 0.5)
            shift = _random_codes(rng, (N,), ldt, 0.1)
            g64, t64 = exact.codes_to_float64(gamma, ldt), exact.codes_to_float64(shift, ldt)
        eps = 1e-5
        Y, H, S = _ln_call(o, M, N, K, A, B, C, cdt, beta=1.0, bias=bias, bias_dtype=BF16,
                           gamma=gamma, shift=shift, ln_dtype=ldt, eps=eps, dt=dt)
        R, S2 = o.gemm_ex("N", "N", M, N, K, 1.0, A, K, B, N, 1.0, C, N, dt, cdt, bias, BF16, 0)
        codes = o.round_output(R, cdt)
        Hw = (codes.view(np.float32).astype(np.float64) if cdt == F32
              else exact.codes_to_float64(codes, cdt))
        assert (H == Hw).all() and (S == S2).all()
        yt = torch.nn.functional.layer_norm(torch.from_numpy(H), (N,), torch.from_numpy(g64),
                                            torch.from_numpy(t64), eps).numpy()
        assert np.abs(Y - yt).max() <= 1e-12 * max(1.0, np.abs(yt).max())
        rows = np.array([M - 1, 0, M // 2, M - 1])
        Ys, Hs, Ss = _ln_call(o, M, N, K, A, B, C, cdt, beta=1.0, bias=bias, bias_dtype=BF16,
                              gamma=gamma, shift=shift, ln_dtype=ldt, eps=eps, row_ids=rows, dt=dt)
        assert (Ys == Y[rows]).all() and (Hs == H[rows]).all() and (Ss == S[rows]).all()
        Y1, _, _ = _ln_call(o, M, N, K, A, B, C, cdt, beta=1.0, bias=bias, bias_dtype=BF16,
                            gamma=np.ones(N, np.float32), shift=np.zeros(N, np.float32),
                            ln_dtype=F32, eps=eps, dt=dt)
        Y0, _, _ = _ln_call(o, M, N, K, A, B, C, cdt, beta=1.0, bias=bias, bias_dtype=BF16,
                            eps=eps, dt=dt)
        assert (Y1 == Y0).all()
    for bad in (dict(eps=-1.0), dict(gamma=np.ones(3, np.float32), ln_dtype=7)):
        try:
            _ln_call(o, 1, 3, 1, _to_codes([1.0], F16).reshape(1, 1),
                     _to_codes([1.0, 2.0, 3.0], F16).reshape(1, 3), None, F32, **bad)
        except ValueError:
            pass
        else:
            raise AssertionError(f"bad argument accepted: {bad}")


def _to_codes_round(values, dtype):
    """float64 values -> nearest uint16 codes by torch's conversion (test inputs)."""
    import torch
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    return torch.tensor(np.asarray(values, dtype=np.float64)).to(tdt).view(torch.int16) \
        .numpy().view(np.uint16).copy()


ALL_PINS = [
    pin_decode_exhaustive, pin_page_format_limits, pin_round_ieee_table,
    pin_round_roundtrip_exhaustive, pin_round_midpoints, pin_round_random_exact,
    pin_f32_output, pin_gemm_bruteforce, pin_gemm_integer_exact,
    pin_identity_and_permutation, pin_all_ones, pin_rank1_closed_form, pin_linearity,
    pin_quick_returns, pin_bad_arguments, pin_threads_deterministic,
    pin_activation_values, pin_epilogue_bruteforce, pin_epilogue_exact_and_sampled,
    pin_tf32_truncation, pin_gemm_tf32_bruteforce,
    pin_softmax_closed_forms, pin_softmax_library_and_invariants, pin_softmax_special_values,
    pin_conv_vs_torch, pin_conv_exact_bruteforce, pin_conv_closed_forms,
    pin_layernorm_closed_forms, pin_layernorm_vs_library,
]
