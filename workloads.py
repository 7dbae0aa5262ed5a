"""Seeded synthetic GEMM workloads shared by the tests, the smoke check and the
benchmark.

This module holds no GEMM arithmetic: it only draws random numbers and stores
them in the 16-bit (or 32-bit) formats the GEMM consumes.  Both the CUDA path
and the CPU oracle receive exactly these bit patterns.

Recipe (one generator per workload, seed 0, draws in the order A, B, C):
  * U(-1, 1)   : 2 * torch.rand - 1 in FP32,
  * N(0, 1)    : torch.randn in FP32,
  * N(0, 0.02) : 0.02 * torch.randn in FP32 (0.02 read as the standard
                 deviation, the usual weight-initialisation convention),
then converted to FP16/BF16 by torch (round to nearest even).  Matrices are
drawn in their stored shape: A is M x K for 'N' and K x M for 'T'; B is K x N
for 'N' and N x K for 'T' ("weights stored N x K, K-contiguous"); C is M x N.
When a leading dimension exceeds the logical row length, the padding columns
are filled with NaN so that any read outside the logical matrix shows up in the
result.

The named workloads are the five shapes of the mixed-precision GEMM study: a
256^3 FP16 GEMM with FP32 output; a 1024^3 FP16 GEMM with B stored column-major
and FP16 output; a ragged 1000 x 1023 x 777 BF16 GEMM with C = A*B + C in FP32;
three transformer linear layers (8192 tokens, 4096 -> 4096, 4096 -> 14336,
14336 -> 4096, BF16); and a skinny decode GEMM (64 tokens, 8192 -> 16384, FP16).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

DT_F16, DT_BF16, DT_F32 = 0, 1, 2
TORCH_DTYPE = {DT_F16: torch.float16, DT_BF16: torch.bfloat16, DT_F32: torch.float32}
DT_NAME = {DT_F16: "f16", DT_BF16: "bf16", DT_F32: "f32"}
DT_OF = {v: k for k, v in TORCH_DTYPE.items()}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    transA: str
    transB: str
    ab_dtype: int
    c_dtype: int
    alpha: float
    beta: float
    a_dist: str          # "U", "N1" or "N002"
    b_dist: str
    c_dist: Optional[str] = None   # None: C is not an input (beta == 0)
    lda: Optional[int] = None      # None: tight (the stored row length)
    ldb: Optional[int] = None
    ldc: Optional[int] = None
    seed: int = 0

    def a_shape(self):
        return (self.M, self.K) if self.transA in "Nn" else (self.K, self.M)

    def b_shape(self):
        return (self.K, self.N) if self.transB in "Nn" else (self.N, self.K)

    def lds(self):
        return (self.lda or max(1, self.a_shape()[1]), self.ldb or max(1, self.b_shape()[1]),
                self.ldc or max(1, self.N))

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once, C also read when beta != 0."""
        e_ab = 4 if self.ab_dtype == DT_F32 else 2
        e_c = 4 if self.c_dtype == DT_F32 else 2
        b = (self.M * self.K + self.K * self.N) * e_ab + self.M * self.N * e_c
        if self.beta != 0:
            b += self.M * self.N * e_c
        return b


WORKLOADS = {
    w.name: w for w in [
        Workload("square256_f16_f32out", 256, 256, 256, "N", "N", DT_F16, DT_F32,
                 1.0, 0.0, "U", "U"),
        Workload("square1024_f16_nt_f16out", 1024, 1024, 1024, "N", "T", DT_F16, DT_F16,
                 1.0, 0.0, "U", "U"),
        Workload("ragged1000x1023x777_bf16_beta1", 1000, 1023, 777, "N", "N", DT_BF16,
                 DT_F32, 1.0, 1.0, "N1", "N1", "N1"),
        Workload("linear_8192x4096x4096_bf16", 8192, 4096, 4096, "N", "T", DT_BF16,
                 DT_BF16, 1.0, 0.0, "N1", "N002"),
        Workload("linear_8192x14336x4096_bf16", 8192, 14336, 4096, "N", "T", DT_BF16,
                 DT_BF16, 1.0, 0.0, "N1", "N002"),
        Workload("linear_8192x4096x14336_bf16", 8192, 4096, 14336, "N", "T", DT_BF16,
                 DT_BF16, 1.0, 0.0, "N1", "N002"),
        Workload("tf32_linear_8192x4096x4096_f32out", 8192, 4096, 4096, "N", "T", DT_F32,
                 DT_F32, 1.0, 0.0, "N1", "N002"),
        Workload("skinny_64x16384x8192_f16", 64, 16384, 8192, "N", "T", DT_F16, DT_F16,
                 1.0, 0.0, "N1", "N002"),
    ]
}


def _draw(gen: torch.Generator, dist: str, shape) -> torch.Tensor:
    if dist == "U":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "N1":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "N002":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * 0.02
    raise ValueError(f"unknown distribution {dist!r}")


def _stored(values: torch.Tensor, ld: int, dtype: torch.dtype) -> torch.Tensor:
    rows, cols = values.shape
    if ld == cols:
        return values.to(dtype).contiguous()
    buf = torch.full((rows, ld), float("nan"), dtype=dtype)
    buf[:, :cols] = values.to(dtype)
    return buf


@dataclasses.dataclass
class Inputs:
    A: torch.Tensor   # stored (rows x lda), CPU, FP16/BF16 (or FP32 used as TF32)
    B: torch.Tensor   # stored (rows x ldb)
    C: Optional[torch.Tensor]   # stored (M x ldc) in the output dtype, or None
    lda: int
    ldb: int
    ldc: int


def make_inputs(w: Workload) -> Inputs:
    """Draw A, then B, then C (if beta != 0) from one seeded CPU generator."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    lda, ldb, ldc = w.lds()
    ab_t = TORCH_DTYPE[w.ab_dtype]
    A = _stored(_draw(gen, w.a_dist, w.a_shape()), lda, ab_t)
    B = _stored(_draw(gen, w.b_dist, w.b_shape()), ldb, ab_t)
    C = None
    if w.c_dist is not None:
        C = _stored(_draw(gen, w.c_dist, (w.M, w.N)), ldc, TORCH_DTYPE[w.c_dtype])
    return Inputs(A, B, C, lda, ldb, ldc)


def as_codes(t: torch.Tensor):
    """Raw bit patterns of a CPU tensor as a numpy array (uint16 or uint32)."""
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.contiguous().view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.contiguous().numpy().view("uint32")
    raise TypeError(t.dtype)


# ------------------------------------------------------------------ softmax

@dataclasses.dataclass(frozen=True)
class SoftmaxWorkload:
    """Row softmax of a rows x cols matrix of logits (SGEMM tutorial page,
    section 2).  dist: "N1" = N(0, 1) logits, "N4" = 4 N(0, 1) (peakier rows).
    mask: None, or "causal" -- row r keeps columns j <= r mod cols and sets
    the rest to -inf (the masked-attention pattern; row 0 of every block of
    cols rows keeps one entry)."""
    name: str
    rows: int
    cols: int
    x_dtype: int
    y_dtype: int
    dist: str = "N1"
    mask: Optional[str] = None
    ldx: Optional[int] = None
    ldy: Optional[int] = None
    seed: int = 0

    def lds(self):
        return (self.ldx or max(1, self.cols), self.ldy or max(1, self.cols))

    def algorithmic_bytes(self) -> int:
        """X read once, Y written once."""
        ex = 4 if self.x_dtype == DT_F32 else 2
        ey = 4 if self.y_dtype == DT_F32 else 2
        return self.rows * self.cols * (ex + ey)


SOFTMAX_WORKLOADS = {w.name: w for w in [
    SoftmaxWorkload("softmax_16384x4096_f32", 16384, 4096, DT_F32, DT_F32),
    SoftmaxWorkload("softmax_65536x1024_bf16", 65536, 1024, DT_BF16, DT_BF16),
    SoftmaxWorkload("softmax_8192x8192_bf16_causal", 8192, 8192, DT_BF16, DT_BF16, "N4", "causal"),
    SoftmaxWorkload("softmax_2048x65536_f32", 2048, 65536, DT_F32, DT_F32),
    SoftmaxWorkload("softmax_128x1048576_f32", 128, 1048576, DT_F32, DT_F32),
]}


def make_softmax_input(w: SoftmaxWorkload) -> torch.Tensor:
    """The stored rows x ldx CPU tensor of w.x_dtype (padding NaN), drawn in
    FP32 from one seeded generator, then masked, then cast (RNE)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    ldx, _ = w.lds()
    scale = {"N1": 1.0, "N4": 4.0}[w.dist]
    x = torch.randn((w.rows, w.cols), generator=gen, dtype=torch.float32) * scale
    if w.mask == "causal" and w.cols > 0:
        keep = torch.arange(w.cols).view(1, -1) <= (torch.arange(w.rows) % w.cols).view(-1, 1)
        x = torch.where(keep, x, torch.full_like(x, float("-inf")))
    elif w.mask is not None:
        raise ValueError(f"unknown mask {w.mask!r}")
    return _stored(x, ldx, TORCH_DTYPE[w.x_dtype])


# -------------------------------------------------------------- convolution

@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    """Forward 2-D convolution (CATLASS page, section 5.1), NHWC input,
    KRSC filter, NPQK output; activations N(0, 1), weights N(0, 0.02)."""
    name: str
    N: int
    H: int
    W: int
    C: int
    K: int
    R: int
    S: int
    pad: tuple
    stride: tuple
    dil: tuple
    x_dtype: int
    y_dtype: int
    seed: int = 0

    def out_hw(self):
        P = (self.H + 2 * self.pad[0] - self.dil[0] * (self.R - 1) - 1) // self.stride[0] + 1
        Q = (self.W + 2 * self.pad[1] - self.dil[1] * (self.S - 1) - 1) // self.stride[1] + 1
        return P, Q

    def gemm_mnk(self):
        P, Q = self.out_hw()
        return self.N * P * Q, self.K, self.R * self.S * self.C

    def flops(self) -> float:
        M, N, K = self.gemm_mnk()
        return 2.0 * M * N * K


CONV_WORKLOADS = {w.name: w for w in [
    ConvWorkload("conv3x3_n32_56x56_c64_k64_bf16", 32, 56, 56, 64, 64, 3, 3, (1, 1), (1, 1),
                 (1, 1), DT_BF16, DT_BF16),
    ConvWorkload("conv3x3_n32_28x28_c128_k128_bf16", 32, 28, 28, 128, 128, 3, 3, (1, 1), (1, 1),
                 (1, 1), DT_BF16, DT_BF16),
    ConvWorkload("conv3x3_n16_64x64_c256_k256_bf16", 16, 64, 64, 256, 256, 3, 3, (1, 1), (1, 1),
                 (1, 1), DT_BF16, DT_BF16),
    ConvWorkload("conv3x3_n32_14x14_c512_k512_bf16", 32, 14, 14, 512, 512, 3, 3, (1, 1), (1, 1),
                 (1, 1), DT_BF16, DT_BF16),
]}


def make_conv_inputs(w: ConvWorkload):
    """(X NHWC, Wt KRSC) CPU tensors of w.x_dtype, drawn X then Wt in FP32 from
    one seeded generator, then rounded."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    x = torch.randn((w.N, w.H, w.W, w.C), generator=gen, dtype=torch.float32)
    wt = torch.randn((w.K, w.R, w.S, w.C), generator=gen, dtype=torch.float32) * 0.02
    t = TORCH_DTYPE[w.x_dtype]
    return x.to(t), wt.to(t)
