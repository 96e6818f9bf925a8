"""Seeded synthetic inputs and the named workloads of the batched product.

This module holds no arithmetic of the product itself: it only draws random
numbers, rounds them to the 16-bit input formats and lays them out with the
strides a workload names.  Both the GPU tests and the fp64 oracle take their
inputs from here, so a parity test compares the two on identical bytes.

Generator: numpy's PCG64 bit generator seeded per operand
(seed = 1000*workload + operand index, A=1, B=2, C_in=3), uniform values via
``Generator.random`` mapped to [-1, 1) and normal values via
``Generator.standard_normal``, both drawn in float32 and rounded to bf16 or
fp16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

SEED_A, SEED_B, SEED_C, SEED_V = 1, 2, 3, 4


def draw(n: int, seed: int, dist: str) -> np.ndarray:
    """n float32 samples from ``dist`` ("uniform" on [-1,1) or "normal")."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dist == "uniform":
        x = rng.random(n, dtype=np.float32)
        x *= 2.0
        x -= 1.0
        return x
    if dist == "normal":
        return rng.standard_normal(n, dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def round16(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to bf16/fp16 (RNE); return the raw uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "f16":
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(f"unknown 16-bit type {dtype!r}")


def bits16(n: int, seed: int, dist: str, dtype: str) -> np.ndarray:
    """n seeded values rounded to a 16-bit format, as uint16 bits."""
    return round16(draw(n, seed, dist), dtype)


def as_torch16(bits: np.ndarray, dtype: str) -> torch.Tensor:
    """View uint16 bits as a torch bf16/fp16 CPU tensor (no copy)."""
    t = torch.from_numpy(np.ascontiguousarray(bits)).view(torch.int16)
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def small_ints16(n: int, seed: int, lo: int, hi: int, dtype: str) -> np.ndarray:
    """n seeded integers in [lo, hi] stored exactly in a 16-bit format."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.integers(lo, hi + 1, size=n).astype(np.float32)
    return round16(x, dtype)


@dataclasses.dataclass(frozen=True)
class Problem:
    """One batched product C[b] = alpha*op(A[b])*op(B[b]) + beta*C[b].

    Storage is row-major with element strides: A[b] is M x K (transA=0) or
    K x M (transA=1); B[b] is K x N (transB=0) or N x K (transB=1); C[b] is
    M x N.  A stride of 0 between batch items broadcasts A or B."""
    batch: int
    M: int
    N: int
    K: int
    transA: bool = False
    transB: bool = False
    type_ab: str = "bf16"
    type_c: str = "f32"
    alpha: float = 1.0
    beta: float = 0.0
    lda: int | None = None
    ldb: int | None = None
    ldc: int | None = None
    sA: int | None = None
    sB: int | None = None
    sC: int | None = None
    dist_ab: str = "uniform"
    dist_c: str = "uniform"
    seed: int = 0
    name: str = ""

    # shapes of the stored matrices
    @property
    def a_rows(self):
        return self.K if self.transA else self.M

    @property
    def a_cols(self):
        return self.M if self.transA else self.K

    @property
    def b_rows(self):
        return self.N if self.transB else self.K

    @property
    def b_cols(self):
        return self.K if self.transB else self.N

    def strides(self):
        lda = self.lda if self.lda is not None else self.a_cols
        ldb = self.ldb if self.ldb is not None else self.b_cols
        ldc = self.ldc if self.ldc is not None else self.N
        sA = self.sA if self.sA is not None else self.a_rows * lda
        sB = self.sB if self.sB is not None else self.b_rows * ldb
        sC = self.sC if self.sC is not None else self.M * ldc
        return dict(lda=lda, ldb=ldb, ldc=ldc, sA=sA, sB=sB, sC=sC)

    def storage_elems(self):
        """Elements each buffer must hold, from the strides and shapes."""
        s = self.strides()

        def need(batch, stride, rows, ld, cols):
            if batch == 0 or rows == 0 or cols == 0:
                return 0
            return (batch - 1) * stride + (rows - 1) * ld + cols

        return (need(self.batch, s["sA"], self.a_rows, s["lda"], self.a_cols),
                need(self.batch, s["sB"], self.b_rows, s["ldb"], self.b_cols),
                need(self.batch, s["sC"], self.M, s["ldc"], self.N))

    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once, C read once more if beta != 0."""
        e = 2
        ec = 4 if self.type_c == "f32" else 2
        a = (1 if self.sA == 0 else self.batch) * self.M * self.K * e
        b = (1 if self.sB == 0 else self.batch) * self.K * self.N * e
        c = self.batch * self.M * self.N * ec
        return a + b + c * (2 if self.beta != 0.0 else 1)

    def oracle_kwargs(self):
        s = self.strides()
        return dict(batch=self.batch, M=self.M, N=self.N, K=self.K, transA=self.transA,
                    transB=self.transB, type_ab=self.type_ab, type_c=self.type_c,
                    alpha=self.alpha, beta=self.beta, **s)


@dataclasses.dataclass
class Inputs:
    """Host copies of one problem's inputs: uint16 bits for A and B, and
    C_in as float32 values or bf16 bits (None when beta == 0)."""
    A: np.ndarray
    B: np.ndarray
    C_in: np.ndarray | None


def make_inputs(p: Problem, *, c_fill: str = "random") -> Inputs:
    """Seeded inputs for ``p``.  Padding elements between rows (ld larger
    than the row) are drawn too; they never enter the product."""
    na, nb, nc = p.storage_elems()
    base = 1000 * p.seed
    A = bits16(na, base + SEED_A, p.dist_ab, p.type_ab)
    B = bits16(nb, base + SEED_B, p.dist_ab, p.type_ab)
    C_in = None
    if p.beta != 0.0:
        x = draw(nc, base + SEED_C, p.dist_c)
        C_in = x if p.type_c == "f32" else round16(x, "bf16")
    return Inputs(A, B, C_in)


# ---------------------------------------------------------------- workloads
#
# The five workloads the product is specified and measured on.  Seeds are
# 1000*index + operand.

SMALL = Problem(batch=2, M=64, N=64, K=64, type_ab="bf16", type_c="f32",
                dist_ab="uniform", seed=1, name="bmm_b2_64x64x64_bf16_f32")

GEMM_4096 = Problem(batch=1, M=4096, N=4096, K=4096, transB=True, type_ab="bf16",
                    type_c="bf16", dist_ab="normal", seed=2, name="gemm_4096x4096x4096_tn_bf16")

RAGGED = Problem(batch=16, M=1000, N=999, K=1000, transA=True, type_ab="f16",
                 type_c="f32", alpha=0.5, beta=1.0, dist_ab="uniform", dist_c="uniform",
                 seed=3, name="ragged_b16_1000x999x1000_ta_f16_f32")

ATTN_SCALE = 1.0 / math.sqrt(128.0)
ATTN_QK = Problem(batch=128, M=2048, N=2048, K=128, transB=True, type_ab="bf16",
                  type_c="f32", alpha=float(np.float32(ATTN_SCALE)), dist_ab="normal",
                  seed=4, name="attn_qk_b128_2048x2048x128_bf16_f32")
ATTN_PV = Problem(batch=128, M=2048, N=128, K=2048, type_ab="bf16", type_c="bf16",
                  dist_ab="normal", seed=4, name="attn_pv_b128_2048x128x2048_bf16")

SKINNY = Problem(batch=1024, M=16, N=256, K=4096, type_ab="bf16", type_c="bf16",
                 dist_ab="uniform", seed=5, name="skinny_b1024_16x256x4096_bf16")

WORKLOADS = {p.name: p for p in (SMALL, GEMM_4096, RAGGED, ATTN_QK, ATTN_PV, SKINNY)}

# A square-GEMM neighbour whose tile count is no multiple of the 76 CTA pairs
# (16 x 18 = 288 tiles of 256 x 256: 3.79 rounds), measured beside the
# headline to show how the persistent schedule handles a leftover round.
UNEVEN_GEMM = Problem(batch=1, M=4000, N=4500, K=4096, transB=True, type_ab="bf16", type_c="bf16",
                      dist_ab="normal", seed=6, name="gemm_4000x4500x4096_tn_bf16")


def attention_qkv(batch=128, L=2048, D=128, Lk=None, seed=None):
    """Q [batch, L, D] and K, V [batch, Lk, D] bit arrays (bf16 normal; Lk = L
    unless given) for the attention pair and its fused form."""
    base = 1000 * (ATTN_QK.seed if seed is None else seed)
    Lk = L if Lk is None else Lk
    Q = bits16(batch * L * D, base + SEED_A, "normal", "bf16").reshape(batch, L, D)
    Kt = bits16(batch * Lk * D, base + SEED_B, "normal", "bf16").reshape(batch, Lk, D)
    V = bits16(batch * Lk * D, base + SEED_V, "normal", "bf16").reshape(batch, Lk, D)
    return Q, Kt, V
