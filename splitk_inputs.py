"""Seeded synthetic operands for split-K GEMM with prepared, transposed weights.

This module only draws and rounds inputs; it holds none of the GEMM's
arithmetic.  Both the oracle-side tests and the GPU-side tests and benchmark
take their operands from here, so the two sides see the same bit patterns.

Recipe (the pages' test inputs, "Wider consecutive-weight NAX GEMM", section
"Launch contract and correctness": a zero first A row and a last row at four
times the ordinary scale; uniform values in [-1, 1]):

* ``numpy.random.Generator(PCG64(seed))``; A[M,K] is drawn first, then B[N,K],
  each as float64 ``uniform(-1, 1)``;
* cast to float32, then rounded to the element format with round-to-nearest-
  even (numpy for binary16, torch for bfloat16, nothing for binary32);
* A[0,:] = 0, then A[M-1,:] *= 4 on the rounded values (exact in every format).

Operands are returned as arrays of bit patterns: ``uint16`` for f16/bf16 and
``float32`` for f32, row-major, with B already in the prepared [N,K] layout.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

DTYPES = ("f32", "f16", "bf16")


@dataclass
class Operands:
    A: np.ndarray          # [M, K] bit patterns (uint16) or float32
    B: np.ndarray          # [N, K] bit patterns (uint16) or float32
    dtype: str
    seed: int
    recipe: str

    @property
    def M(self) -> int:
        return self.A.shape[0]

    @property
    def N(self) -> int:
        return self.B.shape[0]

    @property
    def K(self) -> int:
        return self.A.shape[1]


def _round(x32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> bit patterns of ``dtype``, round-to-nearest-even."""
    x32 = np.ascontiguousarray(x32, np.float32)
    if dtype == "f32":
        return x32.copy()
    if dtype == "f16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch

        t = torch.from_numpy(x32).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unknown dtype {dtype!r}")


def _to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns -> float32 values (exact: every format widens exactly)."""
    if dtype == "f32":
        return bits.astype(np.float32)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32)


def _scale_row(bits: np.ndarray, row: int, factor: float, dtype: str) -> None:
    vals = _to_f32(bits[row], dtype) * np.float32(factor)
    bits[row] = _round(vals, dtype)


def uniform(M: int, N: int, K: int, dtype: str, seed: int = 0,
            zero_first_row: bool = True, scale_last_row: bool = True) -> Operands:
    """The pages' operands: uniform[-1,1], zero first A row, x4 last A row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.uniform(-1.0, 1.0, size=(M, K)).astype(np.float32)
    b = rng.uniform(-1.0, 1.0, size=(N, K)).astype(np.float32)
    A, B = _round(a, dtype), _round(b, dtype)
    if zero_first_row:
        A[0] = _round(np.zeros(K, np.float32), dtype)
    if scale_last_row and M > 1:
        _scale_row(A, M - 1, 4.0, dtype)
    return Operands(A, B, dtype, seed, "uniform[-1,1], A[0]=0, A[M-1]*=4")


def integers(M: int, N: int, K: int, dtype: str, seed: int = 0, lo: int = -8,
             hi: int = 8) -> Operands:
    """Integers in [lo, hi]; exact in every format, so every product and every
    partial sum below 2^24 is exact in F32 too."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.integers(lo, hi, size=(M, K), endpoint=True).astype(np.float32)
    b = rng.integers(lo, hi, size=(N, K), endpoint=True).astype(np.float32)
    return Operands(_round(a, dtype), _round(b, dtype), dtype, seed,
                    f"integers in [{lo},{hi}]")


def ones(M: int, N: int, K: int, dtype: str) -> Operands:
    """All-ones A and B."""
    o = np.ones((M, K), np.float32)
    return Operands(_round(o, dtype), _round(np.ones((N, K), np.float32), dtype),
                    dtype, 0, "all ones")


def identity_b(M: int, N: int, K: int, dtype: str, seed: int = 0) -> Operands:
    """Uniform A, and B[n,k] = 1 if k == n else 0 (requires N <= K)."""
    assert N <= K
    u = uniform(M, N, K, dtype, seed)
    b = np.zeros((N, K), np.float32)
    b[np.arange(N), np.arange(N)] = 1.0
    return Operands(u.A, _round(b, dtype), dtype, seed, "uniform A, B = [I | 0]")


def unit_rows_a(M: int, N: int, K: int, dtype: str, seed: int = 0) -> Operands:
    """A[m,k] = 1 if k == m % K else 0; uniform B."""
    u = uniform(M, N, K, dtype, seed)
    a = np.zeros((M, K), np.float32)
    a[np.arange(M), np.arange(M) % K] = 1.0
    return Operands(_round(a, dtype), u.B, dtype, seed, "A rows = e_(m mod K), uniform B")


def weight_kn(K: int, N: int, dtype: str, seed: int = 0) -> np.ndarray:
    """An unprepared weight W[K,N] (row-major), uniform[-1,1], rounded like
    the operands: the input of the weight preparation B[n,k] = W[k,n]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _round(rng.uniform(-1.0, 1.0, size=(K, N)).astype(np.float32), dtype)


def to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen bit patterns to float32 values (for building torch tensors)."""
    return _to_f32(np.asarray(bits), dtype)
