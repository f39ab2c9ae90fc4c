"""Shared helpers for the GPU parity tests: device operands from the seeded
bit patterns, poisoned output buffers with trailing guards, and the scaled
comparison against the oracle.

Poison 7.0 and 64 trailing guards of 11.0 follow the page "Wider
consecutive-weight NAX GEMM", section "Launch contract and correctness";
tolerances (partials 1e-4; outputs F32 1e-4, F16 2e-3, BF16 2e-2, each times
sum_k |a*b|) follow "Aligned shared rows for pipelined NAX on CUDA", section
"Contract and correctness".
"""
from __future__ import annotations

import json
import os
from functools import lru_cache

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
with open(os.path.join(GOLDEN, "pages_contract.json")) as _f:
    PAGES = json.load(_f)

TOL_PARTIAL = PAGES["tolerance_partials"]["value"]
TOL_FINAL = {k: PAGES["tolerance_final"][k] for k in ("f32", "f16", "bf16")}
POISON = PAGES["poison_value"]["value"]
GUARD_VALUE = PAGES["guard"]["value"]
GUARDS = PAGES["guard"]["count"]


def device_operand(bits: np.ndarray, dtype: str):
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(bits, np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


class Guarded:
    """A flat F32 device buffer: n elements of poison, then GUARDS guard values."""

    def __init__(self, n: int, poison: float = POISON):
        import torch

        self.n = n
        self.buf = torch.full((n + GUARDS,), poison, dtype=torch.float32, device="cuda")
        self.buf[n:] = GUARD_VALUE

    @property
    def data(self):
        return self.buf[: self.n]

    def guards_intact(self) -> bool:
        import torch

        g = self.buf[self.n:]
        want = torch.full_like(g, GUARD_VALUE)
        return bool(torch.equal(g.view(torch.int32), want.view(torch.int32)))

    def numpy(self) -> np.ndarray:
        return self.data.cpu().numpy()


def max_scaled_error(got: np.ndarray, ref: np.ndarray, bound: np.ndarray) -> float:
    """max |got-ref| / bound; elements with bound 0 must be exactly 0 (else inf).
    NaN anywhere gives inf."""
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    if not np.all(np.isfinite(err)):
        return float("inf")
    zero = bound == 0
    if np.any(err[zero] != 0):
        return float("inf")
    if np.all(zero):
        return 0.0
    return float(np.max(err[~zero] / bound[~zero]))


def workspace(M, N, K, S, kps, poison: float = POISON):
    """A gemm_bt workspace (the partials), poisoned, guards behind."""
    import split_bf16_gemm_gb300 as sk

    nbytes = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
    return Guarded(nbytes // 4, poison), nbytes


@lru_cache(maxsize=64)
def oracle_case(M, N, K, S, kps, dtype, recipe="uniform", seed=0):
    """(operands, P*, SP, O*, SO) for a seeded case; cached per process."""
    import oracle
    import splitk_inputs as gen

    if recipe == "uniform":
        ops = gen.uniform(M, N, K, dtype, seed)
    elif recipe == "integers":
        ops = gen.integers(M, N, K, dtype, seed)
    elif recipe == "ones":
        ops = gen.ones(M, N, K, dtype)
    elif recipe == "identity_b":
        ops = gen.identity_b(M, N, K, dtype, seed)
    else:
        raise ValueError(recipe)
    P, SP = oracle.partials(ops.A, ops.B, dtype, K, S, kps)
    O, SO = oracle.output(ops.A, ops.B, dtype)
    return ops, P, SP, O, SO
