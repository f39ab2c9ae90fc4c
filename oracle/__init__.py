"""F64 CPU oracle for split-K GEMM with prepared, transposed weights.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  The product library
(``split_bf16_gemm_gb300``) never imports it, and the two share no code: this
package wraps ``splitk_oracle.c`` (plain C, built with gcc), which decodes the
input bit patterns itself and sums every dot product in F64, k ascending.

What it computes is the contract of the pages "Aligned shared rows for pipelined
NAX on CUDA" (section "Contract and correctness") and "Wider consecutive-weight
NAX GEMM" (section "Launch contract and correctness"):

* ``partials``: P[s,m,n] = sum over split s of A[m,k]*B[n,k], with the error
  scale SP = the same sum of |A[m,k]*B[n,k]|;
* ``output``: the unsplit O[m,n] = sum over all k, with its scale SO;
* ``points``: selected elements of either, for matrices too big to do whole;
* ``contract``: 0 for a legal geometry, 1 when the shape rule fails (M, K, kps
  positive multiples of 32, N of 64), 2 when the split rule fails (each split
  starts below K, together they cover K);
* ``decode``: the element formats' field definitions;
* ``transpose``: the weight preparation B[n,k] = W[k,n] ("Wider consecutive-
  weight NAX GEMM", section "Performance method": the transposed layout is
  prepared once, outside timing).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, library cross-checks and invariants); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "splitk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# Element formats, in the numbering the oracle's C entry points take.
F32, F16, BF16 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (portable flags: same results on x86 and Arm)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_decode.argtypes = [i32, vp, i64, vp]
            lib.oracle_contract.argtypes = [i64, i64, i64, i64, i64]
            lib.oracle_split_range.argtypes = [i64, i64, i64, vp, vp]
            lib.oracle_transpose.argtypes = [i32, vp, i64, i64, vp]
            lib.oracle_transpose.restype = i32
            lib.oracle_partials.argtypes = [i32, vp, vp, i64, i64, i64, i64, i64, vp, vp, i32]
            lib.oracle_output.argtypes = [i32, vp, vp, i64, i64, i64, vp, vp, i32]
            lib.oracle_points.argtypes = [i32, vp, vp, i64, i64, i64, i64, i64, i64,
                                          vp, vp, vp, vp, vp]
            for f in (lib.oracle_decode, lib.oracle_contract, lib.oracle_partials,
                      lib.oracle_output, lib.oracle_points):
                f.restype = i32
            lib.oracle_split_range.restype = None
            _lib = lib
    return _lib


def _threads(threads):
    if threads is None:
        return max(1, len(os.sched_getaffinity(0)))
    return int(threads)


def _bits(x: np.ndarray, code: int) -> np.ndarray:
    want = np.uint32 if code == F32 else np.uint16
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32 and code == F32:
        x = x.view(np.uint32)
    if x.dtype.itemsize != np.dtype(want).itemsize:
        raise TypeError(f"operand has {x.dtype}, expected {np.dtype(want).itemsize}-byte patterns")
    return x.view(want)


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode an array of element bit patterns of ``dtype`` into float64."""
    code = DTYPE_CODES[dtype]
    b = _bits(bits, code)
    out = np.empty(b.shape, np.float64)
    rc = _load().oracle_decode(code, _ptr(b), b.size, _ptr(out))
    if rc:
        raise ValueError(f"oracle_decode failed ({rc})")
    return out


def transpose(W: np.ndarray) -> np.ndarray:
    """Row-major W[K,N] (2- or 4-byte elements) -> row-major B[N,K], bits copied."""
    w = np.ascontiguousarray(W)
    rows, cols = w.shape
    out = np.empty((cols, rows), w.dtype)
    rc = _load().oracle_transpose(w.dtype.itemsize, _ptr(w), rows, cols, _ptr(out))
    if rc:
        raise ValueError(f"oracle_transpose failed ({rc})")
    return out


def contract(M: int, N: int, K: int, splits: int, kps: int) -> int:
    """0 for a legal geometry, 1 when the shape rule fails, 2 when the split rule fails."""
    return int(_load().oracle_contract(M, N, K, splits, kps))


def split_range(K: int, kps: int, s: int) -> tuple[int, int]:
    """Half-open k range of split s: [s*kps, min((s+1)*kps, K))."""
    k0, k1 = ctypes.c_int64(), ctypes.c_int64()
    _load().oracle_split_range(K, kps, s, ctypes.byref(k0), ctypes.byref(k1))
    return k0.value, k1.value


def partials(A, B, dtype: str, K: int, splits: int, kps: int, threads=None):
    """(P, SP), both float64 [splits, M, N], from bit-pattern operands A[M,K], B[N,K]."""
    code = DTYPE_CODES[dtype]
    a, b = _bits(A, code), _bits(B, code)
    M, N = a.shape[0], b.shape[0]
    assert a.shape == (M, K) and b.shape == (N, K)
    P = np.empty((splits, M, N), np.float64)
    SP = np.empty_like(P)
    rc = _load().oracle_partials(code, _ptr(a), _ptr(b), M, N, K, splits, kps,
                                 _ptr(P), _ptr(SP), _threads(threads))
    if rc:
        raise ValueError(f"oracle_partials: geometry rejected or failed ({rc})")
    return P, SP


def output(A, B, dtype: str, threads=None):
    """(O, SO), both float64 [M, N]: the unsplit product and its error scale."""
    code = DTYPE_CODES[dtype]
    a, b = _bits(A, code), _bits(B, code)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape == (N, K)
    O = np.empty((M, N), np.float64)
    SO = np.empty_like(O)
    rc = _load().oracle_output(code, _ptr(a), _ptr(b), M, N, K, _ptr(O), _ptr(SO),
                               _threads(threads))
    if rc:
        raise ValueError(f"oracle_output failed ({rc})")
    return O, SO


def points(A, B, dtype: str, kps: int, splits: int, s_idx, m_idx, n_idx):
    """(val, bound) at selected points; s < 0 selects the unsplit output O[m,n]."""
    code = DTYPE_CODES[dtype]
    a, b = _bits(A, code), _bits(B, code)
    M, K = a.shape
    N = b.shape[0]
    s = np.ascontiguousarray(s_idx, np.int64)
    m = np.ascontiguousarray(m_idx, np.int64)
    n = np.ascontiguousarray(n_idx, np.int64)
    assert s.shape == m.shape == n.shape
    val = np.empty(s.shape, np.float64)
    bound = np.empty(s.shape, np.float64)
    rc = _load().oracle_points(code, _ptr(a), _ptr(b), M, N, K, kps, splits, s.size,
                               _ptr(s), _ptr(m), _ptr(n), _ptr(val), _ptr(bound))
    if rc:
        raise ValueError(f"oracle_points failed ({rc})")
    return val, bound
