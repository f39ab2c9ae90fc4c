"""Host-side tests of libsplitk (no GPU): the library loads, exports every
function include/splitk.h declares, and its validation agrees with the oracle's
statement of the pages' contract.  Every call here fails validation before any
CUDA call, so nothing touches a device (fake pointers are never dereferenced).
"""
import ctypes
import json
import os
import re

import pytest

import split_bf16_gemm_gb300 as sk
from split_bf16_gemm_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splitk.h")


@pytest.fixture(scope="module")
def L():
    sk.build()
    return sk.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(bd.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_library_symbols_are_c_abi(L):
    # nm -D lists the dynamic symbols; C linkage means unmangled names
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", sk.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


def test_geometry_matches_oracle_contract(L, orc):
    """libsplitk's contract decision == the oracle's, bit for bit, over a grid."""
    code = {0: 0, 1: bd.ERR_SHAPE, 2: bd.ERR_SPLIT}
    for M in (-32, 0, 16, 32, 48, 96, 128, 256):
        for N in (0, 32, 64, 96, 128, 512):
            for K in (0, 32, 64, 96, 160, 2048):
                for kps in (0, 16, 32, 64, 96, 512, 4096):
                    for S in (0, 1, 2, 3, 4, 5, 16, 64):
                        want = code[orc.contract(M, N, K, S, kps)]
                        assert sk.splitk_check_geometry(M, N, K, S, kps) == want, (M, N, K, S, kps)


def test_geometry_pages_cases(L):
    with open(os.path.join(ROOT, "tests", "golden", "pages_contract.json")) as f:
        cases = json.load(f)["contract_cases"]["cases"]
    code = {0: 0, 1: bd.ERR_SHAPE, 2: bd.ERR_SPLIT}
    for M, N, K, S, kps, expect in cases:
        assert sk.splitk_check_geometry(M, N, K, S, kps) == code[expect]


def test_implementation_limits(L):
    big = (1 << 22) + 32
    assert sk.splitk_check_geometry(big, 64, 64, 1, 64) == bd.ERR_SHAPE
    assert sk.splitk_check_geometry(32, (1 << 22) + 64, 64, 1, 64) == bd.ERR_SHAPE
    assert sk.splitk_check_geometry(32, 64, 32 * 5000, 5000, 32) == bd.ERR_SPLIT


# fake device addresses: validation rejects every call below before any CUDA call
A0, B0, P0, O0, W0 = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000
GOOD = dict(M=32, N=64, K=128, S=2, kps=64)


def call_gemm(L, A=A0, B=B0, P=P0, M=32, N=64, K=128, S=2, kps=64, dtype=bd.BF16):
    return L.gemm_splitk_bt(A, B, P, M, N, K, S, kps, dtype, None)


def test_gemm_rejections(L):
    assert call_gemm(L, M=48) == bd.ERR_SHAPE
    assert call_gemm(L, N=32) == bd.ERR_SHAPE
    assert call_gemm(L, S=3) == bd.ERR_SPLIT
    assert call_gemm(L, dtype=7) == bd.ERR_DTYPE
    assert call_gemm(L, A=0) == bd.ERR_NULL
    assert call_gemm(L, B=0) == bd.ERR_NULL
    assert call_gemm(L, P=0) == bd.ERR_NULL
    assert call_gemm(L, A=A0 + 8) == bd.ERR_ALIGN
    assert call_gemm(L, P=P0 + 4) == bd.ERR_ALIGN
    # partials [2,32,64] F32 = 16 KiB; A [32,128] BF16 = 8 KiB
    assert call_gemm(L, P=A0) == bd.ERR_ALIAS
    assert call_gemm(L, P=A0 + 8192 - 16) == bd.ERR_ALIAS
    assert call_gemm(L, P=B0 - 16384 + 16) == bd.ERR_ALIAS
    # the shape rule is reported before pointer problems
    assert call_gemm(L, M=48, A=0) == bd.ERR_SHAPE


def test_reduce_rejections(L):
    assert L.splitk_reduce(P0, O0, 2, 0, 64, None) == bd.ERR_SHAPE
    assert L.splitk_reduce(P0, O0, 0, 32, 64, None) == bd.ERR_SPLIT
    assert L.splitk_reduce(0, O0, 2, 32, 64, None) == bd.ERR_NULL
    assert L.splitk_reduce(P0, 0, 2, 32, 64, None) == bd.ERR_NULL
    assert L.splitk_reduce(P0 + 4, O0, 2, 32, 64, None) == bd.ERR_ALIGN
    assert L.splitk_reduce(P0, P0 + 16384 - 16, 2, 32, 64, None) == bd.ERR_ALIAS


def test_gemm_bt_rejections(L):
    need = sk.gemm_bt_workspace_bytes(32, 64, 128, 2, 64)
    assert need >= 2 * 32 * 64 * 4

    def call(out=O0, ws=W0, wsb=need, fused=0, **kw):
        g = dict(GOOD, **kw)
        return L.gemm_bt(A0, B0, out, ws, wsb, g["M"], g["N"], g["K"], g["S"], g["kps"], bd.BF16,
                         fused, None)

    assert call(M=96, K=100) == bd.ERR_SHAPE
    assert call(fused=2) == bd.ERR_CONFIG
    assert call(out=0) == bd.ERR_NULL
    assert call(ws=0) == bd.ERR_NULL
    assert call(wsb=need - 4) == bd.ERR_WORKSPACE
    assert call(ws=W0 + 8) == bd.ERR_ALIGN
    assert call(out=A0) == bd.ERR_ALIAS
    assert call(ws=O0) == bd.ERR_ALIAS
    assert call(ws=B0 + 64) == bd.ERR_ALIAS
    assert call(fused=2) == bd.ERR_CONFIG
    assert call(fused=4) == bd.ERR_CONFIG
    # the fused calls take the same workspace (the two-kernel path runs where no cluster sums)
    assert call(ws=0, fused=1) == bd.ERR_NULL
    assert call(wsb=0, fused=1) == bd.ERR_WORKSPACE
    assert L.gemm_bt_workspace_init(0, 64, None) == bd.ERR_NULL
    assert L.gemm_bt_workspace_init(W0 + 4, 64, None) == bd.ERR_ALIGN


def test_workspace_bytes(L):
    # the F32 partials [splits, M, N]
    assert sk.gemm_bt_workspace_bytes(256, 1024, 2048, 2, 1024) == 2 * 256 * 1024 * 4
    assert sk.gemm_bt_workspace_bytes(64, 128, 160, 3, 64) == 3 * 64 * 128 * 4
    assert sk.gemm_bt_workspace_bytes(64, 128, 160, 3, 64, 1) == sk.gemm_bt_workspace_bytes(64, 128, 160, 3, 64, 0)
    assert sk.gemm_bt_workspace_bytes(64, 128, 160, 2, 64) == 0


def test_status_strings(L):
    for code in range(-10, 1):
        assert sk.splitk_status_string(code) != "unknown status"
    assert sk.splitk_status_string(-99) == "unknown status"


def test_tile_override_validation(L):
    for bn, ch, kb in [(32, 0, 0), (0, 3, 0), (512, 1, 0), (64, 32, 0), (0, 0, 3), (0, 0, 8)]:
        with pytest.raises(sk.SplitKError):
            sk.splitk_set_tile_override(bn, ch, kb)
    sk.splitk_set_tile_override(0, 0, 0)


def test_describe_launch_plans(L):
    sk.splitk_set_tile_override(0, 0, 0)
    d = sk.splitk_describe_launch(256, 1024, 2048, 2, 1024, "bf16", fused=0)
    assert d["path"] == 0 and d["kernels_per_call"] == 2
    assert d["grid_x"] * d["bn"] == 1024 and d["grid_y"] == 2
    assert d["grid_z"] == 2 * d["chunks"] and d["cluster"] == d["chunks"]
    assert d["chunk_len"] * d["chunks"] >= 1024 and d["chunk_len"] % 32 == 0
    assert d["smem_bytes"] <= 227 * 1024
    f = sk.splitk_describe_launch(256, 1024, 2048, 2, 1024, "bf16", fused=1)
    assert f["fused_in_kernel"] == 1 and f["kernels_per_call"] == 1
    # the headline's 2 splits x chunks share one cluster: the split sum stays on chip
    assert f["split_sum"] == 2 and f["cluster"] == 2 * f["chunks"] <= 8
    # same chunking in both modes: the fused output equals the two-kernel output bitwise
    assert (f["bn"], f["chunks"], f["chunk_len"]) == (d["bn"], d["chunks"], d["chunk_len"])
    # F32 runs 3xTF32 on the tensor cores: 32-element k-blocks, stages twice the loaded bytes,
    # the split sum in the launch as for 16-bit operands
    g = sk.splitk_describe_launch(96, 512, 2048, 4, 512, "f32", fused=1)
    assert g["path"] == 2 and g["kernels_per_call"] == 1 and g["fused_in_kernel"] == 1
    g0 = sk.splitk_describe_launch(96, 512, 2048, 4, 512, "f32", fused=0)
    assert g0["path"] == 2 and g0["kernels_per_call"] == 2
    assert g0["chunk_len"] % 32 == 0 and g0["smem_bytes"] <= 227 * 1024
    # more splits than one cluster holds: gemm_bt(fused=1) runs the two kernels
    # (bitwise the same result), since summing through global memory measured slower
    h = sk.splitk_describe_launch(32, 64, 32 * 32, 32, 32, "bf16", fused=1)
    assert h["fused_in_kernel"] == 0 and h["kernels_per_call"] == 2 and h["split_sum"] == 0
    for S in (1, 2, 4, 8, 16):
        e = sk.splitk_describe_launch(32, 512, 2048, S, 2048 // S, "f16", fused=1)
        assert e["smem_bytes"] <= 226 * 1024
        if e["fused_in_kernel"]:
            assert e["split_sum"] == 2 and e["cluster"] == S * e["chunks"] <= 8 and e["kernels_per_call"] == 1
        else:
            assert e["split_sum"] == 0 and e["cluster"] == e["chunks"] <= 8 and e["kernels_per_call"] == 2
    # three splits: cluster sizes are powers of two, so no cluster holds them
    k = sk.splitk_describe_launch(64, 128, 160, 3, 64, "f16", fused=1)
    assert k["fused_in_kernel"] == 0 and k["split_sum"] == 0


def test_describe_launch_override(L):
    try:
        sk.splitk_set_tile_override(64, 2)
        d = sk.splitk_describe_launch(64, 128, 160, 3, 64, "bf16")
        assert d["bn"] == 64 and d["chunks"] == 2 and d["chunk_len"] == 32
        # K = 160 is not a multiple of 64: one k-block per stage, 2-D loads
        assert d["kblocks_per_stage"] == 1 and d["three_d"] == 0
        # a width that does not divide N keeps the automatic width
        sk.splitk_set_tile_override(256, 1)
        d = sk.splitk_describe_launch(64, 128, 160, 3, 64, "bf16")
        assert d["bn"] in (64, 128)
        # stages of 2 k-blocks as 3-D boxes where K and k_per_split allow it
        sk.splitk_set_tile_override(128, 4, 2)
        d = sk.splitk_describe_launch(256, 1024, 2048, 2, 1024, "bf16")
        assert d["kblocks_per_stage"] == 2 and d["three_d"] == 1 and d["chunk_len"] % 64 == 0
    finally:
        sk.splitk_set_tile_override(0, 0, 0)


def test_unbuilt_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(bd, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(bd, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        bd.lib()


def test_prepare_rejections(L):
    W, B = 0x10000000, 0x20000000
    assert L.splitk_prepare_bt(W, B, 48, 64, bd.BF16, None) == bd.ERR_SHAPE
    assert L.splitk_prepare_bt(W, B, 64, 96, bd.BF16, None) == bd.ERR_SHAPE
    assert L.splitk_prepare_bt(W, B, 0, 64, bd.BF16, None) == bd.ERR_SHAPE
    assert L.splitk_prepare_bt(W, B, 64, 64, 9, None) == bd.ERR_DTYPE
    assert L.splitk_prepare_bt(0, B, 64, 64, bd.BF16, None) == bd.ERR_NULL
    assert L.splitk_prepare_bt(W, 0, 64, 64, bd.BF16, None) == bd.ERR_NULL
    assert L.splitk_prepare_bt(W + 2, B, 64, 64, bd.BF16, None) == bd.ERR_ALIGN
    # W is 64 * 64 * 2 = 8 KiB; a B starting inside it overlaps
    assert L.splitk_prepare_bt(W, W + 8192 - 16, 64, 64, bd.BF16, None) == bd.ERR_ALIAS


def test_host_staging_bytes(L):
    # count A slots, count output slots (each group packed), one gemm_bt workspace
    M, N, K, S, kps = 256, 1024, 2048, 2, 1024
    ws = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
    assert sk.gemm_bt_host_staging_bytes(8, M, N, K, S, kps, "bf16") == 8 * M * K * 2 + 8 * M * N * 4 + ws
    assert sk.gemm_bt_host_staging_bytes(1, 32, 64, 128, 2, 64, "f32") == \
        32 * 128 * 4 + 32 * 64 * 4 + sk.gemm_bt_workspace_bytes(32, 64, 128, 2, 64)
    assert sk.gemm_bt_host_staging_bytes(0, M, N, K, S, kps, "bf16") == 0
    assert sk.gemm_bt_host_staging_bytes((1 << 16) + 1, M, N, K, S, kps, "bf16") == 0
    assert sk.gemm_bt_host_staging_bytes(2, 48, N, K, S, kps, "bf16") == 0
    assert L.gemm_bt_host_staging_bytes(2, M, N, K, S, kps, 9) == 0


def test_host_batch_rejections(L):
    """Every rejection happens before the library touches CUDA (no GPU here)."""
    M, N, K, S, kps = 32, 64, 128, 2, 64
    need = sk.gemm_bt_host_staging_bytes(2, M, N, K, S, kps, "bf16")
    Ah, Oh, ST = 0x50000000, 0x60000000, 0x70000000
    Bs = bd.pointer_array([B0, B0])

    def call(A=Ah, B=Bs, O=Oh, count=2, st=ST, stb=need, fused=0, opc=0, dtype=bd.BF16, **kw):
        g = dict(GOOD, **kw)
        b = ctypes.cast(B, ctypes.c_void_p) if isinstance(B, ctypes.Array) else B
        return L.gemm_bt_host_batch(A, b, O, count, st, stb, g["M"], g["N"], g["K"], g["S"], g["kps"],
                                    dtype, fused, opc, None)

    assert call(M=48) == bd.ERR_SHAPE
    assert call(S=3) == bd.ERR_SPLIT
    assert call(dtype=5) == bd.ERR_DTYPE
    assert call(count=0) == bd.ERR_CONFIG
    assert call(count=(1 << 16) + 1) == bd.ERR_CONFIG
    assert call(opc=-1) == bd.ERR_CONFIG
    assert call(fused=2) == bd.ERR_CONFIG
    assert call(A=0) == bd.ERR_NULL
    assert call(B=0) == bd.ERR_NULL
    assert call(O=0) == bd.ERR_NULL
    assert call(st=0) == bd.ERR_NULL
    assert call(B=bd.pointer_array([B0, 0])) == bd.ERR_NULL
    assert call(st=ST + 8) == bd.ERR_ALIGN
    assert call(B=bd.pointer_array([B0, B0 + 2])) == bd.ERR_ALIGN
    assert call(stb=need - 16) == bd.ERR_WORKSPACE
    # A_host [2,32,128] BF16 = 16 KiB; out_host [2,32,64] F32 = 16 KiB
    assert call(O=Ah + 16384 - 16) == bd.ERR_ALIAS
    assert call(B=bd.pointer_array([B0, ST + need - 64])) == bd.ERR_ALIAS
    assert call(st=Oh - 64) == bd.ERR_ALIAS
    assert call(M=48, A=0) == bd.ERR_SHAPE


def test_batch_rejections(L):
    """gemm_bt_batch checks every operation and the outputs against one
    another, every input and the workspace before it touches CUDA (no GPU
    here)."""
    M, N, K, S, kps = 32, 64, 128, 2, 64
    a_bytes, o_bytes = M * K * 2, M * N * 4                     # 8 KiB each
    need = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)

    def call(A=(A0, A0 + a_bytes), B=(B0, B0), O=(O0, O0 + o_bytes), count=2, ws=W0, wsb=need, fused=1,
             dtype=bd.BF16, **kw):
        g = dict(GOOD, **kw)
        arrs = [ctypes.cast(bd.pointer_array(list(x)), ctypes.c_void_p) if x is not None else None
                for x in (A, B, O)]
        return L.gemm_bt_batch(*arrs, count, ws, wsb, g["M"], g["N"], g["K"], g["S"], g["kps"], dtype, fused,
                               None)

    assert call(count=0) == bd.ERR_CONFIG
    assert call(count=(1 << 16) + 1) == bd.ERR_CONFIG
    assert call(fused=2) == bd.ERR_CONFIG
    assert call(fused=3) == bd.ERR_CONFIG
    assert call(A=None) == bd.ERR_NULL
    assert call(O=None) == bd.ERR_NULL
    assert call(B=(B0, 0)) == bd.ERR_NULL
    assert call(M=48) == bd.ERR_SHAPE
    assert call(S=3) == bd.ERR_SPLIT
    assert call(dtype=5) == bd.ERR_DTYPE
    assert call(O=(O0, O0 + 8)) == bd.ERR_ALIGN
    assert call(wsb=need - 16) == bd.ERR_WORKSPACE
    assert call(O=(O0, O0 + o_bytes - 16)) == bd.ERR_ALIAS            # two outputs overlap
    assert call(O=(O0, A0 + 64)) == bd.ERR_ALIAS                      # an output over another call's input
    assert call(A=(A0, O0 + 256)) == bd.ERR_ALIAS                     # an input over another call's output
    assert call(O=(O0, W0 + 16)) == bd.ERR_ALIAS                      # an output over the workspace
    assert call(M=48, A=None) == bd.ERR_NULL                          # the arrays first


def test_batch_alias_rule(L):
    """gemm_bt_batch's overlap check against brute force on seeded random
    layouts: every layout where some output overlaps another output, an input
    or the workspace is rejected with ERR_ALIAS before any device work.
    (Layouts that pass would launch on these made-up addresses, so they are
    not called: the GPU tests run the accepted layouts on real buffers.)"""
    import numpy as np

    M, N, K, S, kps = 32, 64, 128, 2, 64
    a_bytes, b_bytes, o_bytes = M * K * 2, N * K * 2, M * N * 4
    ws_bytes = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
    rng = np.random.Generator(np.random.PCG64(11))
    seen = {True: 0, False: 0}
    for _ in range(300):
        count = int(rng.integers(1, 5))
        slot = lambda: 0x10000000 + 1024 * int(rng.integers(0, 160))   # 16-byte aligned, often overlapping
        A = [slot() for _ in range(count)]
        B = [slot() for _ in range(count)]
        O = [slot() for _ in range(count)]
        W = slot()
        ranges = [(a, a + a_bytes, False) for a in A] + [(b, b + b_bytes, False) for b in B] + \
                 [(o, o + o_bytes, True) for o in O] + [(W, W + ws_bytes, True)]
        alias = any(r[2] and q is not r and r[0] < q[1] and q[0] < r[1] for r in ranges for q in ranges)
        seen[alias] += 1
        if not alias:
            continue
        arrs = [ctypes.cast(bd.pointer_array(x), ctypes.c_void_p) for x in (A, B, O)]
        st = L.gemm_bt_batch(*arrs, count, W, ws_bytes, M, N, K, S, kps, bd.BF16, 1, None)
        assert st == bd.ERR_ALIAS, (A, B, O, W, st)
    assert seen[True] > 20, seen


def test_choose_splits_is_legal(L, orc):
    """The model's choice is always a legal geometry drawn from the candidates:
    the largest candidate whose estimate is within 2% of the smallest."""
    for M in (32, 96, 256):
        for N in (64, 512, 1024):
            for K in (32, 128, 160, 512, 2048, 4096):
                for dt in ("bf16", "f16", "f32"):
                    for fused in (0, 1):
                        S, kps, t = sk.splitk_choose_splits(M, N, K, dt, fused)
                        assert orc.contract(M, N, K, S, kps) == 0, (M, N, K, S, kps)
                        assert kps % 32 == 0 and all(v is not None and v > 0 for v in t.values())
                        low = min(t.values())
                        best = max(c for c, v in t.items() if v <= low * 1.02)
                        k_best = -(-(-(-K // best)) // 32) * 32
                        assert (S, kps) == (-(-K // k_best), k_best)
                        legal = set()
                        for n in (1, 2, 4, 8, 16):
                            k = -(-(-(-K // n)) // 32) * 32
                            legal.add((-(-K // k), k))
                        assert (S, kps) in legal


def test_choose_splits_rejections(L):
    out = (ctypes.c_int64 * 2)()
    assert L.splitk_choose_splits(48, 64, 128, bd.BF16, 0, ctypes.byref(out, 0), ctypes.byref(out, 8), None) \
        == bd.ERR_SHAPE
    assert L.splitk_choose_splits(32, 96, 128, bd.BF16, 0, ctypes.byref(out, 0), ctypes.byref(out, 8), None) \
        == bd.ERR_SHAPE
    assert L.splitk_choose_splits(32, 64, 128, 7, 0, ctypes.byref(out, 0), ctypes.byref(out, 8), None) \
        == bd.ERR_DTYPE
    assert L.splitk_choose_splits(32, 64, 128, bd.BF16, 2, ctypes.byref(out, 0), ctypes.byref(out, 8), None) \
        == bd.ERR_CONFIG
    assert L.splitk_choose_splits(32, 64, 128, bd.BF16, 0, None, ctypes.byref(out, 8), None) == bd.ERR_NULL


def test_autotune_rejections(L):
    """Every rejection happens before the library touches CUDA (no GPU here)."""
    M, N, K = 32, 64, 128
    need16 = max(sk.gemm_bt_workspace_bytes(M, N, K, -(-K // k), k) for k in (32, 64, 128))
    s, k = ctypes.c_int64(), ctypes.c_int64()

    def call(A=A0, B=B0, O=O0, W=W0, wsb=need16, M=M, N=N, K=K, dtype=bd.BF16, fused=0, reps=5):
        return L.splitk_autotune_splits(A, B, O, W, wsb, M, N, K, dtype, fused, reps, None, ctypes.byref(s),
                                        ctypes.byref(k), None)

    assert call(M=48) == bd.ERR_SHAPE
    assert call(dtype=9) == bd.ERR_DTYPE
    assert call(fused=2) == bd.ERR_CONFIG
    assert call(reps=0) == bd.ERR_CONFIG
    assert call(reps=1001) == bd.ERR_CONFIG
    assert call(A=0) == bd.ERR_NULL
    assert call(O=0) == bd.ERR_NULL
    assert call(W=0) == bd.ERR_NULL
    assert call(A=A0 + 8) == bd.ERR_ALIGN
    assert call(O=A0) == bd.ERR_ALIAS
    assert call(wsb=16) == bd.ERR_WORKSPACE
    assert L.splitk_autotune_splits(A0, B0, O0, W0, need16, M, N, K, bd.BF16, 0, 5, None, None, ctypes.byref(k),
                                    None) == bd.ERR_NULL


def test_kn_rejections(L):
    """The [K,N] entry points check exactly what their [N,K] twins check."""
    need = sk.gemm_bt_workspace_bytes(32, 64, 128, 2, 64)
    for fn_bt, fn_kn in ((L.gemm_splitk_bt, L.gemm_splitk_kn),):
        for kw in (dict(M=48), dict(N=32), dict(S=3), dict(dtype=7), dict(A=0), dict(B=0), dict(P=0),
                   dict(A=A0 + 8), dict(P=P0 + 4), dict(P=A0), dict(P=B0 - 16384 + 16)):
            g = dict(dict(A=A0, B=B0, P=P0, M=32, N=64, K=128, S=2, kps=64, dtype=bd.BF16), **kw)
            args = (g["A"], g["B"], g["P"], g["M"], g["N"], g["K"], g["S"], g["kps"], g["dtype"], None)
            assert fn_kn(*args) == fn_bt(*args) != 0, kw
    for kw in (dict(out=0), dict(ws=0), dict(wsb=need - 4), dict(ws=W0 + 8), dict(out=A0), dict(ws=O0),
               dict(fused=2), dict(M=96, K=100)):
        g = dict(dict(out=O0, ws=W0, wsb=need, fused=0, M=32, N=64, K=128), **kw)
        args = (A0, B0, g["out"], g["ws"], g["wsb"], g["M"], g["N"], g["K"], 2, 64, bd.BF16, g["fused"], None)
        assert L.gemm_kn(*args) == L.gemm_bt(*args) != 0, kw
