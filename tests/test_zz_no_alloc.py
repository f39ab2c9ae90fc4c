"""gemm_bt_noalloc: gemm_bt for callers that cannot allocate device memory.

Hosts such as inference-runtime plugins hand an operator only its input and
output buffers and forbid allocation while it runs, so they have no workspace
to pass to gemm_bt.  gemm_bt_noalloc runs the same operation on a scratch
array the library keeps in device memory.  These tests call it through the C
ABI and compare it with gemm_bt (given a caller workspace) on two calls in a
row with different operands, so a call that picked up the previous call's
scratch contents would fail.  The file is named to be collected last.
"""
import numpy as np
import pytest

from harness import TOL_FINAL, Guarded, device_operand, max_scaled_error, oracle_case, workspace

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sk():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    sk.splitk_set_tile_override(0, 0, 0)
    return sk


CASES = [
    (256, 1024, 2048, 2, 1024, "bf16"),   # the benchmark workload: splits summed inside the cluster
    (64, 128, 160, 3, 64, "f16"),         # three splits: no cluster holds them, two kernels
    (96, 512, 512, 16, 32, "bf16"),       # sixteen splits
    (96, 512, 2048, 4, 512, "f32"),       # F32 operands: two kernels
]


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}" for c in CASES])
def test_noalloc_matches_gemm_bt_on_two_calls(sk, case, fused):
    M, N, K, S, kps, dt = case
    for seed in (0, 5):
        ops, _, _, Or, SO = oracle_case(M, N, K, S, kps, dt, "uniform", seed)
        A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
        ws, nbytes = workspace(M, N, K, S, kps)
        ref = Guarded(M * N)
        sk.gemm_bt(A, B, ref.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
        got = Guarded(M * N)
        sk.gemm_bt_noalloc(A, B, got.data, M, N, K, S, kps, dt, fused=fused)
        assert sk.splitk_get_device_status() == 0
        assert got.guards_intact()
        g = got.numpy().reshape(M, N)
        r = ref.numpy().reshape(M, N)
        # against the workspace entry point, within the final-output tolerance
        assert max_scaled_error(g, r.astype(np.float64), SO) <= TOL_FINAL[dt]
        assert max_scaled_error(g, Or, SO) <= TOL_FINAL[dt]
        # the same kernels add the same numbers: equal bit for bit
        assert np.array_equal(g.view(np.uint32), r.view(np.uint32))


def test_noalloc_rejects_shapes_beyond_its_scratch(sk):
    from split_bf16_gemm_gb300 import binding as bd

    # partials: 2 * 2048 * 4096 * 4 bytes = 64 MiB, twice the scratch; one split
    # (exactly 32 MiB) still fits
    M, N, K = 2048, 4096, 4096
    assert sk.gemm_bt_workspace_bytes(M, N, K, 1, K) == bd.NOALLOC_MAX_BYTES
    assert sk.gemm_bt_workspace_bytes(M, N, K, 2, K // 2) > bd.NOALLOC_MAX_BYTES
    st = sk.lib().gemm_bt_noalloc(0x10000000, 0x20000000, 0x30000000, M, N, K, 2, K // 2, bd.BF16, 0, None)
    assert st == bd.ERR_WORKSPACE
    assert "scratch" in sk.splitk_last_error()
    # a shape that fits is accepted (and computed) right after the rejection
    ops, _, _, Or, SO = oracle_case(32, 64, 128, 2, 64, "bf16")
    out = Guarded(32 * 64)
    sk.gemm_bt_noalloc(device_operand(ops.A, "bf16"), device_operand(ops.B, "bf16"), out.data,
                       32, 64, 128, 2, 64, "bf16", fused=1)
    assert max_scaled_error(out.numpy().reshape(32, 64), Or, SO) <= TOL_FINAL["bf16"]
    assert out.guards_intact()
