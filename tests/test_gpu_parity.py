"""GPU parity: libsplitk through its C ABI against the F64 oracle.

Every case poisons the partials and the output (7.0) and puts 64 guards of
11.0 behind each; a NaN-poison pass removes the chance that a stale 7.0 lands
within tolerance.  Shapes cover the pages' workloads (the single tile, M96,
M256/N512, the M256/N1024 headline, the dtype x split sweep with the skinny,
short-K and short-final-split shapes) and the pages' test categories
(non-square, odd tile counts, long K, larger matrices).
"""
import numpy as np
import pytest

from harness import (TOL_FINAL, TOL_PARTIAL, Guarded, device_operand, max_scaled_error,
                     oracle_case, workspace)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    sk.splitk_set_tile_override(0, 0, 0)
    yield sk
    sk.splitk_set_tile_override(0, 0, 0)


WORKLOADS = [  # (M, N, K, splits, kps, dtype): the pages' workloads
    (32, 64, 128, 2, 64, "bf16"),
    (96, 512, 2048, 4, 512, "bf16"),
    (256, 512, 2048, 4, 512, "bf16"),
    (256, 512, 2048, 2, 1024, "bf16"),
    (256, 1024, 2048, 2, 1024, "bf16"),
]
SWEEP = []
for _dt in ("f32", "f16", "bf16"):
    for _S in (1, 2, 4, 8, 16):
        SWEEP.append((32, 512, 2048, _S, 2048 // _S, _dt))
        SWEEP.append((96, 512, 512, _S, 512 // _S, _dt))
    SWEEP.append((64, 128, 160, 3, 64, _dt))
CATEGORIES = [
    (32, 64, 32, 1, 32, "bf16"),         # single tile, one split
    (160, 192, 320, 3, 128, "bf16"),     # M tail past one 128-row tile, 3 N tiles, short final split
    (96, 320, 1024, 2, 512, "f16"),      # odd tile count along N (5 x 64)
    (64, 128, 8192, 4, 2048, "bf16"),    # long K
    (512, 2048, 4096, 4, 1024, "bf16"),  # larger matrices
    (32, 64, 64, 1, 128, "bf16"),        # k_per_split larger than K
    (288, 256, 96, 3, 32, "f16"),        # 32-long splits everywhere
    (64, 128, 2048, 64, 32, "bf16"),     # 64 splits: a fused call runs the two kernels
    (160, 192, 320, 3, 128, "f32"),      # F32 (3xTF32): M tail, short final split
    (64, 128, 8192, 4, 2048, "f32"),     # F32, long K
    (288, 256, 96, 3, 32, "f32"),        # F32, 32-long splits everywhere
]


def ids(cases):
    return [f"{dt}-M{M}N{N}K{K}S{S}" for M, N, K, S, kps, dt in cases]


def run_two_pass(sk, ops, S, kps, poison=7.0):
    M, N, K = ops.M, ops.N, ops.K
    A = device_operand(ops.A, ops.dtype)
    B = device_operand(ops.B, ops.dtype)
    P = Guarded(S * M * N, poison)
    out = Guarded(M * N, poison)
    sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, ops.dtype)
    sk.splitk_reduce(P.data, out.data, S, M, N)
    assert sk.splitk_get_device_status() == 0
    return A, B, P, out


def check_case(sk, case, poison=7.0, recipe="uniform"):
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt, recipe)
    A, B, P, out = run_two_pass(sk, ops, S, kps, poison)
    assert P.guards_intact() and out.guards_intact()
    ep = max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP)
    eo = max_scaled_error(out.numpy().reshape(M, N), Or, SO)
    assert ep <= TOL_PARTIAL, f"partials: max |err|/sum|ab| = {ep:.3e}"
    assert eo <= TOL_FINAL[dt], f"output: max |err|/sum|ab| = {eo:.3e}"
    return A, B, P, out


@pytest.mark.parametrize("case", WORKLOADS + SWEEP + CATEGORIES, ids=ids(WORKLOADS + SWEEP + CATEGORIES))
def test_two_pass_matches_oracle(lib, case):
    check_case(lib, case)


@pytest.mark.parametrize("case", WORKLOADS + CATEGORIES[:4] + SWEEP[-11:], ids=ids(WORKLOADS + CATEGORIES[:4] + SWEEP[-11:]))
def test_nan_poison(lib, case):
    check_case(lib, case, poison=float("nan"))


@pytest.mark.parametrize("case", WORKLOADS + SWEEP[::3] + CATEGORIES, ids=ids(WORKLOADS + SWEEP[::3] + CATEGORIES))
def test_gemm_bt_both_modes_bitwise(lib, case):
    """gemm_bt with fused = 0, 1 and 3 gives the two-kernel output bit for bit;
    fused = 0 and 3 leave gemm_splitk_bt's partials in the workspace."""
    sk = lib
    M, N, K, S, kps, dt = case
    A, B, P, out = check_case(sk, case)
    ref_out = out.numpy()
    ref_P = P.numpy()
    plan = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=1)
    for fused in (0, 1, 3):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
        assert sk.splitk_get_device_status() == 0
        assert o.guards_intact() and ws.guards_intact()
        assert np.array_equal(o.numpy().view(np.uint32), ref_out.view(np.uint32)), f"fused={fused}"
        w = ws.numpy()
        if fused in (0, 3) or plan["split_sum"] != 2:
            assert np.array_equal(w[:S * M * N].view(np.uint32), ref_P.view(np.uint32)), f"fused={fused}"
        else:
            assert np.all(w[:S * M * N] == 7.0), "fused=1 with the split sum on chip keeps no partials"


def test_fused_repeated_calls_and_overwrite(lib):
    """Many fused calls on one workspace and output stay bitwise the same, and a
    later call with other operands overwrites the output."""
    sk = lib
    M, N, K, S, kps, dt = 96, 512, 2048, 4, 512, "bf16"
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    ops2, _, _, Or2, SO2 = oracle_case(M, N, K, S, kps, dt, "uniform", 7)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    A2, B2 = device_operand(ops2.A, dt), device_operand(ops2.B, dt)
    ws, nbytes = workspace(M, N, K, S, kps)
    o = Guarded(M * N)
    first = None
    for i in range(6):
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
        r = o.numpy().copy()
        first = r if first is None else first
        assert np.array_equal(r.view(np.uint32), first.view(np.uint32))
    assert max_scaled_error(first.reshape(M, N), Or, SO) <= TOL_FINAL[dt]
    # back-to-back launches on one stream, same workspace and output
    sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
    sk.gemm_bt(A2, B2, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
    assert max_scaled_error(o.numpy().reshape(M, N), Or2, SO2) <= TOL_FINAL[dt]
    assert sk.splitk_get_device_status() == 0


def test_reads_follow_previous_kernel(lib):
    """A kernel launched just before (here a torch copy into A) is complete
    before the GEMM reads A: the dependent-launch wait covers it."""
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    src = device_operand(ops.A, dt)
    B = device_operand(ops.B, dt)
    ws, nbytes = workspace(M, N, K, S, kps)
    for _ in range(3):
        A = torch.zeros_like(src)
        o = Guarded(M * N)
        A.copy_(src)
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
        assert max_scaled_error(o.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt]


INT_CASES = [
    (32, 64, 32, 1, 32, "bf16"),
    (32, 64, 128, 2, 64, "bf16"),
    (64, 128, 160, 3, 64, "f16"),
    (256, 1024, 2048, 2, 1024, "bf16"),
    (96, 512, 2048, 4, 512, "f32"),
]


@pytest.mark.parametrize("case", INT_CASES, ids=ids(INT_CASES))
def test_integer_inputs_bitwise(lib, case):
    """Integer operands in [-8,8]: every product and partial sum is exact in
    F32, so the GPU must equal the oracle exactly."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt, "integers", 3)
    _, _, P, out = run_two_pass(sk, ops, S, kps)
    assert np.array_equal(P.numpy().reshape(S, M, N).astype(np.float64), Pr)
    assert np.array_equal(out.numpy().reshape(M, N).astype(np.float64), Or)
    assert P.guards_intact() and out.guards_intact()


def test_golden_int_tile(lib):
    from test_oracle_pins import load_int_tile

    import splitk_inputs as gen

    P_ref, O_ref = load_int_tile()
    ops = gen.integers(32, 64, 128, "bf16", seed=3)
    _, _, P, out = run_two_pass(lib, ops, 2, 64)
    assert np.array_equal(P.numpy().reshape(2, 32, 64).astype(np.float64), P_ref)
    assert np.array_equal(out.numpy().reshape(32, 64).astype(np.float64), O_ref)


def test_closed_forms(lib):
    sk = lib
    ops, *_ = oracle_case(64, 128, 160, 3, 64, "bf16", "ones")
    _, _, P, out = run_two_pass(sk, ops, 3, 64)
    P = P.numpy().reshape(3, 64, 128)
    assert np.all(P[0] == 64) and np.all(P[1] == 64) and np.all(P[2] == 32)
    assert np.all(out.numpy() == 160)
    ops, *_ = oracle_case(64, 128, 256, 2, 128, "f16", "identity_b", 4)
    _, _, P, out = run_two_pass(sk, ops, 2, 128)
    a = ops.A.view(np.float16).astype(np.float32)
    assert np.array_equal(out.numpy().reshape(64, 128), a[:, :128])


def test_zero_first_row_and_split_independence(lib):
    sk = lib
    outs = []
    for S in (1, 2, 4, 8, 16):
        ops, Pr, SP, Or, SO = oracle_case(96, 512, 512, S, 512 // S, "bf16")
        _, _, P, out = run_two_pass(sk, ops, S, 512 // S)
        o = out.numpy().reshape(96, 512)
        assert np.all(o[0] == 0) and np.all(P.numpy().reshape(S, 96, 512)[:, 0] == 0)
        outs.append(o.astype(np.float64))
    for o in outs[1:]:
        assert max_scaled_error(o, outs[0], SO) <= 2 * TOL_FINAL["bf16"]
        assert max_scaled_error(o, outs[0], SO) <= 1e-5   # F32 accumulation, much tighter in practice


TILINGS = [(bn, ch, kb) for bn in (64, 128, 256) for ch in (1, 2, 4, 8) for kb in (1, 2, 4)]


@pytest.mark.parametrize("case", [(64, 128, 160, 3, 64, "bf16"), (256, 1024, 2048, 2, 1024, "bf16"),
                                  (96, 512, 2048, 4, 512, "f16"), (64, 128, 160, 3, 64, "f32"),
                                  (256, 1024, 2048, 2, 1024, "f32")],
                         ids=["K160", "headline", "M96", "K160-f32", "headline-f32"])
def test_every_tiling(lib, case):
    """Each tile width and chunk count (including chunks past a short final
    split, which hold no K at all) gives a correct result, and the fused path
    matches the two-kernel path bitwise under the same tiling."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A = device_operand(ops.A, dt)
    B = device_operand(ops.B, dt)
    try:
        for bn, ch, kb in TILINGS:
            sk.splitk_set_tile_override(bn, ch, kb)
            P = Guarded(S * M * N)
            out = Guarded(M * N)
            fused = Guarded(M * N)
            ws, nbytes = workspace(M, N, K, S, kps)
            sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
            sk.splitk_reduce(P.data, out.data, S, M, N)
            sk.gemm_bt(A, B, fused.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
            assert sk.splitk_get_device_status() == 0
            assert P.guards_intact() and out.guards_intact() and fused.guards_intact()
            assert max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL, (bn, ch, kb)
            assert max_scaled_error(out.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt], (bn, ch, kb)
            assert np.array_equal(fused.numpy().view(np.uint32), out.numpy().view(np.uint32)), (bn, ch, kb)
    finally:
        sk.splitk_set_tile_override(0, 0, 0)


@pytest.mark.parametrize("case", [(256, 1024, 2048, 2, 1024, "bf16"), (96, 512, 2048, 4, 512, "bf16"),
                                  (256, 512, 2048, 4, 512, "f16"), (160, 512, 640, 2, 320, "bf16"),
                                  (128, 512, 1024, 2, 512, "f32")],
                         ids=["headline", "M96", "M256N512-f16", "M160-tail", "f32"])
def test_tile_width_does_not_change_bits(lib, case):
    """For a given chunking, the tile width (64, 128 or 256 columns) does not
    change one bit of the partials: each output element gets the same MMA K
    steps in the same order.  The compact layout inside graph captures relies
    on this when it widens a plan's tiles."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A = device_operand(ops.A, dt)
    B = device_operand(ops.B, dt)
    try:
        for ch in (1, 2, 4):
            got = {}
            for bn in (64, 128, 256):
                sk.splitk_set_tile_override(bn, ch, 0)
                d = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=0)
                if d["bn"] != bn or d["chunks"] != ch:
                    continue
                P = Guarded(S * M * N)
                sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
                assert sk.splitk_get_device_status() == 0 and P.guards_intact()
                got[bn] = P.numpy().view(np.uint32).copy()
                assert max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL, (bn, ch)
            widths = sorted(got)
            assert len(widths) >= 2, (ch, widths)
            for w in widths[1:]:
                assert np.array_equal(got[widths[0]], got[w]), (ch, widths[0], w)
    finally:
        sk.splitk_set_tile_override(0, 0, 0)


def test_cuda_graph_capture_and_side_stream(lib):
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A = device_operand(ops.A, dt)
    B = device_operand(ops.B, dt)
    nbytes = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    ws2 = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    sk.gemm_bt_workspace_init(ws2, nbytes)
    outs = [torch.full((M, N), 7.0, device="cuda") for _ in range(2)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sk.gemm_bt(A, B, outs[0], ws, nbytes, M, N, K, S, kps, dt, fused=0)
        sk.gemm_bt(A, B, outs[1], ws2, nbytes, M, N, K, S, kps, dt, fused=1)
    for _ in range(3):
        outs[0].fill_(7.0)
        outs[1].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for o in outs:
            assert max_scaled_error(o.cpu().numpy(), Or, SO) <= TOL_FINAL[dt]
        assert torch.equal(outs[0], outs[1])
    assert sk.splitk_get_device_status() == 0


def test_bounded_wait_reports_and_context_survives(lib):
    sk = lib
    from split_bf16_gemm_gb300 import binding as bd

    assert sk.splitk_get_device_status() == 0
    assert sk.splitk_selftest_bounded_wait(2_000_000) == bd.ERR_DEVICE_TIMEOUT
    assert sk.splitk_get_device_status() == 0          # read-and-clear
    check_case(sk, (32, 64, 128, 2, 64, "bf16"))        # the context is still usable


def test_kernel_timeout_path_reports_and_context_survives(lib):
    """The tensor-core kernel's own time-out path: in a fused launch the wait
    for the final accumulator gives up at once, while the last MMAs still run
    (a self-test entry point).  The launch records the time-out, still sends
    and awaits every cluster message, waits for its MMAs before freeing its
    tensor memory and finishes inside its output's bounds; the context stays
    usable: the next calls match the oracle, and a run of launches after it
    still gets its tensor memory."""
    sk = lib
    from split_bf16_gemm_gb300 import binding as bd

    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    assert sk.splitk_get_device_status() == 0
    for _ in range(3):
        out = Guarded(M * N)
        assert sk.splitk_selftest_kernel_timeout(A, B, out.data, M, N, K, S, kps, dt) == bd.ERR_DEVICE_TIMEOUT
        assert out.guards_intact()
    assert sk.splitk_get_device_status() == 0          # read-and-clear
    check_case(sk, (M, N, K, S, kps, dt))               # parity on the same context
    ws, nbytes = workspace(M, N, K, S, kps)
    o = Guarded(M * N)
    for _ in range(20):
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
    assert sk.splitk_get_device_status() == 0
    assert max_scaled_error(o.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt] and o.guards_intact()
    # a call that would not sum its splits inside the launch is refused
    assert sk.splitk_selftest_kernel_timeout(A, B, o.data, M, N, K, 8, 256, dt) == bd.ERR_CONFIG


PREP_CASES = [(32, 64, "bf16"), (160, 128, "f16"), (96, 320, "f32"), (2048, 1024, "bf16"), (4096, 2048, "f16")]


@pytest.mark.parametrize("case", PREP_CASES, ids=[f"{c[2]}-K{c[0]}N{c[1]}" for c in PREP_CASES])
def test_prepare_matches_oracle_bitwise(lib, case):
    """Weight preparation B[n,k] = W[k,n] equals the oracle's transpose bit for
    bit, leaves the guards behind B intact, and a GEMM on the prepared weight
    equals one on the oracle-prepared weight bit for bit."""
    import oracle
    import splitk_inputs as gen

    sk = lib
    K, N, dt = case
    w = gen.weight_kn(K, N, dt, seed=K ^ N)
    ref = oracle.transpose(w)
    W = device_operand(w, dt)
    esz = 4 if dt == "f32" else 2
    guard_words = 64
    Bbuf = torch.full((N * K * esz // 4 + guard_words,), 7.0, dtype=torch.float32, device="cuda")
    Bbuf[N * K * esz // 4:] = 11.0
    B = Bbuf[:N * K * esz // 4].view(torch.int32)
    sk.splitk_prepare_bt(W, B, K, N, dt)
    torch.cuda.synchronize()
    got = B.cpu().numpy().view(np.uint8)
    assert np.array_equal(got, np.ascontiguousarray(ref).view(np.uint8).reshape(-1))
    assert torch.all(Bbuf[N * K * esz // 4:] == 11.0)
    if K >= 64 and dt != "f32":
        M = 96
        kps = -(-(K // 2) // 32) * 32          # two splits where K allows, k_per_split a multiple of 32
        S = -(-K // kps)
        ops = gen.uniform(M, N, K, dt, seed=1)
        A = device_operand(ops.A, dt)
        Bdev = B.view(torch.bfloat16 if dt == "bf16" else torch.float16).view(N, K)
        Bref = device_operand(ref, dt)
        o1, o2 = Guarded(M * N), Guarded(M * N)
        ws, nbytes = workspace(M, N, K, S, kps)
        sk.gemm_bt(A, Bdev, o1.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=0)
        sk.gemm_bt(A, Bref, o2.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=0)
        assert np.array_equal(o1.numpy().view(np.uint32), o2.numpy().view(np.uint32))
    assert sk.splitk_get_device_status() == 0


# (M, N, K, splits, kps, dtype, count, ops_per_copy)
HOST_CASES = [(64, 128, 160, 3, 64, "bf16", 5, 2), (96, 512, 2048, 4, 512, "f16", 3, 0),
              (32, 64, 128, 2, 64, "f32", 4, 1), (256, 1024, 2048, 2, 1024, "bf16", 4, 0)]


def host_operand(bits_list, dtype, pinned):
    flat = np.concatenate([np.ascontiguousarray(b).reshape(-1) for b in bits_list])
    if dtype == "f32":
        t = torch.from_numpy(flat.astype(np.float32))
    else:
        t = torch.from_numpy(flat.view(np.int16)).view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("case", HOST_CASES, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}x{c[6]}g{c[7]}"
                                                  for c in HOST_CASES])
def test_host_batch_matches_device_call_and_oracle(lib, case):
    """gemm_bt_host_batch: host activations in, host results out, each
    operation bitwise the device-resident gemm_bt result for its operands and
    within the pages' tolerance of the oracle; pinned and pageable host
    memory; guards behind the host output intact."""
    from harness import GUARD_VALUE, GUARDS

    sk = lib
    M, N, K, S, kps, dt, count, opc = case
    cs = [oracle_case(M, N, K, S, kps, dt, "uniform", seed) for seed in range(count)]
    Bs = [device_operand(c[0].B, dt) for c in cs]
    ref = []
    for c, B in zip(cs, Bs):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_bt(device_operand(c[0].A, dt), B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=0)
        ref.append(o.numpy().reshape(M, N))
    sb = sk.gemm_bt_host_staging_bytes(count, M, N, K, S, kps, dt)
    for pinned in (True, False):
        A_host = host_operand([c[0].A for c in cs], dt, pinned)
        for fused in (0, 1):
            staging = torch.zeros(sb // 4 + 16, dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            out_host = torch.full((count * M * N + GUARDS,), 7.0, dtype=torch.float32)
            out_host[count * M * N:] = GUARD_VALUE
            out_host = out_host.pin_memory() if pinned else out_host
            stream = torch.cuda.Stream()
            sk.gemm_bt_host_batch(A_host, Bs, out_host, count, staging, sb, M, N, K, S, kps, dt,
                                  fused=fused, ops_per_copy=opc, stream=stream)
            stream.synchronize()
            assert sk.splitk_get_device_status(stream) == 0
            if fused == 1 and dt == "bf16" and (M, N) == (256, 1024):
                # two operations per copy, each pair in one launch
                assert sk.splitk_last_launch()["group"] == 2
            got = out_host.numpy()
            assert np.all(got[count * M * N:] == GUARD_VALUE)
            for i, c in enumerate(cs):
                oi = got[i * M * N:(i + 1) * M * N].reshape(M, N)
                assert np.array_equal(oi.view(np.uint32), ref[i].view(np.uint32)), (pinned, fused, i)
                assert max_scaled_error(oi, c[3], c[4]) <= TOL_FINAL[dt]
            # the results pass through the staging's output slots
            esize = 4 if dt == "f32" else 2
            off = (count * M * K * esize + 255) // 256 * 256 // 4
            slots = staging[off:off + count * M * N].cpu().numpy()
            assert np.array_equal(slots.view(np.uint32), got[:count * M * N].view(np.uint32))


def test_host_batch_back_to_back_shared_staging(lib):
    """Two batches on one stream share one staging with no synchronisation
    between them; the second waits for the first's copies out, and both
    results are right.  One weight serves every operation of a batch."""
    sk = lib
    M, N, K, S, kps, dt, count = 96, 512, 2048, 4, 512, "bf16", 6
    c1 = [oracle_case(M, N, K, S, kps, dt, "uniform", 20 + i) for i in range(count)]
    B = device_operand(c1[0][0].B, dt)
    want = []
    for c in c1:
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_bt(device_operand(c[0].A, dt), B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
        want.append(o.numpy())
    sb = sk.gemm_bt_host_staging_bytes(count, M, N, K, S, kps, dt)
    staging = torch.zeros(sb // 4, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    a1 = host_operand([c[0].A for c in c1], dt, True)
    a2 = host_operand([c[0].A for c in reversed(c1)], dt, True)
    o1 = torch.zeros(count * M * N, dtype=torch.float32).pin_memory()
    o2 = torch.zeros(count * M * N, dtype=torch.float32).pin_memory()
    stream = torch.cuda.Stream()
    ptrs = sk.pointer_array([B] * count)
    sk.gemm_bt_host_batch(a1, ptrs, o1, count, staging, sb, M, N, K, S, kps, dt, fused=1, stream=stream)
    sk.gemm_bt_host_batch(a2, ptrs, o2, count, staging, sb, M, N, K, S, kps, dt, fused=1, stream=stream)
    stream.synchronize()
    assert sk.splitk_get_device_status(stream) == 0
    for i in range(count):
        r1 = o1.numpy()[i * M * N:(i + 1) * M * N]
        r2 = o2.numpy()[(count - 1 - i) * M * N:(count - i) * M * N]
        assert np.array_equal(r1.view(np.uint32), want[i].view(np.uint32)), i
        assert np.array_equal(r2.view(np.uint32), want[i].view(np.uint32)), i


@pytest.mark.parametrize("case", [(96, 512, 512, "bf16", 1), (96, 512, 512, "bf16", 0), (64, 128, 160, "f16", 1),
                                  (32, 512, 2048, "bf16", 1), (32, 64, 128, "f32", 0)],
                         ids=lambda c: f"{c[3]}-M{c[0]}N{c[1]}K{c[2]}-fused{c[4]}")
def test_autotune_splits(lib, case):
    """The measured split choice is the fastest candidate it timed, a legal
    geometry; `out` then holds a correct result, and a later gemm_bt with the
    chosen split on the same workspace gives it again."""
    sk = lib
    M, N, K, dt, fused = case
    cand = {}
    for n in (1, 2, 4, 8, 16):
        kps = -(-(-(-K // n)) // 32) * 32
        cand[n] = (-(-K // kps), kps)
    nbytes = max(sk.gemm_bt_workspace_bytes(M, N, K, S, kps) for S, kps in cand.values())
    ops, _, _, Or, SO = oracle_case(M, N, K, cand[1][0], cand[1][1], dt)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    ws = Guarded(nbytes // 4, 0.0)
    out = Guarded(M * N)
    S, kps, us = sk.splitk_autotune_splits(A, B, out.data, ws.data, nbytes, M, N, K, dt, fused=fused, reps=10)
    torch.cuda.synchronize()
    assert (S, kps) in cand.values()
    timed = {c: t for c, t in us.items() if t is not None}
    assert timed and all(t > 0 for t in timed.values())
    assert min(timed.values()) == timed[min(timed, key=timed.get)]
    assert cand[min(timed, key=timed.get)] == (S, kps)
    seen = set()
    for n in (1, 2, 4, 8, 16):   # a repeated split count is timed once
        assert (us[n] is None) == (cand[n][0] in seen)
        seen.add(cand[n][0])
    assert out.guards_intact() and ws.guards_intact()
    got = out.numpy().reshape(M, N)
    assert max_scaled_error(got, Or, SO) <= TOL_FINAL[dt]
    again = Guarded(M * N)
    sk.gemm_bt(A, B, again.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
    assert sk.splitk_get_device_status() == 0
    assert np.array_equal(again.numpy().view(np.uint32), out.numpy().view(np.uint32))


KN_CASES = WORKLOADS + [(64, 128, 160, 3, 64, "bf16"), (96, 512, 512, 4, 128, "f16"), (32, 512, 2048, 16, 128, "bf16"),
                        (64, 128, 160, 3, 64, "f32"), (96, 512, 2048, 4, 512, "f32")]


def kn_weight(orc, ops):
    """W = B^T (the [K,N] weight whose prepared form is B), by the oracle's transpose."""
    return device_operand(orc.transpose(ops.B.reshape(ops.N, ops.K)), ops.dtype)


@pytest.mark.parametrize("case", KN_CASES, ids=ids(KN_CASES))
def test_kn_layout_matches_oracle(lib, orc, case):
    """gemm_splitk_kn / gemm_kn with W = B^T: partials and output against the
    oracle, guards intact, and the fused and two-kernel calls bitwise equal."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A, W = device_operand(ops.A, dt), kn_weight(orc, ops)
    P = Guarded(S * M * N)
    out = Guarded(M * N)
    sk.gemm_splitk_kn(A, W, P.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(P.data, out.data, S, M, N)
    assert sk.splitk_get_device_status() == 0
    assert P.guards_intact() and out.guards_intact()
    assert max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL
    assert max_scaled_error(out.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt]
    for fused in (0, 1, 3):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_kn(A, W, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
        assert sk.splitk_get_device_status() == 0
        assert o.guards_intact() and ws.guards_intact()
        assert np.array_equal(o.numpy().view(np.uint32), out.numpy().view(np.uint32)), f"fused={fused}"


@pytest.mark.parametrize("case", KN_CASES, ids=ids(KN_CASES))
def test_kn_layout_bitwise_equals_prepared(lib, orc, case):
    """16-bit operands: reading the weight N-contiguous gives the same bits as
    reading its prepared transpose K-contiguous (same products, same
    accumulation).  F32: the [K,N] weight runs exact FMA, the prepared one
    3xTF32; they agree to 3xTF32 accuracy (1e-5 of sum |a*b|, against the
    exact oracle's 1e-4 bound)."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, _, _ = oracle_case(M, N, K, S, kps, dt)
    A, B, W = device_operand(ops.A, dt), device_operand(ops.B, dt), kn_weight(orc, ops)
    P1, P2 = Guarded(S * M * N), Guarded(S * M * N)
    sk.gemm_splitk_bt(A, B, P1.data, M, N, K, S, kps, dt)
    sk.gemm_splitk_kn(A, W, P2.data, M, N, K, S, kps, dt)
    assert sk.splitk_get_device_status() == 0
    if dt != "f32":
        assert np.array_equal(P1.numpy().view(np.uint32), P2.numpy().view(np.uint32))
    else:
        diff = max_scaled_error(P1.numpy().reshape(S, M, N), P2.numpy().reshape(S, M, N).astype(np.float64), SP)
        assert diff <= 1e-5
        assert max_scaled_error(P2.numpy().reshape(S, M, N), Pr, SP) <= 1e-6   # exact FMA


@pytest.mark.parametrize("case", [(64, 128, 160, 3, 64, "bf16"), (256, 1024, 2048, 2, 1024, "bf16")],
                         ids=ids([(64, 128, 160, 3, 64, "bf16"), (256, 1024, 2048, 2, 1024, "bf16")]))
def test_kn_every_tiling(lib, orc, case):
    """Every tile width (one, two or four 64-column boxes of W per stage),
    chunk count and stage depth reads W correctly."""
    sk = lib
    M, N, K, S, kps, dt = case
    ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
    A, W = device_operand(ops.A, dt), kn_weight(orc, ops)
    seen = set()
    try:
        for bn, ch, kb in TILINGS:
            sk.splitk_set_tile_override(bn, ch, kb)
            d = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=0)
            key = (d["bn"], d["chunks"], d["kblocks_per_stage"])
            if key in seen:
                continue
            seen.add(key)
            P = Guarded(S * M * N)
            sk.gemm_splitk_kn(A, W, P.data, M, N, K, S, kps, dt)
            assert sk.splitk_get_device_status() == 0
            assert P.guards_intact()
            assert max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL, key
    finally:
        sk.splitk_set_tile_override(0, 0, 0)
    assert len(seen) > 4


BATCH_CASES = [(256, 1024, 2048, 2, 1024, "bf16", 1, 13), (96, 512, 2048, 4, 512, "f16", 1, 3),
               (32, 512, 2048, 1, 2048, "f32", 1, 2), (256, 1024, 2048, 2, 1024, "bf16", 0, 4),
               (160, 192, 320, 3, 128, "bf16", 1, 5)]


@pytest.mark.parametrize("case", BATCH_CASES, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}-f{c[6]}x{c[7]}"
                                                    for c in BATCH_CASES])
def test_batch_matches_single_calls(lib, case):
    """gemm_bt_batch: every output bitwise the gemm_bt result for its
    operands (one weight repeated for half the operations), guards intact;
    fused 16-bit calls whose plan groups run up to 8 to a launch."""
    sk = lib
    M, N, K, S, kps, dt, fused, count = case
    cs = [oracle_case(M, N, K, S, kps, dt, "uniform", 100 + i) for i in range(count)]
    As = [device_operand(c[0].A, dt) for c in cs]
    Bs = [device_operand(c[0].B, dt) for c in cs]
    Bs = [Bs[i] if i % 2 == 0 else Bs[0] for i in range(count)]   # repeated weights
    ws, nbytes = workspace(M, N, K, S, kps)
    refs = []
    for A, B in zip(As, Bs):
        o = Guarded(M * N)
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
        refs.append(o.numpy().copy())
    outs = [Guarded(M * N) for _ in range(count)]
    sk.gemm_bt_batch(As, Bs, [o.data for o in outs], count, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    assert sk.splitk_get_device_status() == 0
    plan = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)
    if fused and dt != "f32" and plan["fused_in_kernel"] and plan["compact"]:
        assert sk.splitk_last_launch()["group"] == (count - 1) % 8 + 1
    for o, r in zip(outs, refs):
        assert np.array_equal(o.numpy().view(np.uint32), r.view(np.uint32))
        assert o.guards_intact()


@pytest.mark.parametrize("nstreams,opc", [(1, 1), (2, 0), (2, 4)])
def test_host_batch_alternating_staging_in_flight(lib, nstreams, opc):
    """Six batches over two alternating staging buffers, on one stream or two
    alternating streams, no synchronisation until the end: each batch's copy
    in waits only for the previous batch on the same staging, and every
    result is right (with ops_per_copy 0 and 4 the operations of a copy
    group run as one launch)."""
    sk = lib
    M, N, K, S, kps, dt, count, rounds = 128, 256, 1024, 2, 512, "bf16", 4, 6
    cs = [oracle_case(M, N, K, S, kps, dt, "uniform", 40 + i) for i in range(count)]
    Bs = [device_operand(c[0].B, dt) for c in cs]
    want = []
    for c, B in zip(cs, Bs):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_bt(device_operand(c[0].A, dt), B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
        want.append(o.numpy())
    sb = sk.gemm_bt_host_staging_bytes(count, M, N, K, S, kps, dt)
    stagings = [torch.zeros(sb // 4, dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    ptrs = sk.pointer_array(Bs)
    order = [list(range(count)) if r % 2 == 0 else list(reversed(range(count))) for r in range(rounds)]
    hosts = [host_operand([cs[i][0].A for i in o], dt, True) for o in order]
    outs = [torch.zeros(count * M * N, dtype=torch.float32).pin_memory() for _ in range(rounds)]
    streams = [torch.cuda.Stream() for _ in range(nstreams)]
    for r in range(rounds):
        bp = sk.pointer_array([Bs[i] for i in order[r]])
        sk.gemm_bt_host_batch(hosts[r], bp, outs[r], count, stagings[r % 2], sb, M, N, K, S, kps, dt,
                              fused=1, ops_per_copy=opc, stream=streams[r % nstreams])
        if opc == 4:
            assert sk.splitk_last_launch()["group"] == 4
    for st in streams:
        st.synchronize()
    assert sk.splitk_get_device_status(streams[0]) == 0
    for r in range(rounds):
        got = outs[r].numpy()
        for j, i in enumerate(order[r]):
            assert np.array_equal(got[j * M * N:(j + 1) * M * N].view(np.uint32), want[i].view(np.uint32)), (r, j)
    del ptrs
