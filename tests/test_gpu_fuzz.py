"""GPU parity on seeded random legal geometries, and on large shapes checked at
sampled points.

The random cases draw M, N, K, the split length and the element type from the
contract's legal space (M, K and k_per_split multiples of 32, N of 64,
splits = ceil(K / k_per_split)), so that the tile planner meets shapes no
hand-picked list holds: odd chunk counts, clusters that cannot hold every
split, a short final split, chunks past its end.  Each is compared with the
full oracle within the pages' tolerances, with guards, and the fused calls
must give the two-kernel output bit for bit.

The large shapes are too big for the full oracle in a test; the oracle's
per-point evaluation checks partials and outputs at sampled (split, row,
column) points, the rest of the output is checked for finiteness and the
fused result against the two-kernel one.
"""
import numpy as np
import pytest

from harness import TOL_FINAL, TOL_PARTIAL, Guarded, device_operand, max_scaled_error, workspace

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    sk.splitk_set_tile_override(0, 0, 0)
    return sk


def random_cases(n, seed=2024):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    while len(cases) < n:
        M = 32 * int(rng.integers(1, 21))          # 32 .. 640
        N = 64 * int(rng.integers(1, 25))          # 64 .. 1536
        K = 32 * int(rng.integers(1, 97))          # 32 .. 3072
        kps = 32 * int(rng.integers(1, K // 32 + 1))
        S = -(-K // kps)
        dt = ("bf16", "f16", "f32")[int(rng.integers(0, 3))]
        cases.append((M, N, K, S, kps, dt))
    return cases


RANDOM = random_cases(24)


@pytest.mark.parametrize("case", RANDOM, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}kps{c[4]}" for c in RANDOM])
def test_random_geometry(lib, orc, case):
    import splitk_inputs as gen

    sk = lib
    M, N, K, S, kps, dt = case
    assert orc.contract(M, N, K, S, kps) == 0
    ops = gen.uniform(M, N, K, dt, seed=M + N + K)
    Pr, SP = orc.partials(ops.A, ops.B, dt, K, S, kps)
    Or, SO = orc.output(ops.A, ops.B, dt)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    P, out = Guarded(S * M * N), Guarded(M * N)
    sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(P.data, out.data, S, M, N)
    assert sk.splitk_get_device_status() == 0
    assert P.guards_intact() and out.guards_intact()
    assert max_scaled_error(P.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL
    assert max_scaled_error(out.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt]
    for fused in (1, 3):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
        assert sk.splitk_get_device_status() == 0
        assert o.guards_intact() and ws.guards_intact()
        assert np.array_equal(o.numpy().view(np.uint32), out.numpy().view(np.uint32)), fused


LARGE = [(2048, 4096, 8192, 4, 2048, "bf16"), (1056, 2112, 5120, 5, 1024, "f16"),
         (4096, 8192, 4096, 1, 4096, "bf16"), (1024, 2048, 8192, 2, 4096, "f32"),
         (2048, 8192, 8192, 2, 4096, "bf16"), (2048, 4096, 4096, 1, 4096, "f32"),
         # 256-row tiles whose last tile is ragged: the second half empty (M = 3872),
         # or partly below M (M = 4000)
         (3872, 8192, 2048, 1, 2048, "bf16"), (4000, 8192, 2048, 1, 2048, "f16")]


def check_sampled(orc, ops, dt, M, N, S, kps, P, out, npts=600):
    """Partials and outputs at seeded (split, row, column) points against the
    oracle's per-point evaluation, the first eight on the zero first row, the
    scaled last row and the corners."""
    rng = np.random.Generator(np.random.PCG64(M + ops.A.shape[1]))
    s = rng.integers(-1, S, npts)
    m = rng.integers(0, M, npts)
    n = rng.integers(0, N, npts)
    m[:8] = [0, 0, M - 1, M - 1, 0, M - 1, M // 2, 1]     # the zero first row and the x4 last row
    n[:8] = [0, N - 1, 0, N - 1, N // 2, N // 2, 0, N - 1]
    val, bound = orc.points(ops.A, ops.B, dt, kps, S, s, m, n)
    Pn = P.view(S, M, N)
    On = out.view(M, N)
    idx_s = torch.from_numpy(np.maximum(s, 0)).cuda()
    idx_m = torch.from_numpy(m).cuda()
    idx_n = torch.from_numpy(n).cuda()
    got_p = Pn[idx_s, idx_m, idx_n].cpu().numpy()
    got_o = On[idx_m, idx_n].cpu().numpy()
    got = np.where(s >= 0, got_p, got_o)
    part = s >= 0
    assert max_scaled_error(got[part], val[part], bound[part]) <= TOL_PARTIAL
    assert max_scaled_error(got[~part], val[~part], bound[~part]) <= TOL_FINAL[dt]


@pytest.mark.parametrize("case", LARGE, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}" for c in LARGE])
def test_large_shape_sampled(lib, orc, case):
    import splitk_inputs as gen

    sk = lib
    M, N, K, S, kps, dt = case
    ops = gen.uniform(M, N, K, dt, seed=7)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    P = Guarded(S * M * N)
    out = Guarded(M * N)
    sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(P.data, out.data, S, M, N)
    ws, nbytes = workspace(M, N, K, S, kps)
    fused = torch.empty(M * N, dtype=torch.float32, device="cuda")
    sk.gemm_bt(A, B, fused, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
    assert sk.splitk_get_device_status() == 0
    assert P.guards_intact() and out.guards_intact() and ws.guards_intact()
    assert torch.equal(fused.view(torch.int32), out.data.view(torch.int32))
    del fused
    kept = torch.empty(M * N, dtype=torch.float32, device="cuda")
    sk.gemm_bt(A, B, kept, ws.data, nbytes, M, N, K, S, kps, dt, fused=3)   # the partials kept too
    assert sk.splitk_get_device_status() == 0 and ws.guards_intact()
    assert torch.equal(kept.view(torch.int32), out.data.view(torch.int32))
    assert torch.equal(ws.data[: S * M * N].view(torch.int32), P.data.view(torch.int32))
    del kept
    assert bool(torch.isfinite(out.data).all()) and bool(torch.isfinite(P.data).all())
    check_sampled(orc, ops, dt, M, N, S, kps, P.data, out.data)


ROW_FIRST_KN = [(4096, 8192, 4096, 1, 4096, "bf16"), (2048, 4096, 4096, 1, 4096, "f32")]


@pytest.mark.parametrize("case", ROW_FIRST_KN, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}" for c in ROW_FIRST_KN])
def test_large_kn_row_first(lib, orc, case):
    """The [K,N] weight on large shapes that the planner puts in the row-first
    tile order: 16-bit operands give the [N,K] path's partials and outputs bit
    for bit, F32 the oracle's values at sampled points; the fused call gives
    the two-kernel output bit for bit."""
    import splitk_inputs as gen

    sk = lib
    M, N, K, S, kps, dt = case
    assert sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=0)["rows_first"] == 1
    ops = gen.uniform(M, N, K, dt, seed=5)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    W = B.t().contiguous()
    Pk, outk = Guarded(S * M * N), Guarded(M * N)
    sk.gemm_splitk_kn(A, W, Pk.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(Pk.data, outk.data, S, M, N)
    ws, nbytes = workspace(M, N, K, S, kps)
    fused = Guarded(M * N)
    sk.gemm_kn(A, W, fused.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=1)
    assert sk.splitk_get_device_status() == 0
    assert Pk.guards_intact() and outk.guards_intact() and fused.guards_intact() and ws.guards_intact()
    assert torch.equal(fused.data.view(torch.int32), outk.data.view(torch.int32))
    if dt != "f32":
        del W
        P, out = Guarded(S * M * N), Guarded(M * N)
        sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
        sk.splitk_reduce(P.data, out.data, S, M, N)
        assert torch.equal(Pk.data.view(torch.int32), P.data.view(torch.int32))
        assert torch.equal(outk.data.view(torch.int32), out.data.view(torch.int32))
    check_sampled(orc, ops, dt, M, N, S, kps, Pk.data, outk.data)


GROUPINGS = [(1, 1), (2, 1), (1, 2), (4, 1), (2, 2), (1, 4), (8, 1), (4, 2), (2, 4), (1, 8)]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("grouping", GROUPINGS, ids=[f"S{s}C{c}" for s, c in GROUPINGS])
def test_cluster_split_sum_groupings(lib, orc, grouping, dt):
    """Every (splits, chunks) grouping that one cluster sums on chip (splits x
    chunks a power of two up to 8), with the partials discarded (fused=1) or
    kept (fused=3): the output and kept partials equal the two-kernel path's
    bit for bit, and the output is within the pages' tolerance of the oracle."""
    import splitk_inputs as gen

    sk = lib
    S, C = grouping
    M, N = 96, 128
    kps = C * 64
    K = S * kps
    ops = gen.uniform(M, N, K, dt, seed=S * 16 + C)
    Or, SO = orc.output(ops.A, ops.B, dt)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    try:
        sk.splitk_set_tile_override(64, C, 0)
        plan = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=1)
        assert plan["chunks"] == C and plan["cluster"] == S * C and plan["split_sum"] == 2, plan
        P, out = Guarded(S * M * N), Guarded(M * N)
        sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
        sk.splitk_reduce(P.data, out.data, S, M, N)
        ref_bits = out.numpy().view(np.uint32)
        assert max_scaled_error(out.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt]
        for fused in (1, 3):
            ws, nbytes = workspace(M, N, K, S, kps)
            o = Guarded(M * N)
            sk.gemm_bt(A, B, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=fused)
            assert sk.splitk_get_device_status() == 0
            assert o.guards_intact() and ws.guards_intact()
            assert np.array_equal(o.numpy().view(np.uint32), ref_bits), fused
            if fused == 3:
                kept = ws.numpy()[:S * M * N].view(np.uint32)
                assert np.array_equal(kept, P.numpy().view(np.uint32))
    finally:
        sk.splitk_set_tile_override(0, 0, 0)


@pytest.mark.parametrize("case", RANDOM, ids=[f"{c[5]}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}kps{c[4]}" for c in RANDOM])
def test_random_geometry_kn_and_prepare(lib, orc, case):
    """The same random geometries with the weight in its [K,N] layout: weight
    preparation gives the exact transpose; the [K,N] path gives the [N,K]
    path's partials and outputs bit for bit with 16-bit operands (the same
    products in the same order), and F32 (exact FMA there, 3xTF32 here)
    within the pages' tolerances of the oracle."""
    import splitk_inputs as gen

    sk = lib
    M, N, K, S, kps, dt = case
    ops = gen.uniform(M, N, K, dt, seed=M + N + K)
    A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
    W = B.t().contiguous()
    B2 = torch.full_like(B, 0)
    sk.splitk_prepare_bt(W, B2, K, N, dt)
    torch.cuda.synchronize()
    assert torch.equal(B2.view(torch.int16 if dt != "f32" else torch.int32),
                       B.view(torch.int16 if dt != "f32" else torch.int32))
    P, out = Guarded(S * M * N), Guarded(M * N)
    sk.gemm_splitk_bt(A, B, P.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(P.data, out.data, S, M, N)
    Pk, outk = Guarded(S * M * N), Guarded(M * N)
    sk.gemm_splitk_kn(A, W, Pk.data, M, N, K, S, kps, dt)
    sk.splitk_reduce(Pk.data, outk.data, S, M, N)
    fused = []
    for f in (1, 3):
        ws, nbytes = workspace(M, N, K, S, kps)
        o = Guarded(M * N)
        sk.gemm_kn(A, W, o.data, ws.data, nbytes, M, N, K, S, kps, dt, fused=f)
        fused.append((o, ws))
    assert sk.splitk_get_device_status() == 0
    assert all(g.guards_intact() for g in (P, out, Pk, outk)) and all(o.guards_intact() and w.guards_intact() for o, w in fused)
    if dt != "f32":
        assert np.array_equal(Pk.numpy().view(np.uint32), P.numpy().view(np.uint32))
        assert np.array_equal(outk.numpy().view(np.uint32), out.numpy().view(np.uint32))
    else:
        Pr, SP = orc.partials(ops.A, ops.B, dt, K, S, kps)
        Or, SO = orc.output(ops.A, ops.B, dt)
        assert max_scaled_error(Pk.numpy().reshape(S, M, N), Pr, SP) <= TOL_PARTIAL
        assert max_scaled_error(outk.numpy().reshape(M, N), Or, SO) <= TOL_FINAL[dt]
    for o, _ in fused:   # the fused [K,N] call adds the [K,N] partials in the reduce kernel's order
        assert np.array_equal(o.numpy().view(np.uint32), outk.numpy().view(np.uint32))


def test_concurrent_host_threads(lib):
    """Four host threads, each on its own stream, call gemm_bt (fused and not)
    on different shapes and element types at the same time (ctypes releases
    the GIL); every result equals the single-threaded one bit for bit."""
    import threading

    import splitk_inputs as gen

    sk = lib
    cases = [(256, 1024, 2048, 2, 1024, "bf16"), (96, 512, 2048, 4, 512, "f16"),
             (160, 192, 320, 3, 128, "bf16"), (64, 256, 1024, 2, 512, "f32")]
    prepared = []
    for M, N, K, S, kps, dt in cases:
        ops = gen.uniform(M, N, K, dt, seed=M + K)
        A, B = device_operand(ops.A, dt), device_operand(ops.B, dt)
        ws, nbytes = workspace(M, N, K, S, kps)
        ref = torch.empty(M * N, dtype=torch.float32, device="cuda")
        sk.gemm_bt(A, B, ref, ws.data, nbytes, M, N, K, S, kps, dt, fused=0)
        torch.cuda.synchronize()
        prepared.append((M, N, K, S, kps, dt, A, B, ref))
    errors = []

    def worker(idx):
        try:
            M, N, K, S, kps, dt, A, B, ref = prepared[idx]
            stream = torch.cuda.Stream()
            ws, nbytes = workspace(M, N, K, S, kps)
            outs = [torch.empty(M * N, dtype=torch.float32, device="cuda") for _ in range(2)]
            torch.cuda.synchronize()   # the workspace's set-up ran on torch's default stream
            for it in range(20):
                sk.gemm_bt(A, B, outs[it & 1], ws.data, nbytes, M, N, K, S, kps, dt, fused=it % 2, stream=stream)
            stream.synchronize()
            for o in outs:
                if not torch.equal(o.view(torch.int32), ref.view(torch.int32)):
                    errors.append((idx, "result differs"))
        except Exception as e:   # reported below, in the main thread
            errors.append((idx, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(prepared))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert sk.splitk_get_device_status() == 0
