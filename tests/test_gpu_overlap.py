"""GPU tests of launches that start beside the launch before them inside a
CUDA graph capture ("overlap"; include/splitk.h, top comment).

The library may let a launch load before the previous grid ends only where no
launch that can still be running writes what the new one reads (overlap 1);
it also stores before that grid ends only where none of them reads or
writes what the new one writes (overlap 2), and every launch still waits for
the previous grid before it finishes.  A fused launch that overlaps may give
each thread block two consecutive chunks of its split (chunks_per_block 2),
or where the splits are full, after the first call, every chunk of every
split (no cluster), with the same sums; consecutive calls of one shape may
join one launch (group).  Each test captures a sequence of calls, checks
which launches overlapped (splitk_last_launch, read right after each call),
replays the graph several times and compares every output bitwise with the
same calls made eagerly, where each launch waits for the one before it.  The
eager results themselves are pinned to the F64 oracle by test_gpu_parity.py;
the headline case is checked against the oracle here too.
"""
import numpy as np
import pytest

from harness import TOL_FINAL, TOL_PARTIAL, device_operand, max_scaled_error, oracle_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    sk.splitk_set_tile_override(0, 0, 0)
    sk.splitk_set_overlap(1)   # overlap, one launch per call (grouping: its own tests below)
    yield sk
    sk.splitk_set_overlap(2)


def operands(M, N, K, dt, seed):
    import splitk_inputs as gen

    ops = gen.uniform(M, N, K, dt, seed)
    return device_operand(ops.A, dt), device_operand(ops.B, dt)


def capture(body):
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    return g


def bitwise(a, b) -> bool:
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def instances(sk, M, N, K, S, kps, dt, n, seed0=0):
    out = []
    for i in range(n):
        A, B = operands(M, N, K, dt, seed0 + i)
        nb = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
        ws = torch.zeros(nb // 4, dtype=torch.float32, device="cuda")
        out.append(dict(A=A, B=B, ws=ws, nb=nb, out=torch.full((M, N), 7.0, device="cuda"),
                        ref=torch.full((M, N), 7.0, device="cuda")))
    return out


@pytest.mark.parametrize("shape", [
    (256, 1024, 2048, 2, 1024),   # the headline
    (96, 512, 2048, 4, 512),      # a cluster of 8 CTAs
    (256, 512, 2048, 4, 512),
    (32, 64, 128, 2, 64),         # the single tile
    (160, 192, 320, 3, 128),      # M tail, three splits (two kernels)
    (256, 1024, 1920, 2, 1024),   # the last split's second chunk short
    (256, 1024, 1536, 2, 1024),   # ... and empty
])
@pytest.mark.parametrize("fused", [0, 1, 3])
def test_independent_calls_overlap_bitwise(lib, shape, fused):
    sk = lib
    M, N, K, S, kps = shape
    dt = "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 6)
    for it in insts:   # eager: every launch waits for the one before
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    refs_ws = [it["ws"].clone() for it in insts]
    in_kernel = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)["fused_in_kernel"]
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert all(d["capturing"] == 1 for d in seen)
    assert seen[0]["overlap"] == 0                       # nothing of ours precedes it
    # fused in one launch: each call reads only its own A and B, which no
    # earlier call writes, and writes only its own output and workspace.
    # Two kernels: each call's partial pass follows the previous call's
    # reduce, whose output it neither reads nor writes.
    assert all(d["overlap"] == 2 for d in seen[1:]), seen
    if in_kernel and N == 1024:
        assert all(d["compact"] == 1 for d in seen), seen
        # every compact launch takes both chunks of its split (512 each,
        # 64-column tiles) into one block: a cluster of the splits only
        assert all(d["chunks_per_block"] == 2 and d["cluster"] == S for d in seen), seen
    for _ in range(3):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    if fused != 1:   # the kept partials too (fused=0: the workspace holds them)
        for it, w in zip(insts, refs_ws):
            P = S * M * N
            assert bitwise(it["ws"][:P], w[:P])
    assert sk.splitk_get_device_status() == 0
    if (M, N, K, S) == (256, 1024, 2048, 2):
        ops, Pr, SP, Or, SO = oracle_case(M, N, K, S, kps, dt)
        assert max_scaled_error(insts[0]["out"].cpu().numpy(), Or, SO) <= TOL_FINAL[dt]


def test_dependent_chain_waits(lib):
    """F32 operands, so that an output can be the next call's A.  Expected:
    a: X -> Y          head (no call of ours before it): waits
    b: P -> Q          independent of a: overlaps, stores early
    c: Y -> Z          reads Y, which a (still in b's window) writes: waits
    d: Z -> W          reads what c writes: waits
    e: R -> T          independent of d: overlaps, stores early
    f: (U, Q) -> V     reads Q, written by b before the wait in c: overlaps
    g: W -> Y2         reads W, written by d (in the window d, e, f): waits"""
    sk = lib
    dt = "f32"
    M, K = 128, 256
    S, kps = 2, 128

    def mat(rows, cols, seed):
        g = torch.Generator(device="cpu").manual_seed(seed)
        return (torch.rand(rows, cols, generator=g) * 2 - 1).cuda()

    X, P, R, U = mat(M, K, 1), mat(M, K, 2), mat(M, K, 3), mat(M, K, 4)
    Bs = {k: mat(256, K, 10 + i) for i, k in enumerate("abcdeg")}
    nb = sk.gemm_bt_workspace_bytes(M, 256, K, S, kps)
    ws = {k: torch.zeros(nb // 4, device="cuda") for k in "abcdefg"}
    outs = {k: torch.full((M, 256), 7.0, device="cuda") for k in "abcdeg"}
    outs["f"] = torch.full((M, 128), 7.0, device="cuda")
    Y, Q, Z, W, T, V, Y2 = outs["a"], outs["b"], outs["c"], outs["d"], outs["e"], outs["f"], outs["g"]
    calls = [
        ("a", X, Bs["a"], Y, 256), ("b", P, Bs["b"], Q, 256), ("c", Y, Bs["c"], Z, 256),
        ("d", Z, Bs["d"], W, 256), ("e", R, Bs["e"], T, 256), ("f", U, Q, V, 128), ("g", W, Bs["g"], Y2, 256),
    ]

    def run(record=None):
        for name, A, B, O, N in calls:
            sk.gemm_bt(A, B, O, ws[name], nb, M, N, K, S, kps, dt, fused=1)
            if record is not None:
                record.append((name, sk.splitk_last_launch()["overlap"]))

    run()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in outs.items()}
    seen = []
    g = capture(lambda: run(seen))
    assert seen == [("a", 0), ("b", 2), ("c", 0), ("d", 0), ("e", 2), ("f", 2), ("g", 0)], seen
    for _ in range(3):
        for v in outs.values():
            v.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for k in outs:
            assert bitwise(outs[k], ref[k]), k
    assert sk.splitk_get_device_status() == 0


def test_store_waits_for_previous_reader(lib):
    """b overlaps a (it reads neither Y nor anything a writes), but b's output
    is a's input X: b may load early, yet must not store before a has read X
    (overlap 1, not 2).  The graph is replayed from the same starting X each
    time."""
    sk = lib
    dt = "f32"
    M, N, K, S, kps = 128, 256, 256, 2, 128
    g0 = torch.Generator(device="cpu").manual_seed(5)
    X0 = (torch.rand(M, K, generator=g0) * 2 - 1).cuda()
    B1 = (torch.rand(N, K, generator=g0) * 2 - 1).cuda()
    A2 = (torch.rand(M, K, generator=g0) * 2 - 1).cuda()
    B2 = (torch.rand(N, K, generator=g0) * 2 - 1).cuda()
    X = X0.clone()
    Y = torch.empty(M, N, device="cuda")
    nb = sk.gemm_bt_workspace_bytes(M, N, K, S, kps)
    w1 = torch.zeros(nb // 4, device="cuda")
    w2 = torch.zeros(nb // 4, device="cuda")
    seen = []

    def run(record=None):
        sk.gemm_bt(X, B1, Y, w1, nb, M, N, K, S, kps, dt, fused=1)
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])
        sk.gemm_bt(A2, B2, X, w2, nb, M, N, K, S, kps, dt, fused=1)   # overwrites a's input
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])

    run()
    torch.cuda.synchronize()
    Y_ref, X_ref = Y.clone(), X.clone()
    g = capture(lambda: run(seen))
    assert seen == [0, 1]
    for _ in range(5):
        X.copy_(X0)
        Y.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert bitwise(Y, Y_ref) and bitwise(X, X_ref)
    assert sk.splitk_get_device_status() == 0


def test_other_work_between_calls_waits(lib):
    """A copy captured between two calls writes the second call's A: the second
    call follows that node, not the library's launch, so it waits; the call
    after it overlaps again."""
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 3)
    src = operands(M, N, K, dt, 99)[0]
    seen = []

    def run(record=None):
        it0, it1, it2 = insts
        sk.gemm_bt(it0["A"], it0["B"], it0["out"], it0["ws"], it0["nb"], M, N, K, S, kps, dt, fused=1)
        it1["A"].copy_(src)
        sk.gemm_bt(it1["A"], it1["B"], it1["out"], it1["ws"], it1["nb"], M, N, K, S, kps, dt, fused=1)
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])
        sk.gemm_bt(it2["A"], it2["B"], it2["out"], it2["ws"], it2["nb"], M, N, K, S, kps, dt, fused=1)
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])

    g = capture(lambda: run(seen))
    assert seen == [0, 2]
    for rep in range(3):
        src.copy_(operands(M, N, K, dt, 100 + rep)[0])
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        got = [it["out"].clone() for it in insts]
        run()   # eagerly, from the same state
        torch.cuda.synchronize()
        for a, it in zip(got, insts):
            assert bitwise(a, it["out"])
    assert sk.splitk_get_device_status() == 0


def test_overlap_switch(lib):
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 4)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            seen.append(sk.splitk_last_launch())

    try:
        sk.splitk_set_overlap(False)
        g = capture(body)
    finally:
        sk.splitk_set_overlap(1)
    assert all(d["overlap"] == 0 and d["compact"] == 0 and d["capturing"] == 0 for d in seen)
    g.replay()
    torch.cuda.synchronize()
    for it in insts:
        assert bitwise(it["out"], it["ref"])


def test_kn_layout_overlap_bitwise(lib):
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 4)
    for it in insts:
        it["W"] = it["B"].t().contiguous()
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_kn(it["A"], it["W"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            seen.append(sk.splitk_last_launch()["overlap"])

    g = capture(body)
    assert seen == [0, 2, 2, 2]
    g.replay()
    torch.cuda.synchronize()
    for it in insts:
        assert bitwise(it["out"], it["ref"])   # the [K,N] path is bitwise the [N,K] path
    assert sk.splitk_get_device_status() == 0


def test_reduce_heads_or_extends_runs(lib):
    """A reduce after foreign work waits for it and only then lets the next
    launch start, so it heads a run: the fused call after it overlaps, and so
    does the partial pass after that.  The reduces that follow (of partials
    no running launch writes) load at once and let their successors start
    early.  Every result is the eager one, bit for bit."""
    sk = lib
    M, N, K, S, kps, dt = 96, 512, 2048, 4, 512, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 4)
    # partials to reduce: from eager partial passes
    Ps = []
    for it in insts:
        P = torch.empty(S * M * N, device="cuda")
        sk.gemm_splitk_bt(it["A"], it["B"], P, M, N, K, S, kps, dt)
        Ps.append(P)
    outs_ref = [torch.empty(M, N, device="cuda") for _ in range(4)]
    outs = [torch.full((M, N), 7.0, device="cuda") for _ in range(4)]
    fused_ref = torch.empty(M, N, device="cuda")
    fused_out = torch.full((M, N), 7.0, device="cuda")
    side = torch.zeros(16, device="cuda")
    Pfresh = torch.empty(S * M * N, device="cuda")

    def run(o, fo, record=None):
        side.add_(1.0)                                          # foreign work first
        sk.splitk_reduce(Ps[0], o[0], S, M, N)                  # heads a run
        it = insts[1]
        sk.gemm_bt(it["A"], it["B"], fo, it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])
        sk.gemm_splitk_bt(insts[2]["A"], insts[2]["B"], Pfresh, M, N, K, S, kps, dt)   # overlaps the fused call
        if record is not None:
            record.append(sk.splitk_last_launch()["overlap"])
        for j in (1, 2, 3):                                     # partials nothing running writes
            sk.splitk_reduce(Ps[j], o[j], S, M, N)

    run(outs_ref, fused_ref)
    torch.cuda.synchronize()
    seen = []
    g = capture(lambda: run(outs, fused_out, seen))
    assert seen == [2, 2], seen
    for _ in range(3):
        for o in outs:
            o.fill_(7.0)
        fused_out.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, outs_ref):
            assert bitwise(a, b)
        assert bitwise(fused_out, fused_ref)
    assert sk.splitk_get_device_status() == 0


def test_store_waits_for_previous_writer(lib):
    """b writes the output a writes (its own operands are independent): b may
    load early but stores only after a has finished (overlap 1), so the
    output holds b's result, as eagerly."""
    sk = lib
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 2)
    O = torch.full((M, N), 7.0, device="cuda")
    seen = []

    def run(record=None):
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], O, it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            if record is not None:
                record.append(sk.splitk_last_launch()["overlap"])

    run()
    torch.cuda.synchronize()
    ref = O.clone()
    g = capture(lambda: run(seen))
    assert seen == [0, 1]
    for _ in range(5):
        O.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert bitwise(O, ref)
    assert sk.splitk_get_device_status() == 0


def test_long_run_starts_a_new_window(lib):
    """40 independent calls in one capture: the library follows at most 32
    launches of a run, so the 33rd waits for the previous grid and heads a
    new run, and the calls after it overlap again; every output is the eager
    one, bit for bit."""
    sk = lib
    M, N, K, S, kps, dt = 256, 512, 2048, 4, 512, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 40)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            seen.append(sk.splitk_last_launch()["overlap"])

    g = capture(body)
    assert seen[0] == 0 and seen[32] == 0, seen
    assert all(v == 2 for i, v in enumerate(seen) if i not in (0, 32)), seen
    for _ in range(2):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    assert sk.splitk_get_device_status() == 0


@pytest.mark.parametrize("shape", [(96, 512, 512, 4, 128), (256, 1024, 2048, 2, 1024), (160, 192, 320, 3, 128)])
@pytest.mark.parametrize("fused", [0, 1])
def test_f32_calls_overlap_bitwise(lib, shape, fused):
    """F32 operands (3xTF32) in graphs: the calls after the first overlap and
    take the compact layout (two CTAs per SM, a pair of chunks per CTA where
    a split has two or more), and every output is the eager one, bit for
    bit."""
    sk = lib
    M, N, K, S, kps = shape
    dt = "f32"
    insts = instances(sk, M, N, K, S, kps, dt, 5)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert seen[0]["overlap"] == 0 and all(d["overlap"] == 2 for d in seen[1:]), seen
    plan = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)
    cpc = 2 if plan["fused_in_kernel"] and plan["chunks"] % 2 == 0 else 1
    assert plan["compact_chunks_per_block"] == cpc, plan
    assert all(d["chunks_per_block"] == cpc for d in seen), seen
    if M * N <= 256 * 1024:
        assert all(d["compact"] == 1 for d in seen), seen
    for _ in range(2):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    assert sk.splitk_get_device_status() == 0


# ---- grouping: consecutive independent calls of one shape in one launch

@pytest.fixture
def grouping(lib):
    lib.splitk_set_overlap(2)
    yield lib
    lib.splitk_set_overlap(1)


@pytest.mark.parametrize("shape", [
    (256, 1024, 2048, 2, 1024),   # the headline: both chunks of a split per block, clusters of 2
    (96, 512, 2048, 4, 512),      # clusters of 4
    (256, 512, 2048, 4, 512),     # one chunk per split
    (256, 1024, 1536, 2, 1024),   # an empty last chunk
    (32, 512, 2048, 1, 2048),     # clusters of 8 (8 chunks)
    (96, 512, 512, 2, 256),       # clusters of 8 (2 splits x 4 chunks)
])
@pytest.mark.parametrize("fused", [1, 3])
def test_grouped_calls_bitwise(grouping, shape, fused):
    """12 independent calls of one shape: the first launches (heading the
    run), the next 7 join its launch, the 9th launches again and the last 3
    join that one.  Every output (and kept partials) is the eager one, bit
    for bit."""
    sk = grouping
    M, N, K, S, kps = shape
    dt = "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 12)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    refs_ws = [it["ws"].clone() for it in insts]
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert [d["group"] for d in seen] == [1, 2, 3, 4, 5, 6, 7, 8, 1, 2, 3, 4], seen
    assert seen[0]["overlap"] == 0 and seen[8]["overlap"] == 2, seen
    for _ in range(3):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    if fused == 3:
        for it, w in zip(insts, refs_ws):
            P = S * M * N
            assert bitwise(it["ws"][:P], w[:P])
    assert sk.splitk_get_device_status() == 0


def test_grouping_only_same_shape_and_independent(grouping):
    """Calls of two shapes in turn never group; a call that reads the output
    of the call before it does not join it (it waits), and the independent
    call after it joins that one."""
    sk = grouping
    dt = "bf16"
    s1, s2 = (256, 1024, 2048, 2, 1024), (256, 512, 2048, 4, 512)
    a = instances(sk, *s1, dt, 3)
    b = instances(sk, *s2, dt, 3)
    seen = []

    def alternate(record=None):
        for x, y in zip(a, b):
            sk.gemm_bt(x["A"], x["B"], x["out"], x["ws"], x["nb"], *s1, dt, fused=1)
            if record is not None:
                record.append(sk.splitk_last_launch()["group"])
            sk.gemm_bt(y["A"], y["B"], y["out"], y["ws"], y["nb"], *s2, dt, fused=1)
            if record is not None:
                record.append(sk.splitk_last_launch()["group"])

    g = capture(lambda: alternate(seen))
    assert seen == [1] * 6, seen
    for x, y in zip(a, b):
        x["out"].fill_(7.0)
        y["out"].fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    got = [t["out"].clone() for t in a + b]
    alternate()
    torch.cuda.synchronize()
    assert all(bitwise(u, t["out"]) for u, t in zip(got, a + b))

    # a call writing what the call before it writes does not join it (it
    # stores only after that launch has finished); the call after it, touching
    # nothing in flight, joins it
    c = instances(sk, *s1, dt, 3)
    O = torch.empty(s1[0], s1[1], device="cuda")
    rec = []

    def waw(record=None):
        for k, it in enumerate(c):
            o = O if k < 2 else it["out"]
            sk.gemm_bt(it["A"], it["B"], o, it["ws"], it["nb"], *s1, dt, fused=1)
            if record is not None:
                d = sk.splitk_last_launch()
                record.append((d["overlap"], d["group"]))

    waw()
    torch.cuda.synchronize()
    ref_o, ref_c = O.clone(), c[2]["out"].clone()
    g2 = capture(lambda: waw(rec))
    assert rec == [(0, 1), (1, 1), (1, 2)], rec
    O.fill_(7.0)
    c[2]["out"].fill_(7.0)
    g2.replay()
    torch.cuda.synchronize()
    assert bitwise(O, ref_o) and bitwise(c[2]["out"], ref_c)
    assert sk.splitk_get_device_status() == 0


def test_grouped_kn_bitwise(grouping):
    """The [K,N] weight groups the same way, bitwise the [N,K] path."""
    sk = grouping
    M, N, K, S, kps, dt = 256, 1024, 2048, 2, 1024, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 8)
    for it in insts:
        it["W"] = it["B"].t().contiguous()
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_kn(it["A"], it["W"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            seen.append(sk.splitk_last_launch()["group"])

    g = capture(body)
    assert seen == list(range(1, 9)), seen
    g.replay()
    torch.cuda.synchronize()
    for it in insts:
        assert bitwise(it["out"], it["ref"])
    assert sk.splitk_get_device_status() == 0


@pytest.mark.parametrize("shape", [
    (128, 2048, 4096, 4, 1024),   # 16 whole-K blocks a call, one chunk per split
    (512, 1024, 4096, 2, 2048),   # 32 a call, two chunks per split
    (224, 2048, 4096, 4, 1024),   # an M tail: the second row tile has 96 live rows
    (96, 4096, 4096, 2, 2048),    # M below one tile
])
@pytest.mark.parametrize("fused", [1, 3])
def test_whole_k_calls_bitwise(grouping, shape, fused):
    """Full splits whose compact plan takes more than half the SMs: the first
    call of the capture launches with the compact plan (a cluster of the
    splits); the calls after it take whole-K blocks (every chunk of every
    split in one block, no cluster), and the second converts the first's
    launch to that plan and joins it.  Every output, and the partials a call
    keeps, is the eager one, bit for bit."""
    sk = grouping
    M, N, K, S, kps = shape
    dt = "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 12)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    refs_ws = [it["ws"].clone() for it in insts]
    C = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)["chunks"]
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert seen[0]["chunks_per_block"] <= C and seen[0]["cluster"] > 1, seen[0]
    assert all(d["chunks_per_block"] == S * C and d["cluster"] == 1 and d["bn"] == 128 for d in seen[1:]), seen
    assert [d["group"] for d in seen] == [1, 2, 3, 4, 5, 6, 7, 8, 1, 2, 3, 4], seen
    for _ in range(3):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    if fused == 3:
        for it, w in zip(insts, refs_ws):
            P = S * M * N
            assert bitwise(it["ws"][:P], w[:P])
    assert sk.splitk_get_device_status() == 0


@pytest.mark.parametrize("shape", [
    (96, 512, 512, 4, 128),       # clusters of 4
    (256, 1024, 2048, 2, 1024),   # the headline shape with F32 operands
    (32, 512, 2048, 1, 2048),     # one split, eight chunks
])
@pytest.mark.parametrize("fused", [1, 3])
def test_grouped_f32_calls_bitwise(grouping, shape, fused):
    """F32 operands (3xTF32) group the same way: 12 independent calls, the
    first launching with its usual plan, the second converting that launch
    to the compact plan and joining it, up to 8 per launch.  Every output
    (and kept partials) is the eager one, bit for bit."""
    sk = grouping
    M, N, K, S, kps = shape
    dt = "f32"
    if not sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)["fused_in_kernel"]:
        pytest.skip("this shape runs the two kernels")
    insts = instances(sk, M, N, K, S, kps, dt, 12)
    for it in insts:
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    refs_ws = [it["ws"].clone() for it in insts]
    seen = []

    def body():
        for it in insts:
            sk.gemm_bt(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert [d["group"] for d in seen] == [1, 2, 3, 4, 5, 6, 7, 8, 1, 2, 3, 4], seen
    assert all(d["compact"] == 1 for d in seen[1:]), seen
    for _ in range(2):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for it in insts:
            assert bitwise(it["out"], it["ref"])
    if fused == 3:
        for it, w in zip(insts, refs_ws):
            P = S * M * N
            assert bitwise(it["ws"][:P], w[:P])
    assert sk.splitk_get_device_status() == 0


def test_whole_k_kn_bitwise(grouping):
    """Whole-K blocks reading the [K,N] weight (MN-major operand), with an M
    tail: bitwise the [N,K] path's eager results."""
    sk = grouping
    M, N, K, S, kps, dt = 352, 1024, 4096, 2, 2048, "bf16"
    insts = instances(sk, M, N, K, S, kps, dt, 8)
    for it in insts:
        it["W"] = it["B"].t().contiguous()
        sk.gemm_bt(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
    torch.cuda.synchronize()
    seen = []

    def body():
        for it in insts:
            sk.gemm_kn(it["A"], it["W"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=1)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    C = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=1)["chunks"]
    assert all(d["chunks_per_block"] == S * C and d["cluster"] == 1 for d in seen[1:]), seen
    assert [d["group"] for d in seen] == list(range(1, 9)), seen
    g.replay()
    torch.cuda.synchronize()
    for it in insts:
        assert bitwise(it["out"], it["ref"])
    assert sk.splitk_get_device_status() == 0


def random_graph_cases(n, seed=77):
    """Seeded shapes for graphs of independent calls: full splits (K = S * kps,
    where whole-K blocks may apply) and short last splits, 1 to 8 splits, all
    three element types, both weight layouts for 16-bit operands."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    while len(cases) < n:
        M = 32 * int(rng.integers(1, 17))          # 32 .. 512
        N = 64 * int(rng.integers(1, 33))          # 64 .. 2048
        S = int(rng.choice([1, 2, 3, 4, 8]))
        kps = 64 * int(rng.integers(1, 33))        # 64 .. 2048
        short = 32 * int(rng.integers(0, kps // 32)) if rng.integers(0, 2) else 0
        K = S * kps - short
        if (S - 1) * kps >= K:
            continue
        dt = ("bf16", "f16", "f32")[int(rng.integers(0, 3))]
        kn = dt != "f32" and bool(rng.integers(0, 2))
        fused = (1, 3)[int(rng.integers(0, 2))]
        cases.append((M, N, K, S, kps, dt, kn, fused))
    return cases


GRAPH_CASES = random_graph_cases(16) + [
    (224, 2048, 4096, 4, 1024, "bf16", True, 3),   # whole-K blocks: [K,N] weight, kept partials, M tail
    (512, 1024, 4096, 2, 2048, "f16", False, 1),
    (96, 4096, 4096, 2, 2048, "bf16", True, 1),
    (352, 1024, 4096, 2, 2048, "f16", True, 3),
]


@pytest.mark.parametrize("case", GRAPH_CASES,
                         ids=[f"{c[5]}{'-kn' if c[6] else ''}-M{c[0]}N{c[1]}K{c[2]}S{c[3]}-f{c[7]}" for c in GRAPH_CASES])
def test_random_graphs_bitwise(grouping, orc, case):
    """Six independent calls of a random shape captured into one graph
    (grouping on: joined launches, merged chunks, whole-K blocks and the
    conversion of a run's first launch wherever the planner takes them):
    every output, and the partials kept with fused=3, bitwise the same calls
    made eagerly, and the first call's at 300 seeded points within the
    pages' tolerances of the oracle."""
    import splitk_inputs as gen

    sk = grouping
    M, N, K, S, kps, dt, kn, fused = case
    insts = instances(sk, M, N, K, S, kps, dt, 6, seed0=M + N + K)
    call = sk.gemm_kn if kn else sk.gemm_bt
    for it in insts:
        if kn:
            it["B"] = it["B"].t().contiguous()   # the [K,N] weight itself
        call(it["A"], it["B"], it["ref"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
    torch.cuda.synchronize()
    refs_ws = [it["ws"].clone() for it in insts]
    seen = []

    def body():
        for it in insts:
            call(it["A"], it["B"], it["out"], it["ws"], it["nb"], M, N, K, S, kps, dt, fused=fused)
            seen.append(sk.splitk_last_launch())

    g = capture(body)
    assert all(d["capturing"] == 1 for d in seen), seen
    for _ in range(2):
        for it in insts:
            it["out"].fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for i, it in enumerate(insts):
            assert bitwise(it["out"], it["ref"]), (i, seen[i])
    if fused == 3:
        for it, w in zip(insts, refs_ws):
            assert bitwise(it["ws"][:S * M * N], w[:S * M * N])
    assert sk.splitk_get_device_status() == 0
    # the first call against the oracle at seeded points (split -1: the output)
    ops = gen.uniform(M, N, K, dt, seed=M + N + K)
    rng = np.random.Generator(np.random.PCG64(K))
    npts = 300
    sp = rng.integers(-1, S if fused == 3 else 0, npts)
    m, n = rng.integers(0, M, npts), rng.integers(0, N, npts)
    sp[:4] = -1
    m[:4], n[:4] = [0, M - 1, 0, M - 1], [0, 0, N - 1, N - 1]   # the zero first row, the x4 last row
    val, bound = orc.points(ops.A, ops.B, dt, kps, S, sp, m, n)
    got = insts[0]["out"].cpu().numpy()[m, n]
    if fused == 3:
        P0 = insts[0]["ws"][:S * M * N].view(S, M, N).cpu().numpy()
        got = np.where(sp >= 0, P0[np.maximum(sp, 0), m, n], got)
    part = sp >= 0
    assert max_scaled_error(got[~part], val[~part], bound[~part]) <= TOL_FINAL[dt]
    if part.any():
        assert max_scaled_error(got[part], val[part], bound[part]) <= TOL_PARTIAL
