"""Host-side geometry of every tile plan the library makes (no GPU needed).

The tensor-core kernel trusts the plan that `splitk_describe_launch` reports:
which K range each CTA loads, how its shared memory is laid out, which
pieces of the output tile each cluster rank owns and where the peers'
contributions land.  This test restates that index arithmetic on the CPU and
checks, for hand-picked shapes, the seeded random geometries of the GPU
tests, and every tile override:

- the chunks of each split load every k of the split exactly once, each TMA
  box starting on a 16-byte boundary and inside K;
- the shared-memory size is the stage ring (or the accumulator staging, if
  larger), one receive slot per peer and the alignment slack, within the
  per-block limit;
- the grid covers every tile once, with the row tiles along x exactly when
  the launch is more than one wave, B's slab is over 32 MB and A's is the
  smaller; 256-row tiles only where the planner's rule allows them, and
  then with the whole shared memory of a block;
- a rank's share of the tile is a whole number of 32 x 32 boxes (each warp
  pushes whole boxes), every 16-byte piece has exactly one owner, and every
  contribution sent to or read from a receive slot stays inside that slot;
- the compact layout (taken inside graph captures, by fused calls and by
  the partial pass of the two-kernel call): the same tiles, chunks and sums, a ring that still covers every k once, the receive slots inside
  the ring after the staging area, and two or three thread blocks' shared
  and tensor memory within one SM's; where a block takes two consecutive
  chunks of its split (chunks_per_block 2), each chunk starts on a stage
  boundary, its accumulators fit the block's share of tensor memory, and
  the cluster holds half as many blocks; where a block takes all of K
  (whole-K), its chunks cover K once in order and it is alone on its SM.
"""
import itertools

import pytest

from test_gpu_fuzz import LARGE, RANDOM

SMEM_LIMIT = 226 * 1024
TMEM256_SMEM = 100 * 1024     # a 256-column block's shared memory, at least (the tensor-memory rule)
COMPACT_LIMIT = 112 * 1024
COMPACT3_LIMIT = 74 * 1024    # three thread blocks to an SM
SM_SMEM = 228 * 1024          # per SM; 1 KB of it reserved per thread block
STATIC_SMEM = 240             # the kernel's barriers and flags (nvcc -Xptxas -v)
TILE_M = 128
RESIDENT_CLUSTERS = {1: 148, 2: 72, 4: 36, 8: 15}   # clusters of 1-8 CTAs a GB300 keeps resident


@pytest.fixture(scope="module")
def lib():
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    return sk


def tmem_fits(cols, smem):
    """The tensor-memory rule of the planner: one column per 512 bytes of
    shared memory, 256 columns from 100 KB on, or all 512 for a block that
    takes the whole per-block limit (alone on its SM)."""
    return cols * 512 <= smem or (cols == 256 and smem >= TMEM256_SMEM) or (cols == 512 and smem >= SMEM_LIMIT)


def test_tmem_rule_never_oversubscribes():
    """Whatever mix of these kernels' blocks fits on an SM by shared memory
    (228 KB, 1 KB reserved per block and the static part), their tensor-
    memory columns fit in its 512.  Each plan's shared memory is at least its
    accumulator staging area, 512 bytes per 128-row column: 32 KB for 64
    columns, 64 KB for 128; the smallest footprint for each column count
    that the rule allows is enumerated, and every multiset of them that fits
    is checked."""
    import functools

    per_sm = SM_SMEM
    # 256-row tiles and whole-K blocks take all of a block's shared memory
    kinds = [(512, SMEM_LIMIT + 1024 + STATIC_SMEM)]
    for cols in (64, 128, 256):
        smem = min(s for s in range(1024, SMEM_LIMIT + 1, 1024) if tmem_fits(cols, s) and s >= cols * 256)
        kinds.append((cols, smem + 1024 + STATIC_SMEM))

    @functools.lru_cache(maxsize=None)
    def most(room, start):
        best = 0
        for i in range(start, len(kinds)):
            cols, foot = kinds[i]
            if foot <= room:
                best = max(best, cols + most(room - foot, i))
        return best

    assert most(per_sm, 0) <= 512, kinds


def piece(g):
    """Staging offset, tile row and tile column of 16-byte piece g (the
    kernel's layout: 32 x 32 float boxes, 128-byte rows, 16-byte pieces
    swizzled by the row)."""
    b, rb, j = g >> 8, (g >> 3) & 31, g & 7
    return ((g >> 3) << 7) | ((j ^ (rb & 7)) << 4), (b & 3) * 32 + rb, (b >> 2) * 32 + j * 4


def check_plan(sk, M, N, K, S, kps, fused, dt, bn=0, ch=0, kbs=0):
    sk.splitk_set_tile_override(bn, ch, kbs)
    try:
        d = sk.splitk_describe_launch(M, N, K, S, kps, dt, fused=fused)
    finally:
        sk.splitk_set_tile_override(0, 0, 0)
    x3 = dt == "f32"
    kb_elems, elem = (32, 4) if x3 else (64, 2)
    BN, C, CL, stages = d["bn"], d["chunks"], d["chunk_len"], d["stages"]
    Q, KBS, T3, SS, TM = d["cluster"], d["kblocks_per_stage"], d["three_d"], d["split_sum"], d["tile_m"]
    assert d["path"] == (2 if x3 else 0)
    assert C in (1, 2, 4, 8) and Q in (1, 2, 4, 8) and 1 <= stages <= 8 and 1 <= KBS <= 4
    assert Q == C or (SS == 2 and Q == S * C)
    mt = -(-M // TILE_M)
    # 256-row tiles: BN 256, one CTA per tile keeping or summing its own
    # partials, 16-bit operands, and fewer waves of 148 CTAs even at 1.36x
    # the time per tile
    assert TM in (TILE_M, 2 * TILE_M)
    per_row_tile = (N // BN) * S
    waves1 = -(-mt * per_row_tile // 148)
    waves2 = -(-(-(-mt // 2)) * per_row_tile // 148)
    wins = not x3 and BN == 256 and Q == 1 and SS != 1 and mt > 1 and waves1 > 1 and waves2 * 1.36 < waves1
    if TM == 2 * TILE_M:
        assert wins
    elif not kbs:
        assert not wins
    tiles_xy = (-(-M // TM), N // BN) if d["rows_first"] else (N // BN, -(-M // TM))
    assert (d["grid_x"], d["grid_y"], d["grid_z"]) == (*tiles_xy, S * C)
    assert d["grid_y"] <= 65535
    # row tiles first only for launches of more than one wave whose B slab
    # (one split of B) outgrows a quarter of L2, with A's slab the smaller
    waves = -(-M // TM) * (N // BN) * S * C // Q > RESIDENT_CLUSTERS[Q]
    b_slab = N * kps * (4 if x3 else 2)
    assert d["rows_first"] == int(waves and mt * TILE_M < N and b_slab > 32 << 20 and N // BN <= 65535)
    assert N % BN == 0 and d["grid_z"] % Q == 0
    if T3:
        assert K % kb_elems == 0 and kps % kb_elems == 0 and CL % kb_elems == 0
    else:
        assert KBS == 1

    # shared memory: the ring (or the accumulator staging) + receive slots + slack
    pieces = 32 * BN
    share = -(-(-(-pieces // Q)) // 8) * 8
    stage_bytes = (TM + BN) * 128 * KBS * (2 if x3 else 1)
    epi_bytes = TILE_M * BN * 4
    region0 = -(-max(stages * stage_bytes, epi_bytes) // 1024) * 1024
    if TM == TILE_M:
        assert d["smem_bytes"] == region0 + (Q - 1) * share * 16 + 1024 <= SMEM_LIMIT
    else:   # the whole per-block limit: no other CTA shares the SM's tensor memory
        assert region0 + 1024 <= d["smem_bytes"] == SMEM_LIMIT

    # 256-row tiles: each k-block of A is 256 rows of 128 bytes; the second
    # accumulator's MMAs read rows 128-255 (16 KB in, 1 KB-aligned for the
    # swizzle), inside that k-block; the two accumulators (BN columns each)
    # fill the 512 tensor-memory columns; each half is staged in turn through
    # the same 128 x BN staging area
    if TM == 2 * TILE_M:
        a_kblock = TM * 128
        assert BN == 256 and Q == 1 and not x3 and SS != 1
        assert 16384 % 1024 == 0 and 16384 + TILE_M * 128 <= a_kblock
        assert 2 * BN <= 512
        assert epi_bytes <= region0 and stages * (a_kblock + BN * 128) * KBS <= region0

    check_k_coverage(K, S, kps, C, CL, KBS, T3, kb_elems, elem)
    check_exchange(BN, Q, region0, d["smem_bytes"] - 1024)

    # the compact layout: same tiles and sums, a ring two blocks to an SM,
    # the receive slots inside it after the staging area
    # whole K in a block (a call that follows another): full splits that the
    # chunks tile, every chunk of every split in its own 128-column
    # accumulator (at most 512 columns), no cluster, one block per SM with
    # all of its shared memory; taken where the compact plan would take more
    # than half the SMs, or there is none
    can3d = K % kb_elems == 0 and kps % kb_elems == 0
    whole = not x3 and SS == 2 and S > 1 and can3d and CL % 64 == 0 and K == S * kps and kps == C * CL
    wcols = 128 * S * C
    wctas = -(-M // TM) * (N // 128)
    nkb = -(-CL // kb_elems)
    kfix = kbs and min(kbs, 4)                            # an overridden stage depth
    ring_ok = not kfix or (nkb % kfix == 0 and
                           min(2, -(-nkb * S * C // kfix)) * (TM + 128) * 128 * kfix + 1024 <= SMEM_LIMIT)
    whole_fits = whole and TM == TILE_M and BN <= 128 and N % 128 == 0 and wcols <= 512 and wctas <= 148 and ring_ok
    if d["compact"] and d["compact_chunks_per_block"] > C:
        cst, ckbs, csmem = d["compact_stages"], d["compact_kblocks_per_stage"], d["compact_smem_bytes"]
        cpc, qc, CB = d["compact_chunks_per_block"], d["compact_cluster"], d["compact_bn"]
        assert whole_fits and CB == 128 and cpc == S * C and qc == 1 and d["compact_grid_z"] == 1
        assert wcols & (wcols - 1) == 0
        assert nkb % ckbs == 0 and cst >= min(2, -(-nkb * cpc // ckbs))
        assert csmem == SMEM_LIMIT and tmem_fits(wcols, csmem)
        assert cst * (TM + 128) * 128 * ckbs + 1024 <= SMEM_LIMIT and TILE_M * 128 * 4 + 1024 <= SMEM_LIMIT
        assert SMEM_LIMIT + 1024 + STATIC_SMEM + 1024 + 1024 > SM_SMEM   # nothing else fits beside it
        # one block covers all of K: the splits' chunks back to back, each
        # in its own accumulator, the first k-block of each starting a stage
        check_k_coverage(K, 1, K, S * C, CL, ckbs, int(ckbs > 1), kb_elems, elem, S * C)
        return
    if whole_fits:   # not taken: the compact plan keeps to half the SMs
        assert d["compact"], (M, N, K, S, kps, BN, C)
        assert -(-M // TM) * (N // d["compact_bn"]) * d["compact_grid_z"] <= 74, (M, N, K, S, kps, BN, C)

    if d["compact"]:
        assert TM == TILE_M and BN <= 128
        cst, ckbs, csmem = d["compact_stages"], d["compact_kblocks_per_stage"], d["compact_smem_bytes"]
        cpc, qc, CB = d["compact_chunks_per_block"], d["compact_cluster"], d["compact_bn"]
        assert 1 <= cst <= 8 and 1 <= ckbs <= 4 and (ckbs == 1 or T3 or (K % kb_elems == 0 and kps % kb_elems == 0))
        # two consecutive chunks of a split in one block: only where the
        # chunks are whole stages of whole k-blocks, from 64-column tiles
        # (widened to 128 or not)
        mergeable = SS == 2 and C > 1 and can3d and CL % kb_elems == 0
        assert CB == BN or (CB == 128 and BN == 64 and cpc == 2 and mergeable), (BN, CB, cpc)
        assert cpc in (1, 2) and (cpc == 1 or (mergeable and BN == 64 and C % 2 == 0))
        assert qc == Q // cpc and d["compact_grid_z"] == S * C // cpc and d["compact_grid_z"] % qc == 0
        assert N % CB == 0
        cctas = -(-M // TM) * (N // CB) * S * C // cpc
        assert cctas // qc <= RESIDENT_CLUSTERS[qc]       # one wave
        cstage = (TM + CB) * 128 * ckbs * (2 if x3 else 1)
        nkb = -(-CL // kb_elems)
        cnkb = nkb * cpc                                  # k-blocks of a block
        assert cst >= min(2, -(-cnkb // ckbs))            # double-buffered unless one stage holds them all
        if cpc > 1:
            assert nkb % ckbs == 0                        # a chunk's first k-block starts a stage
        cpieces = 32 * CB
        cshare = -(-(-(-cpieces // qc)) // 8) * 8
        cepi = TILE_M * CB * 4
        recv_bytes = (qc - 1) * cshare * 16
        cols = CB * cpc                                   # tensor memory: a power of two >= 32
        floor = cols * 512 if cols <= 128 else TMEM256_SMEM
        cregion = -(-max(cst * cstage, cepi + recv_bytes, floor) // 1024) * 1024
        assert csmem == cregion + 1024 <= COMPACT_LIMIT
        assert 2 * (csmem + STATIC_SMEM + 1024) <= SM_SMEM   # two blocks to an SM
        assert cols & (cols - 1) == 0 and 2 * cols <= 512 and tmem_fits(cols, csmem)
        # three to an SM for merged launches and for launches of more CTAs
        # than half the SMs, with clusters of at most 4 and at most 128
        # columns, wherever a double-buffered ring of single k-block stages
        # and the staging plus receive slots fit in 74 KB
        kmin = kbs if (kbs and T3) else 1                    # the smallest stage the override allows
        stage1 = (TM + CB) * 128 * kmin * (2 if x3 else 1)
        fits3 = max(min(2, -(-cnkb // kmin)) * stage1, cepi + recv_bytes, floor) + 1024 <= COMPACT3_LIMIT
        if qc <= 4 and cols <= 128 and (cctas > 74 or cpc > 1) and fits3:
            assert csmem <= COMPACT3_LIMIT and 3 * (csmem + STATIC_SMEM + 1024) <= SM_SMEM and 3 * cols <= 512
        check_k_coverage(K, S, kps, C, CL, ckbs, int(ckbs > 1), kb_elems, elem, cpc)
        if qc > 1:
            check_exchange(CB, qc, cepi, cregion)
    else:
        assert d["compact_stages"] == d["compact_kblocks_per_stage"] == d["compact_smem_bytes"] == 0
        assert d["compact_chunks_per_block"] == d["compact_cluster"] == d["compact_grid_z"] == 0


def check_k_coverage(K, S, kps, C, CL, KBS, T3, kb_elems, elem, cpc=1):
    """Every k of every split loaded exactly once, boxes aligned; with cpc
    chunks per block, each chunk's k-blocks in their own accumulator, in
    order, the first of each chunk starting it."""
    for s in range(S):
        ks, ke = s * kps, min(s * kps + kps, K)
        covered = []
        for cb in range(C // cpc):                    # the blocks of the split
            lo = ks + cb * cpc * CL
            hi = min(lo + cpc * CL, ke)
            klen = max(0, hi - lo)
            nkb = -(-klen // kb_elems)
            if T3:
                assert lo % kb_elems == 0
            kpc = CL // kb_elems
            jc, kb_in = 0, 0                          # the kernel's accumulator bookkeeping
            for i in range(-(-nkb // KBS)):
                if T3:
                    assert lo // kb_elems + i * KBS < K // kb_elems     # the box starts inside K
                if cpc > 1:
                    assert jc == (i * KBS) // kpc and kb_in == (i * KBS) % kpc
                    kb_in += KBS
                    if kb_in == kpc:
                        kb_in, jc = 0, jc + 1
                for j in range(KBS):
                    kb = i * KBS + j
                    if kb >= nkb:
                        break
                    kx = lo + kb * kb_elems
                    valid = min(kb_elems, klen - kb * kb_elems)
                    assert valid in (32, 64) and (kx * elem) % 16 == 0 and kx < K
                    if cpc > 1:                       # inside the chunk its accumulator holds
                        assert lo + (kb // kpc) * CL <= kx < lo + (kb // kpc + 1) * CL
                    covered += range(kx, kx + valid)
        assert covered == list(range(ks, ke)), (s, ks, ke)


def check_exchange(BN, Q, recv, limit):
    """Ownership of the tile's pieces, and every push into and read of the
    receive slots (which start at `recv`) inside its slot and below `limit`."""
    pieces = 32 * BN
    share = -(-(-(-pieces // Q)) // 8) * 8
    epi_bytes = TILE_M * BN * 4
    if Q > 1:
        assert share % 256 == 0, "a rank's share must be whole 32 x 32 boxes"
    own = [(min(pieces, r * share), min(pieces, min(pieces, r * share) + share)) for r in range(Q)]
    owner = {}
    for r, (lo, hi) in enumerate(own):
        assert lo % 8 == 0 and hi % 8 == 0
        for g in range(lo, hi):
            off, row, col = piece(g)
            assert lo * 16 <= off < hi * 16 and off + 16 <= epi_bytes
            assert (row, col) not in owner
            owner[(row, col)] = r
    assert len(owner) == pieces
    for sender in range(Q):
        for b in range(pieces // 256):              # the box a warp stages and pushes
            r = (b * 256) // share
            if r == sender:
                continue
            assert own[r][0] <= b * 256 and b * 256 + 256 <= own[r][1]
            slot = sender - (1 if sender > r else 0)
            dst = recv + (slot * share + (b * 256 - r * share)) * 16
            assert recv + slot * share * 16 <= dst and dst + 4096 <= recv + (slot + 1) * share * 16
            assert dst + 4096 <= limit
    for me, (lo, hi) in enumerate(own):             # the owner's reads of its peers' slots
        for r in range(Q):
            if r == me:
                continue
            slot = r - (1 if r > me else 0)
            base = recv + slot * share * 16 - lo * 16
            for g in (lo, hi - 1) if hi > lo else ():
                addr = base + piece(g)[0]
                assert recv + slot * share * 16 <= addr and addr + 16 <= recv + (slot + 1) * share * 16


CASES = [(32, 64, 128, 2, 64), (96, 512, 2048, 4, 512), (256, 512, 2048, 4, 512), (256, 1024, 2048, 2, 1024),
         (64, 128, 160, 3, 64), (32, 64, 32, 1, 32), (160, 192, 320, 3, 128), (96, 320, 1024, 2, 512),
         (64, 128, 8192, 4, 2048), (512, 2048, 4096, 4, 1024), (288, 256, 96, 3, 32)]
CASES += [(32, 512, 2048, s, 2048 // s) for s in (1, 2, 4, 8, 16)] + [(96, 512, 512, s, 512 // s) for s in (1, 2, 4, 8, 16)]
# whole-K blocks where the compact plan is larger than half the SMs
CASES += [(128, 2048, 4096, 4, 1024), (512, 1024, 4096, 2, 2048), (256, 2048, 8192, 4, 2048)]
OVERRIDES = [(0, 0, 0)] + list(itertools.product((64, 128, 256), (1, 2, 4, 8), (0, 1, 2, 4)))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_plan_geometry_hand_picked(lib, dt):
    n = 0
    for case in CASES:
        for fused in (0, 1):
            for ov in OVERRIDES:
                check_plan(lib, *case, fused, dt, *ov)
                n += 1
    assert n == len(CASES) * 2 * len(OVERRIDES)


def test_plan_geometry_random_and_large(lib):
    for c in RANDOM + LARGE:
        for fused in (0, 1):
            for ov in OVERRIDES:
                check_plan(lib, *c[:5], fused, c[5], *ov)


@pytest.mark.parametrize("shape,whole", [
    ((256, 1024, 2048, 2, 1024), False),   # 32 compact blocks: keeps two launches on the SMs
    ((256, 512, 4096, 4, 1024), False),    # 64
    ((256, 1024, 4096, 2, 2048), False),   # 32
    ((128, 2048, 4096, 4, 1024), True),    # 128 compact blocks
    ((256, 2048, 8192, 4, 2048), True),
    ((512, 1024, 4096, 2, 2048), True),
    ((128, 4096, 4096, 2, 2048), True),
    ((128, 4096, 8192, 4, 2048), True),
    ((224, 2048, 4096, 4, 1024), True),    # an M tail
    ((96, 4096, 4096, 2, 2048), True),     # M below one tile
    ((256, 1024, 1536, 2, 1024), False),   # the last split short: not full splits
    ((96, 512, 2048, 4, 512), False),      # 2 chunks x 4 splits: 1024 columns
])
def test_whole_k_choice(lib, shape, whole):
    """Which fused BF16 calls that follow another in a capture get whole-K
    blocks (the shapes the choice was measured on), with the same chunks as
    the eager plan."""
    d = lib.splitk_describe_launch(*shape, "bf16", fused=1)
    M, N, K, S, kps = shape
    assert d["fused_in_kernel"] == 1 and d["compact"] == 1
    assert (d["compact_chunks_per_block"] == S * d["chunks"] and d["compact_cluster"] == 1) == whole, d
    if whole:
        assert d["compact_bn"] == 128 and d["compact_grid_z"] == 1


def test_plan_follows_override_changes(lib):
    """Plans are cached per host thread; a change of the tile override must
    still give the plan for the new override, and clearing it the default."""
    shape = (256, 1024, 2048, 2, 1024)
    default = lib.splitk_describe_launch(*shape, "bf16", fused=1)
    seen = []
    try:
        for ov in ((64, 4, 0), (64, 1, 0), (128, 2, 2), (64, 4, 0)):
            lib.splitk_set_tile_override(*ov)
            p = lib.splitk_describe_launch(*shape, "bf16", fused=1)
            assert p["bn"] == ov[0] and p["chunks"] == ov[1], (ov, p)
            if ov[2]:
                assert p["kblocks_per_stage"] == ov[2]
            seen.append(p)
    finally:
        lib.splitk_set_tile_override(0, 0, 0)
    assert seen[0] == seen[3]
    assert lib.splitk_describe_launch(*shape, "bf16", fused=1) == default
    # other dtypes and fused flags of the same shape are distinct entries
    assert lib.splitk_describe_launch(*shape, "f32", fused=1)["path"] == 2
    assert lib.splitk_describe_launch(*shape, "bf16", fused=0)["fused_in_kernel"] == 0
    assert default["fused_in_kernel"] == 1


def test_fused_routing(lib):
    """gemm_bt(fused=1) sums the splits in its launch only where one resident
    cluster holds all of a tile's splits and chunks; elsewhere it runs the two
    kernels (the same chunks, so the same result bit for bit), which measured
    faster on GB300 than summing through global memory; F32 operands follow
    the same rule."""
    sk = lib
    fused_in_kernel = [
        (256, 1024, 2048, 2, 1024, "bf16"), (256, 1024, 2048, 4, 512, "bf16"), (96, 512, 2048, 4, 512, "bf16"),
        (256, 512, 2048, 4, 512, "bf16"), (32, 64, 128, 2, 64, "bf16"), (32, 512, 2048, 8, 256, "f16"),
        (96, 512, 512, 2, 256, "f32"), (32, 512, 2048, 1, 2048, "f32"),
        (32, 512, 2048, 2, 1024, "f32"), (32, 512, 2048, 8, 256, "f32"), (96, 512, 512, 8, 64, "f32"),
    ]
    two_kernels = [
        (256, 1024, 2048, 8, 256, "bf16"), (256, 1024, 2048, 16, 128, "bf16"),   # more than one cluster holds
        (96, 512, 2048, 16, 128, "bf16"), (32, 512, 2048, 16, 128, "f16"),
        (64, 128, 160, 3, 64, "bf16"),                                          # three splits
        (4096, 8192, 4096, 2, 2048, "bf16"),                                    # more tiles than resident clusters
        (32, 512, 2048, 16, 128, "f32"),
    ]
    for c in fused_in_kernel:
        d = sk.splitk_describe_launch(*c, fused=1)
        assert d["fused_in_kernel"] == 1 and d["kernels_per_call"] == 1 and d["split_sum"] == 2, c
    for c in two_kernels:
        d = sk.splitk_describe_launch(*c, fused=1)
        assert d["fused_in_kernel"] == 0 and d["kernels_per_call"] == 2 and d["split_sum"] == 0, c
        # the partial pass of the fused call is the two-kernel call's partial pass
        d0 = sk.splitk_describe_launch(*c, fused=0)
        assert {k: d[k] for k in ("bn", "chunks", "chunk_len", "cluster", "stages")} == \
               {k: d0[k] for k in ("bn", "chunks", "chunk_len", "cluster", "stages")}, c
