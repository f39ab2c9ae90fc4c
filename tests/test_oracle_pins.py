"""Pins for the F64 oracle, each against something other than the oracle itself.

* decoders: every binary16/bfloat16 bit pattern against numpy/torch widening,
  plus textbook values of the formats;
* contract: the hand-written cases in tests/golden/pages_contract.json (taken
  from the pages' rules), and the property that a legal geometry's split
  ranges tile [0, K) with no empty split;
* partials/output: pure-Python brute force (exact integers; math.fsum for
  uniform values), numpy float64 matmul, closed forms (ones, identity B, unit A
  rows), and invariants (splits sum to the unsplit product, zero row is zero,
  the x4 row is four times the plain row);
* the pins have teeth: deliberately wrong oracles (planted here, on the CPU)
  fail at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import splitk_inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_contract():
    with open(os.path.join(GOLDEN, "pages_contract.json")) as f:
        return json.load(f)


# ------------------------------------------------------------------ decoders


def test_decode_f16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_all_patterns(orc):
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_textbook_values(orc):
    # binary16: 1.0, -2.0, smallest subnormal 2^-24, largest finite 65504, -inf
    f16 = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0xFC00, 0x0400], np.uint16)
    assert list(orc.decode(f16, "f16")) == [1.0, -2.0, 2.0**-24, 65504.0, -math.inf, 2.0**-14]
    # bfloat16: 1.0, -2.0, smallest subnormal 2^-133, largest finite, +inf, 0.5
    bf = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x7F80, 0x3F00], np.uint16)
    assert list(orc.decode(bf, "bf16")) == [1.0, -2.0, 2.0**-133,
                                            (2 - 2.0**-7) * 2.0**127, math.inf, 0.5]


def test_decode_f32_random_patterns(orc):
    rng = np.random.Generator(np.random.PCG64(5))
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    got = orc.decode(bits.view(np.float32), "f32")
    with np.errstate(invalid="ignore"):
        ref = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------------ contract


def test_contract_pages_cases(orc):
    for M, N, K, S, kps, expect in load_contract()["contract_cases"]["cases"]:
        assert orc.contract(M, N, K, S, kps) == expect, (M, N, K, S, kps)


def test_contract_matches_split_tiling(orc):
    """Legal split geometry <=> the ranges tile [0,K) and none is empty."""
    for K in range(32, 32 * 14, 32):
        for kps in range(32, 32 * 16, 32):
            for S in range(0, 20):
                ranges = [orc.split_range(K, kps, s) for s in range(S)]
                covered = []
                for k0, k1 in ranges:
                    covered.extend(range(k0, k1))
                tiles = covered == list(range(K)) and all(k1 > k0 for k0, k1 in ranges)
                legal = orc.contract(32, 64, K, S, kps) == 0
                assert legal == tiles, (K, kps, S)


def test_short_final_split_range(orc):
    # K=160 with kps=64: three splits, the last clamped to 32 elements
    assert [orc.split_range(160, 64, s) for s in range(3)] == [(0, 64), (64, 128), (128, 160)]


# --------------------------------------------------------- pin checks (reusable)


class RealOracle:
    def __init__(self, orc):
        self.o = orc

    def partials(self, ops, S, kps):
        return self.o.partials(ops.A, ops.B, ops.dtype, ops.K, S, kps)

    def output(self, ops):
        return self.o.output(ops.A, ops.B, ops.dtype)


def dec(orc, x, dtype):
    return orc.decode(x, dtype)


def pin_bruteforce_integers(impl, orc):
    """Exact integer arithmetic in pure Python, compared bitwise."""
    ops = gen.integers(32, 64, 96, "bf16", seed=3)
    a = dec(orc, ops.A, "bf16").astype(int).tolist()
    b = dec(orc, ops.B, "bf16").astype(int).tolist()
    S, kps = 3, 32
    P, SP = impl.partials(ops, S, kps)
    O, SO = impl.output(ops)
    for m in range(32):
        for n in range(64):
            row, col = a[m], b[n]
            full = 0
            fabs = 0
            for s in range(S):
                ps = sum(row[k] * col[k] for k in range(s * kps, (s + 1) * kps))
                pa = sum(abs(row[k] * col[k]) for k in range(s * kps, (s + 1) * kps))
                assert P[s, m, n] == ps and SP[s, m, n] == pa
                full += ps
                fabs += pa
            assert O[m, n] == full and SO[m, n] == fabs


def pin_fsum(impl, orc, dtype):
    """Products of two inputs are exact in F64; math.fsum rounds their sum once."""
    ops = gen.uniform(32, 64, 64, dtype, seed=11)
    a = dec(orc, ops.A, dtype)
    b = dec(orc, ops.B, dtype)
    O, SO = impl.output(ops)
    P, SP = impl.partials(ops, 2, 32)
    for m in range(0, 32, 3):
        for n in range(0, 64, 5):
            prods = a[m] * b[n]
            assert abs(O[m, n] - math.fsum(prods)) <= 1e-14 * SO[m, n] + 1e-300
            assert abs(SO[m, n] - math.fsum(np.abs(prods))) <= 1e-14 * SO[m, n] + 1e-300
            for s in range(2):
                ps = prods[32 * s:32 * (s + 1)]
                assert abs(P[s, m, n] - math.fsum(ps)) <= 1e-14 * SP[s, m, n] + 1e-300


def pin_numpy(impl, orc, dtype, M=96, N=128, K=160, S=3, kps=64):
    """numpy float64 matmul on the decoded values (a library routine)."""
    ops = gen.uniform(M, N, K, dtype, seed=2)
    a = dec(orc, ops.A, dtype)
    b = dec(orc, ops.B, dtype)
    O, SO = impl.output(ops)
    assert np.all(np.abs(O - a @ b.T) <= 1e-12 * SO)
    assert np.allclose(SO, np.abs(a) @ np.abs(b).T, rtol=1e-12, atol=0)
    P, SP = impl.partials(ops, S, kps)
    for s in range(S):
        k0, k1 = s * kps, min((s + 1) * kps, K)
        ref = a[:, k0:k1] @ b[:, k0:k1].T
        assert np.all(np.abs(P[s] - ref) <= 1e-12 * SP[s])


def pin_closed_forms(impl, orc):
    # all ones: P[s] = length of split s, O = K
    ops = gen.ones(32, 64, 160, "bf16")
    P, SP = impl.partials(ops, 3, 64)
    O, SO = impl.output(ops)
    for s, length in enumerate([64, 64, 32]):
        assert np.all(P[s] == length) and np.all(SP[s] == length)
    assert np.all(O == 160) and np.all(SO == 160)
    # B = [I | 0]: O = A[:, :N]  (checks the [N,K] layout of B)
    ops = gen.identity_b(64, 64, 128, "f16", seed=4)
    O, _ = impl.output(ops)
    assert np.array_equal(O, dec(orc, ops.A, "f16")[:, :64])
    # A rows = e_(m mod K): O[m, :] = B[:, m mod K]  (checks the M indexing)
    ops = gen.unit_rows_a(64, 128, 32, "bf16", seed=6)
    O, _ = impl.output(ops)
    b = dec(orc, ops.B, "bf16")
    for m in range(64):
        assert np.array_equal(O[m], b[:, m % 32])


def pin_invariants(impl, orc):
    ops = gen.uniform(64, 128, 160, "bf16", seed=8)
    P, SP = impl.partials(ops, 3, 64)
    O, SO = impl.output(ops)
    assert np.all(np.abs(P.sum(axis=0) - O) <= 1e-12 * SO)
    assert np.allclose(SP.sum(axis=0), SO, rtol=1e-12, atol=0)
    # zero first row of A gives exactly zero
    assert np.all(O[0] == 0) and np.all(P[:, 0] == 0) and np.all(SO[0] == 0)
    # the x4 last row is exactly four times the row drawn without the scale
    plain = gen.uniform(64, 128, 160, "bf16", seed=8, scale_last_row=False)
    O2, _ = impl.output(plain)
    assert np.array_equal(O[-1], 4.0 * O2[-1])
    assert np.array_equal(O[1:-1], O2[1:-1])
    # results do not depend on the split count
    for S, kps in [(1, 160), (2, 96), (5, 32)]:
        Ps, _ = impl.partials(ops, S, kps)
        assert np.all(np.abs(Ps.sum(axis=0) - O) <= 1e-12 * SO)
    assert np.all(np.abs(O) <= SO)


ALL_PINS = [
    ("bruteforce_integers", lambda i, o: pin_bruteforce_integers(i, o)),
    ("fsum_bf16", lambda i, o: pin_fsum(i, o, "bf16")),
    ("fsum_f16", lambda i, o: pin_fsum(i, o, "f16")),
    ("fsum_f32", lambda i, o: pin_fsum(i, o, "f32")),
    ("numpy_bf16", lambda i, o: pin_numpy(i, o, "bf16")),
    ("numpy_f32", lambda i, o: pin_numpy(i, o, "f32")),
    ("closed_forms", lambda i, o: pin_closed_forms(i, o)),
    ("invariants", lambda i, o: pin_invariants(i, o)),
]


@pytest.mark.parametrize("name,pin", ALL_PINS, ids=[n for n, _ in ALL_PINS])
def test_oracle_pin(orc, name, pin):
    pin(RealOracle(orc), orc)


def test_points_match_full_arrays(orc):
    ops = gen.uniform(96, 128, 160, "f16", seed=9)
    P, SP = orc.partials(ops.A, ops.B, "f16", 160, 3, 64)
    O, SO = orc.output(ops.A, ops.B, "f16")
    rng = np.random.Generator(np.random.PCG64(1))
    s = rng.integers(-1, 3, 300)
    m = rng.integers(0, 96, 300)
    n = rng.integers(0, 128, 300)
    val, bound = orc.points(ops.A, ops.B, "f16", 64, 3, s, m, n)
    for i in range(300):
        if s[i] < 0:
            assert val[i] == O[m[i], n[i]] and bound[i] == SO[m[i], n[i]]
        else:
            assert val[i] == P[s[i], m[i], n[i]] and bound[i] == SP[s[i], m[i], n[i]]


def test_partials_rejects_illegal_geometry(orc):
    ops = gen.uniform(64, 128, 160, "bf16")
    with pytest.raises(ValueError):
        orc.partials(ops.A, ops.B, "bf16", 160, 2, 64)


def test_generator_recipe(orc):
    """The pages' operands: zero first row, x4 last row, values in [-1,1] (x4: [-4,4])."""
    ops = gen.uniform(96, 512, 2048, "bf16", seed=0)
    a = orc.decode(ops.A, "bf16")
    b = orc.decode(ops.B, "bf16")
    assert np.all(a[0] == 0)
    assert np.abs(a[1:-1]).max() <= 1 and np.abs(b).max() <= 1
    assert np.abs(a[-1]).max() <= 4 and np.abs(a[-1]).max() > 1
    # same seed -> same bits; another seed -> different bits
    assert np.array_equal(gen.uniform(96, 512, 2048, "bf16", seed=0).B, ops.B)
    assert not np.array_equal(gen.uniform(96, 512, 2048, "bf16", seed=1).B, ops.B)


# ------------------------------------------------------- the pins have teeth


class Mutant:
    """A numpy oracle with one planted mistake."""

    def __init__(self, orc, kind):
        self.o, self.kind = orc, kind

    def _dec(self, ops):
        a = self.o.decode(ops.A, ops.dtype)
        b = self.o.decode(ops.B, ops.dtype)
        if self.kind == "transposed_b" and b.shape[0] == b.shape[1]:
            b = b.T.copy()
        if self.kind == "transposed_b" and b.shape[0] != b.shape[1]:
            b = b[::-1].copy()          # rows in the wrong order
        return a, b

    def _dot(self, a, b, k0, k1):
        if self.kind == "dropped_term":
            k1 = max(k0, k1 - 1)
        if self.kind == "off_by_one_start":
            k0 = k0 + 1 if k0 > 0 else k0
        p = a[:, k0:k1] @ b[:, k0:k1].T
        sp = np.abs(a[:, k0:k1]) @ np.abs(b[:, k0:k1]).T
        if self.kind == "no_abs":
            sp = np.abs(p)
        return p, sp

    def partials(self, ops, S, kps):
        a, b = self._dec(ops)
        K = a.shape[1]
        P, SP = [], []
        for s in range(S):
            k0, k1 = s * kps, (s + 1) * kps
            if self.kind != "unclamped":
                k1 = min(k1, K)
            p, sp = self._dot(a, b, k0, k1)
            if self.kind == "wrong_sign" and s == S - 1:
                p = -p
            if self.kind == "unclamped" and (s + 1) * kps > K:
                p = p * (s + 1) * kps / K     # what a padded, rescaled tail would give
            P.append(p)
            SP.append(sp)
        return np.stack(P), np.stack(SP)

    def output(self, ops):
        a, b = self._dec(ops)
        return self._dot(a, b, 0, a.shape[1])


MUTANTS = ["transposed_b", "dropped_term", "off_by_one_start", "no_abs", "wrong_sign",
           "unclamped"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(orc, kind):
    caught = []
    for name, pin in ALL_PINS:
        try:
            pin(Mutant(orc, kind), orc)
        except AssertionError:
            caught.append(name)
    assert caught, f"no pin catches the planted mistake {kind!r}"


def test_numpy_mutant_without_mistake_passes(orc):
    """Control: the same numpy oracle with nothing planted passes every pin."""
    for name, pin in ALL_PINS:
        pin(Mutant(orc, "none"), orc)


def load_int_tile():
    """The stored BF16 M=32 N=64 K=128 integer case: (P[2,32,64], O[32,64])."""
    blocks, cur = {}, None
    with open(os.path.join(GOLDEN, "int_tile_bf16.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line[0].isalpha():
                cur = line
                blocks[cur] = []
            else:
                blocks[cur].append([int(v) for v in line.split()])
    return np.array([blocks["P0"], blocks["P1"]], np.float64), np.array(blocks["O"], np.float64)


def test_golden_int_tile(orc):
    P_ref, O_ref = load_int_tile()
    ops = gen.integers(32, 64, 128, "bf16", seed=3)
    P, _ = orc.partials(ops.A, ops.B, "bf16", 128, 2, 64)
    O, _ = orc.output(ops.A, ops.B, "bf16")
    assert np.array_equal(P, P_ref) and np.array_equal(O, O_ref)
    # exact integers: the two split slabs add up to the unsplit product
    assert np.array_equal(P_ref.sum(axis=0), O_ref)


# ------------------------------------------------------- weight preparation


def test_transpose_worked_example(orc):
    w = np.array([[1, 2, 3, 4], [5, 6, 7, 8], [9, 10, 11, 12]], np.uint16)
    assert orc.transpose(w).tolist() == [[1, 5, 9], [2, 6, 10], [3, 7, 11], [4, 8, 12]]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_transpose_matches_numpy_and_inverts(orc, dtype):
    for K, N in [(32, 64), (160, 128), (96, 320), (2048, 1024)]:
        w = gen.weight_kn(K, N, dtype, seed=K + N)
        b = orc.transpose(w)
        assert b.shape == (N, K)
        assert np.array_equal(b, np.ascontiguousarray(w.T))           # library routine
        assert np.array_equal(orc.transpose(b), w)                    # transposing twice
