"""Pins of the oracle's leaves and canonical tree.

The tree is the "canonical FP32-leaf/BF16-node midpoint reduction tree" of
RL-Kernel PR #325, "Design".  Readings (the page leaves them open): leaf width
64, in-leaf orders SEQ and LANE (8 groups of 8), left child = floor(n/2) leaves.
Pins: integer closed forms (every partial sum exact), exact-rational brute
force with an independent rounding rule, hand-enumerated parenthesisations,
and the hand-derived fixtures in tests/golden/.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    from gemm_deterministic_bf16_gb300.inputs import to_bf16_bits
    return to_bf16_bits(np.asarray(vals, np.float32))


def _exact_leaf(a_bits, b_bits, lw, order):
    """Leaf by exact rationals: acc <- RN32(acc + a*b) (the product is exact)."""
    a = [exact.bf16_value(int(v)) for v in a_bits]
    b = [exact.bf16_value(int(v)) for v in b_bits]
    n = len(a)
    if order == 0:
        acc = Fraction(0)
        for k in range(n):
            acc = exact.rn(acc + a[k] * b[k])
        return acc
    gw = lw // 8
    s = []
    for g in range(8):
        acc = Fraction(0)
        for e in range(gw):
            k = g * gw + e
            if k < n:
                acc = exact.rn(acc + a[k] * b[k])
        s.append(acc)
    p = [exact.rn(s[0] + s[1]), exact.rn(s[2] + s[3]), exact.rn(s[4] + s[5]), exact.rn(s[6] + s[7])]
    return exact.rn(exact.rn(p[0] + p[1]) + exact.rn(p[2] + p[3]))


@pytest.mark.parametrize("order", [0, 1])
def test_leaf_integer_closed_form(oracle_mod, order):
    """Integers |a|,|b| <= 8: every partial sum is an integer below 2^24, so
    the leaf is the exact dot product whatever the order."""
    rng = np.random.default_rng(10)
    for K in [1, 7, 8, 9, 33, 63, 64]:
        a = rng.integers(-8, 9, K)
        b = rng.integers(-8, 9, K)
        got = oracle_mod.leaf(_bf16(a), _bf16(b), 64, order)
        assert got == float(np.dot(a, b))


@pytest.mark.parametrize("order", [0, 1])
def test_leaf_exact_rational_brute_force(oracle_mod, order):
    rng = np.random.default_rng(11 + order)
    for trial in range(60):
        K = int(rng.integers(1, 65))
        scale = 10.0 ** rng.integers(-3, 4)
        a = _bf16(rng.standard_normal(K) * scale)
        b = _bf16(rng.standard_normal(K))
        got = oracle_mod.leaf(a, b, 64, order)
        want = _exact_leaf(a, b, 64, order)
        assert Fraction(got) == want, (trial, K)


def test_leaf_orders_differ(oracle_mod):
    """Sanity of the brute force: SEQ and LANE give different leaves on some
    random data, so the pins above distinguish the two orders."""
    rng = np.random.default_rng(12)
    diff = 0
    for _ in range(50):
        a = _bf16(rng.standard_normal(64) * 100)
        b = _bf16(rng.standard_normal(64))
        diff += oracle_mod.leaf(a, b, 64, 0) != oracle_mod.leaf(a, b, 64, 1)
    assert diff > 5


# Hand-enumerated parenthesisations of the midpoint tree with left = floor(n/2).
PAREN = {
    1: 0,
    2: (0, 1),
    3: (0, (1, 2)),
    4: ((0, 1), (2, 3)),
    5: ((0, 1), (2, (3, 4))),
    6: ((0, (1, 2)), (3, (4, 5))),
    7: ((0, (1, 2)), ((3, 4), (5, 6))),
    8: (((0, 1), (2, 3)), ((4, 5), (6, 7))),
    12: (((0, (1, 2)), (3, (4, 5))), ((6, (7, 8)), (9, (10, 11)))),
}


def _eval_paren(p, leaves):
    if isinstance(p, int):
        return Fraction(float(leaves[p]))
    l, r = _eval_paren(p[0], leaves), _eval_paren(p[1], leaves)
    return exact.rn(exact.rn(l + r, exact.F32), exact.BF16)


@pytest.mark.parametrize("L", sorted(PAREN))
def test_tree_matches_enumerated_parenthesisation(oracle_mod, L):
    rng = np.random.default_rng(20 + L)
    for _ in range(200):
        lv = (rng.standard_normal(L) * 10.0 ** rng.integers(-2, 3, L)).astype(np.float32)
        got = oracle_mod.tree_from_leaves(lv)
        root = _eval_paren(PAREN[L], lv)
        want = exact.rn(root, exact.BF16)  # a no-op for internal nodes, rounds a lone leaf
        assert got == exact.bf16_bits_of(float(want))


def test_tree_integer_closed_form(oracle_mod):
    """Entries in {-1,0,1}, K=256 (4 leaves): every leaf and node is an integer
    of magnitude <= 256, exact in BF16, so the output is the exact sum."""
    rng = np.random.default_rng(30)
    A = rng.integers(-1, 2, (7, 256))
    B = rng.integers(-1, 2, (5, 256))
    out = oracle_mod.tree_gemm(_bf16(A), _bf16(B))
    want = _bf16(A @ B.T)
    assert np.array_equal(out, want)


def test_single_leaf_is_rounded_dot(oracle_mod):
    """L = 1: the output is the leaf rounded once to BF16."""
    rng = np.random.default_rng(31)
    a = _bf16(rng.standard_normal(40))
    b = _bf16(rng.standard_normal(40))
    lv = oracle_mod.leaf(a, b, 64, 1)
    out = oracle_mod.tree_gemm(a[None], b[None])[0, 0]
    assert out == oracle_mod.rne_bf16(np.float32([lv]))[0]


def test_empty_contraction_is_positive_zero(oracle_mod):
    out = oracle_mod.tree_gemm(np.zeros((3, 0), np.uint16), np.zeros((2, 0), np.uint16))
    assert out.shape == (3, 2) and not out.any()


def test_gemm_is_leaves_then_tree(oracle_mod):
    """tree_gemm = replay of tree_leaves, and the leaves are the brute-force
    leaves, including a partial last leaf (K = 150 -> 64, 64, 22)."""
    rng = np.random.default_rng(32)
    A = _bf16(rng.standard_normal((3, 150)))
    B = _bf16(rng.standard_normal((2, 150)) * 0.02)
    out = oracle_mod.tree_gemm(A, B)
    lv = oracle_mod.tree_leaves(A, B)
    assert lv.shape == (3, 2, 3)
    assert np.array_equal(oracle_mod.tree_replay(lv), out)
    for r in range(3):
        for c in range(2):
            for j, (k0, k1) in enumerate([(0, 64), (64, 128), (128, 150)]):
                assert Fraction(float(lv[r, c, j])) == _exact_leaf(A[r, k0:k1], B[c, k0:k1], 64, 1)


def test_golden_fixtures(oracle_mod):
    with open(os.path.join(GOLDEN, "tree_cases.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        if case["kind"] == "tree":
            lv = np.float32([float.fromhex(v) for v in case["leaves"]])
            assert oracle_mod.tree_from_leaves(lv) == int(case["expect_bits"], 16), case["name"]
        elif case["kind"] == "rank_tree_bf16":
            bufs = [_bf16([float.fromhex(v)]) for v in case["buffers"]]
            got = oracle_mod.rank_tree(bufs, oracle_mod.BF16)[0]
            assert got == int(case["expect_bits"], 16), case["name"]
        elif case["kind"] == "rank_tree_f16":
            bufs = [np.float16([float.fromhex(v)]).view(np.uint16) for v in case["buffers"]]
            got = oracle_mod.rank_tree(bufs, oracle_mod.F16)[0]
            assert got == int(case["expect_bits"], 16), case["name"]
        elif case["kind"] == "rank_tree_f32":
            bufs = [np.float32([float.fromhex(v)]) for v in case["buffers"]]
            got = oracle_mod.rank_tree(bufs, oracle_mod.F32)
            assert int(got.view(np.uint32)[0]) == int(case["expect_bits"], 16), case["name"]
        elif case["kind"] == "leaf_lane":
            a = _bf16([float.fromhex(v) for v in case["a"]])
            b = _bf16([float.fromhex(v) for v in case["b"]])
            assert oracle_mod.leaf(a, b, 64, 1) == float.fromhex(case["expect"]), case["name"]
        else:
            raise AssertionError(case["kind"])


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_rank_tree_integers_are_exact_in_every_dtype(oracle_mod, n):
    """Small integers add exactly in FP32, FP16 and BF16 whatever the order:
    the rank tree must then return the exact sum (n = 1: the buffer itself)."""
    rng = np.random.default_rng(n)
    ints = [rng.integers(-16, 17, 1000) for _ in range(n)]   # |sum| <= 128: exact in BF16
    want = np.sum(ints, axis=0).astype(np.float32)
    got32 = oracle_mod.rank_tree([v.astype(np.float32) for v in ints], oracle_mod.F32)
    assert np.array_equal(got32, want)
    got16 = oracle_mod.rank_tree([v.astype(np.float16).view(np.uint16) for v in ints], oracle_mod.F16)
    assert np.array_equal(got16.view(np.float16).astype(np.float32), want)
    gotb = oracle_mod.rank_tree([_bf16(v.astype(np.float32)) for v in ints], oracle_mod.BF16)
    assert np.array_equal((gotb.astype(np.uint32) << 16).view(np.float32), want)
