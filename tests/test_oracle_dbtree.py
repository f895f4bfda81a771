"""Pins of the oracle's double-binary-tree all-reduce.

The tutorial "Collective Communication: Ring All-Reduce" compares the ring
with a double-binary-tree all-reduce ("Design Alternatives & Collective
Comparison Matrix: Ring vs. Tree vs. NVLS"): two complementary trees, each
carrying half of the data, about 2 log2(P) latency steps against the ring's
2(P - 1), about 2M bytes sent per rank.  It prints no construction; the
oracle reads it as the two-tree scheme of Sanders, Speck and Traff (2009):
tree 1 the in-order binary tree on labels 1..P (label l on rank l - 1),
tree 2 its mirror image (P even) or its shift by one (P odd).

Pinned here against things the oracle's code does not produce itself:
trees and fold expressions derived by hand for small P, a second
construction of the parent links from bit arithmetic, the step count and
the per-rank volume the tutorial states, the complement property of the two
trees, exact integer sums, and the literal message-passing schedule.
"""
import numpy as np
import pytest

import oracle

SUM, AVG = oracle.SUM, oracle.AVG


def f32(v):
    return np.float32(v)


# ---------------------------------------------------------------- trees by hand
# (root, {rank: (left, right)}) for every rank with children; ranks not listed
# are leaves.  Derived on paper from the labels: the run 1..P splits at the
# label with the most trailing zeros.
HAND = {
    # P=4: labels 4 (root) / 2 / 1, 3.  Tree 1: label l on rank l-1.
    # Tree 2 (P even): label l on rank 4 - l.
    (4, 0): (3, {3: (1, -1), 1: (0, 2)}),
    (4, 1): (0, {0: (2, -1), 2: (3, 1)}),
    # P=5: labels 4 (root) / 2, 5 / 1, 3.  Tree 2 (P odd): label l on rank (l-2) mod 5.
    (5, 0): (3, {3: (1, 4), 1: (0, 2)}),
    (5, 1): (2, {2: (0, 3), 0: (4, 1)}),
    # P=6: labels 4 (root) / 2, 6 / 1, 3, 5 (5 is 6's left child).
    (6, 0): (3, {3: (1, 5), 1: (0, 2), 5: (4, -1)}),
    (6, 1): (2, {2: (4, 0), 4: (5, 3), 0: (1, -1)}),
    # P=3: labels 2 (root) / 1, 3.
    (3, 0): (1, {1: (0, 2)}),
    (3, 1): (0, {0: (2, 1)}),
}


@pytest.mark.parametrize("key", sorted(HAND))
def test_trees_match_hand_derivation(key):
    p, tree = key
    root, kids = HAND[key]
    r, par, lc, rc = oracle.dbtree_build(p, tree)
    assert r == root
    for w in range(p):
        assert (lc[w], rc[w]) == kids.get(w, (-1, -1)), (key, w)
    for w, (a, b) in kids.items():
        for c in (a, b):
            if c >= 0:
                assert par[c] == w
    assert par[root] == -1


def _label_parent(label, p):
    """Parent label in the in-order tree on 1..p from bit arithmetic alone:
    of the two nearest labels with more trailing zeros, i - 2^k and i + 2^k,
    the one inside 1..p with fewer trailing zeros (0: the root)."""
    k = (label & -label).bit_length() - 1
    lo, hi = label - (1 << k), label + (1 << k)
    cands = [c for c in (lo, hi) if 1 <= c <= p]
    if not cands:
        return 0
    return min(cands, key=lambda c: (c & -c))


def _rank_of(label, p, tree):
    if tree == 0:
        return label - 1
    return p - label if p % 2 == 0 else (label - 2) % p


@pytest.mark.parametrize("tree", [0, 1])
def test_parent_links_match_bit_construction(tree):
    for p in range(1, 65):
        root, par, lc, rc = oracle.dbtree_build(p, tree)
        for label in range(1, p + 1):
            up = _label_parent(label, p)
            want = -1 if up == 0 else _rank_of(up, p, tree)
            assert par[_rank_of(label, p, tree)] == want, (p, tree, label)
        # every rank once, one root, children consistent with parents
        assert sorted(np.flatnonzero(par == -1).tolist()) == [root]
        for w in range(p):
            for c in (lc[w], rc[w]):
                if c >= 0:
                    assert par[c] == w


def test_complementary_trees():
    """No rank is interior in both trees (for every P: with the mirror for
    even P and the shift for odd P, tree 1's interior ranks are odd and
    tree 2's even)."""
    for p in range(2, 65):
        interior = []
        for tree in (0, 1):
            _, _, lc, rc = oracle.dbtree_build(p, tree)
            interior.append({w for w in range(p) if lc[w] >= 0 or rc[w] >= 0})
        assert not (interior[0] & interior[1]), p


# ------------------------------------------------------- fold order by hand
def _spread(rng, p, n):
    """fp32 values over many binades, so that the association order of a sum
    shows in its rounding."""
    mag = np.float32(10.0) ** rng.uniform(-4, 4, size=(p, n)).astype(np.float32)
    return [(rng.standard_normal(n).astype(np.float32) * mag[w]).astype(np.float32) for w in range(p)]


def test_p4_fold_matches_hand_expressions():
    rng = np.random.default_rng(11)
    n = 4001
    x = _spread(rng, 4, n)
    got = oracle.dbtree_fold(x, SUM)
    h = oracle.dbtree_half(n)
    assert h == 2001
    # tree 1: rank 3 on top of rank 1 (children 0, 2); tree 2: rank 0 on top of rank 2 (children 3, 1)
    t1 = x[3] + ((x[1] + x[0]) + x[2])
    t2 = x[0] + ((x[2] + x[3]) + x[1])
    np.testing.assert_array_equal(got[:h], t1[:h])
    np.testing.assert_array_equal(got[h:], t2[h:])
    # the order matters for these inputs: the ring order differs somewhere
    assert np.any(got != oracle.ring_fold(x, SUM))
    assert np.any(t1 != t2)


def test_p6_fold_matches_hand_expressions():
    rng = np.random.default_rng(12)
    n = 3000
    x = _spread(rng, 6, n)
    got = oracle.dbtree_fold(x, AVG)
    h = n // 2
    # tree 1: s(3) = (x3 + s(1)) + s(5), s(1) = (x1 + x0) + x2, s(5) = x5 + x4
    t1 = (x[3] + ((x[1] + x[0]) + x[2])) + (x[5] + x[4])
    # tree 2: s(2) = (x2 + s(4)) + s(0), s(4) = (x4 + x5) + x3, s(0) = x0 + x1
    t2 = (x[2] + ((x[4] + x[5]) + x[3])) + (x[0] + x[1])
    np.testing.assert_array_equal(got[:h], t1[:h] / f32(6))
    np.testing.assert_array_equal(got[h:], t2[h:] / f32(6))


def test_p5_shifted_tree_fold():
    rng = np.random.default_rng(13)
    n = 2001
    x = _spread(rng, 5, n)
    got = oracle.dbtree_fold(x, SUM)
    h = 1001
    # tree 1: s(3) = (x3 + s(1)) + x4, s(1) = (x1 + x0) + x2
    t1 = (x[3] + ((x[1] + x[0]) + x[2])) + x[4]
    # tree 2: s(2) = (x2 + s(0)) + x3, s(0) = (x0 + x4) + x1
    t2 = (x[2] + ((x[0] + x[4]) + x[1])) + x[3]
    np.testing.assert_array_equal(got[:h], t1[:h])
    np.testing.assert_array_equal(got[h:], t2[h:])


# ------------------------------------------------------------ tutorial facts
@pytest.mark.parametrize("p", list(range(1, 17)) + [24, 31, 32, 33, 48, 63, 64])
def test_schedule_steps_and_volume(p):
    """About 2 log2(P) latency steps (exactly 2 floor(log2 P) for these
    balanced in-order trees), against the ring's 2(P - 1); every rank but a
    root sends its half once per tree up and each interior rank copies it to
    its children, so the whole job moves 2 (P - 1) n elements, like the
    ring, and no rank sends much more than 2n ("about 2M")."""
    rng = np.random.default_rng(p)
    n = 37
    bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
    steps, sent = oracle.dbtree_schedule([b.copy() for b in bufs], SUM)
    lg = p.bit_length() - 1
    assert steps == 2 * lg
    if p >= 3:
        assert steps < 2 * (p - 1)
    assert sent.sum() == 2 * (p - 1) * n
    assert sent.max() <= n + 2 * oracle.dbtree_half(n)


@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 17, 31, 64])
@pytest.mark.parametrize("op", [SUM, AVG])
def test_schedule_equals_closed_form(p, op):
    rng = np.random.default_rng(100 + p)
    for n in (0, 1, 2, 7, 64, 129):
        x = _spread(rng, p, n) if n else [np.zeros(0, np.float32) for _ in range(p)]
        bufs = [a.copy() for a in x]
        oracle.dbtree_schedule(bufs, op)
        want = oracle.dbtree_fold(x, op)
        for w in range(p):
            np.testing.assert_array_equal(bufs[w], want, err_msg=f"p={p} n={n} rank {w}")


@pytest.mark.parametrize("p", [2, 3, 5, 8, 13, 64])
def test_exact_integer_sums(p):
    """Small integers: every association order gives the exact sum, so a
    dropped or doubled addend shows."""
    rng = np.random.default_rng(200 + p)
    n = 1000
    ints = rng.integers(-1000, 1000, size=(p, n))
    x = [ints[w].astype(np.float32) for w in range(p)]
    np.testing.assert_array_equal(oracle.dbtree_fold(x, SUM), ints.sum(axis=0).astype(np.float32))
    if p & (p - 1) == 0:  # division by a power of two is exact
        np.testing.assert_array_equal(oracle.dbtree_fold(x, AVG), (ints.sum(axis=0) / p).astype(np.float32))


def test_degenerate_cases():
    rng = np.random.default_rng(5)
    x = [rng.standard_normal(9).astype(np.float32)]
    np.testing.assert_array_equal(oracle.dbtree_fold(x, SUM), x[0])
    np.testing.assert_array_equal(oracle.dbtree_fold(x, AVG), x[0])
    y = _spread(rng, 2, 9)
    np.testing.assert_array_equal(oracle.dbtree_fold(y, SUM), y[0] + y[1])
    z = [np.ones(1, np.float32) * 3, np.ones(1, np.float32) * 4, np.ones(1, np.float32) * 5]
    np.testing.assert_array_equal(oracle.dbtree_fold(z, SUM), np.array([12], np.float32))
    assert oracle.dbtree_half(0) == 0 and oracle.dbtree_half(1) == 1 and oracle.dbtree_half(2) == 1
    with pytest.raises(ValueError):
        oracle.dbtree_build(0, 0)
    with pytest.raises(ValueError):
        oracle.dbtree_build(65, 0)


def _to_bf16(a):
    """fp32 -> bf16 bits, nearest even (finite inputs)."""
    u = a.view(np.uint32).astype(np.uint64)
    up = ((u & 0xFFFF) > 0x8000) | (((u & 0xFFFF) == 0x8000) & (((u >> 16) & 1) == 1))
    return ((u >> 16) + up.astype(np.uint64)).astype(np.uint16)


def test_bf16_is_one_rounding_of_the_fp32_fold():
    rng = np.random.default_rng(21)
    p, n = 7, 999
    xb = [_to_bf16(a) for a in _spread(rng, p, n)]
    widened = [(b.astype(np.uint32) << 16).view(np.float32) for b in xb]
    for op in (SUM, AVG):
        np.testing.assert_array_equal(oracle.dbtree_fold(xb, op), _to_bf16(oracle.dbtree_fold(widened, op)))


def test_samples_match_full_fold():
    rng = np.random.default_rng(22)
    p, n = 9, 5001
    x = _spread(rng, p, n)
    idx = np.array([0, 1, 2500, 2501, 2502, 5000, 4321], np.int64)
    vals = np.stack([a[idx] for a in x])
    np.testing.assert_array_equal(oracle.dbtree_fold_samples(vals, n, idx, AVG), oracle.dbtree_fold(x, AVG)[idx])
    xb = [_to_bf16(a) for a in x]
    valsb = np.stack([a[idx] for a in xb])
    np.testing.assert_array_equal(oracle.dbtree_fold_samples(valsb, n, idx, SUM), oracle.dbtree_fold(xb, SUM)[idx])
