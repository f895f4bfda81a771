"""Pins for the oracle's non-uniform THC (THC section 5, Algorithm 2), CPU only.

Fixed by: the page's worked example with T2 = {0, 1, 3, 4} and g = 4 (table
sums equal, index sums differ, same decoded average); the page's statement
that g = 2^b - 1 with the identity table is uniform THC (checked bit for bit
against the uniform oracle); inputs on allowed grid points; the
up-probability between two table values (binomial test); unbiasedness by
exact enumeration of all 2^P outcomes; table validity rules.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "nuhc_t2_example.json")) as f:
        return json.load(f)


def test_t2_worked_example(golden_dir):
    d = _golden(golden_dir)
    b, g, m, M, T = d["b"], d["g"], d["m"], d["M"], d["table"]
    assert oracle.nuhc_table_ok(T, b, g)
    values = [float(Fraction(v)) for v in d["values"]]
    # each table index decodes (one worker) to its quantization value
    vals = oracle.nuhc_decode(np.array(T, np.uint16), m, M, g, 1)
    np.testing.assert_allclose(vals, values, rtol=0, atol=1e-15)
    # the quantized values are grid points, so encoding them is deterministic
    for case in d["cases"]:
        xs = [np.array([float(Fraction(q))], np.float32) for q in case["quantized"]]
        packed = [oracle.nuhc_encode(x, m, M, b, g, T, 123, w) for w, x in enumerate(xs)]
        idx = [int(oracle.thc_unpack(pk, 1, b)[0]) for pk in packed]
        assert idx == case["indices"]
        assert sum(idx) == case["index_sum"]
        Y = oracle.nuhc_aggregate(packed, 1, b, T)
        assert int(Y[0]) == case["table_sum"]
        avg = oracle.nuhc_decode(Y, m, M, g, len(xs))
        assert abs(avg[0] - float(Fraction(d["average_for_table_sum_3"]))) < 1e-15


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_identity_table_is_uniform_thc(b):
    L = (1 << b) - 1
    T = np.arange(L + 1, dtype=np.uint16)
    P, N = 5, 3001
    xs = [np.random.default_rng([111, b, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    avg_u, pk_u = oracle.thc_allreduce(xs, b, 77, m, M, want_packed=True)
    avg_n, pk_n = oracle.nuhc_allreduce(xs, b, L, T, 77, m, M, want_packed=True)
    for a, c in zip(pk_u, pk_n):
        np.testing.assert_array_equal(a, c)
    np.testing.assert_array_equal(avg_u, avg_n)


def test_table_rules():
    assert oracle.nuhc_table_ok([0, 1, 3, 4], 2, 4)
    assert not oracle.nuhc_table_ok([0, 1, 3, 5], 2, 4)     # last entry must be g
    assert not oracle.nuhc_table_ok([1, 2, 3, 4], 2, 4)     # first entry must be 0
    assert not oracle.nuhc_table_ok([0, 2, 2, 4], 2, 4)     # strictly increasing
    assert not oracle.nuhc_table_ok([0, 1, 2], 2, 2)         # g >= 2^b - 1 (and the table is 2^b long)


def test_grid_points_exact():
    # b = 4 with g = 51, the widest granularity the page suggests for b = 4
    b, g = 4, 51
    rng = np.random.default_rng(5)
    inner = np.sort(rng.choice(np.arange(1, g), size=14, replace=False))
    T = np.concatenate([[0], inner, [g]]).astype(np.uint16)
    assert oracle.nuhc_table_ok(T, b, g)
    x = (T.astype(np.float64) / g).astype(np.float32)  # [m, M] = [0, 1]: on the grid only if exact
    exact = (x.astype(np.float64) * g) == T.astype(np.float64)
    pk = oracle.nuhc_encode(x, 0.0, 1.0, b, g, T, 9, 0)
    idx = oracle.thc_unpack(pk, x.size, b)
    # grid points whose fp32 position is exact are sent deterministically
    np.testing.assert_array_equal(idx[exact], np.arange(T.size)[exact])


def test_up_probability_between_table_values():
    # T = {0, 1, 3, 4}, g = 4 on [0, 4]: x = 2 sits halfway between 1 and 3
    T = [0, 1, 3, 4]
    n = 60000
    x = np.full(n, 2.0, np.float32)
    idx = oracle.thc_unpack(oracle.nuhc_encode(x, 0.0, 4.0, 2, 4, T, 31, 0), n, 2)
    assert set(np.unique(idx)) <= {1, 2}
    ups = int((idx == 2).sum())
    assert abs(ups - n / 2) < 5 * math.sqrt(n / 4)
    # x = 1.5: a quarter of the way from 1 to 3
    x = np.full(n, 1.5, np.float32)
    idx = oracle.thc_unpack(oracle.nuhc_encode(x, 0.0, 4.0, 2, 4, T, 32, 1), n, 2)
    ups = int((idx == 2).sum())
    assert abs(ups - n / 4) < 5 * math.sqrt(n * 3 / 16)


def _exact_mean(xs, m, M, b, g, T):
    P, N = len(xs), xs[0].size
    L = (1 << b) - 1
    step = (float(M) - float(m)) / g
    mean = np.zeros(N)
    for e in range(N):
        opts = []
        for w in range(P):
            t = float(oracle.nuhc_position(xs[w][e], m, M, g))
            z = 0
            while z < L - 1 and t >= T[z + 1]:
                z += 1
            lo, hi = float(T[z]), float(T[z + 1])
            p = float(np.float32(np.float32(t - lo) / np.float32(hi - lo)))
            p = math.ceil(p * 2 ** 23) / 2 ** 23
            opts.append((T[z], T[z + 1], p))
        for mask in range(1 << P):
            prob, Y = 1.0, 0
            for w, (lo, hi, p) in enumerate(opts):
                up = (mask >> w) & 1
                prob *= p if up else 1 - p
                Y += hi if up else lo
            mean[e] += prob * (float(m) + Y / P * step)
    return mean


@pytest.mark.parametrize("P", [1, 2, 3])
def test_unbiased_by_enumeration(P):
    b, g = 2, 7
    T = [0, 2, 3, 7]
    N = 32
    xs = [np.random.default_rng([113, P, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    mean = _exact_mean(xs, m, M, b, g, T)
    xbar = np.mean(np.stack(xs).astype(np.float64), axis=0)
    step = (float(M) - float(m)) / g
    bound = step * (4 * 2.0 ** -23 + 4 * g * 2.0 ** -24) + 1e-12
    assert np.all(np.abs(mean - xbar) <= bound)
    # realised averages over many seeds agree with the exact expectation
    K = 2000
    acc = np.zeros(N)
    for seed in range(K):
        acc += oracle.nuhc_allreduce(xs, b, g, T, seed, m, M)
    sigma = step * 4 / (2 * math.sqrt(P)) / math.sqrt(K)  # widest gap (4) bounds the std
    assert np.all(np.abs(acc / K - mean) <= 5.5 * sigma)


def test_aggregate_rejects_overflow():
    T = np.arange(256, dtype=np.uint16)
    T[255] = 300
    with pytest.raises(ValueError):
        oracle.nuhc_aggregate([np.zeros(1, np.uint32)] * 220, 4, 8, T)  # 220 * 300 > 65535


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_encode_at_is_the_whole_vectors_encoding(b):
    """A run of a longer vector, encoded with its global element indices,
    gives that vector's words; with the identity table its indices are the
    uniform round's at those elements."""
    L = (1 << b) - 1
    g = 2 * L + 3
    T = np.rint(np.linspace(0, g, L + 1)).astype(np.uint16)
    N, w = 4099, 3
    x = np.random.default_rng([112, b]).standard_normal(N).astype(np.float32)
    m, M = oracle.thc_range([x])
    full = oracle.nuhc_encode(x, m, M, b, g, T, 91, w)
    per = 32 // b
    for e0 in (0, per, 37 * per, N - N % per):
        run = oracle.nuhc_encode_at(x[e0:], e0, m, M, b, g, T, 91, w)
        np.testing.assert_array_equal(run, full[e0 // per:])
    with pytest.raises(ValueError):  # a run must start on a word boundary
        oracle.nuhc_encode_at(x[1:], 1, m, M, b, g, T, 91, w)
    ident = np.arange(L + 1, dtype=np.uint16)
    e0 = 64 * per
    run = oracle.nuhc_encode_at(x[e0:e0 + 500], e0, m, M, b, L, ident, 91, w)
    vals = np.zeros((w + 1, 500), np.float32)
    vals[w] = x[e0:e0 + 500]
    ind, _ = oracle.thc_allreduce_samples(vals, np.arange(e0, e0 + 500), b, 91, m, M)
    np.testing.assert_array_equal(oracle.thc_unpack(run, 500, b), ind[w])
