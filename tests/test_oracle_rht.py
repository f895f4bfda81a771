"""Pins for the oracle's RHT pre/post-processing (THC section 5), CPU only.

Fixed by: scipy's Sylvester-Hadamard matrix (the transform equals
(1/sqrt(n)) H D x with H from scipy.linalg.hadamard); inverse after forward
is the identity; the transform preserves the norm; a one-hot vector spreads
to magnitude 1/sqrt(n) everywhere; the page's statements that transformed
coordinates approach a normal distribution and that about a p fraction of
them fall outside (t_p / sqrt(n)) ||x|| with t_p = Phi^-1(1 - p/2); and the
rotation commutes with averaging because every worker uses the same signs.
"""
import math

import numpy as np
import pytest

import oracle
import workloads


@pytest.mark.parametrize("k", [0, 1, 2, 3, 5, 8, 10])
def test_matches_explicit_hadamard(k):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    n = 1 << k
    x = np.random.default_rng([161, k]).standard_normal(n)
    d = oracle.rht_signs(n, 12345).astype(np.float64)
    H = scipy_linalg.hadamard(n).astype(np.float64)
    ref = H @ (d * x) / math.sqrt(n)
    np.testing.assert_allclose(oracle.rht(x, 12345), ref, rtol=0, atol=1e-12 * max(1.0, np.abs(x).sum()))
    inv_ref = d * (H @ x) / math.sqrt(n)
    np.testing.assert_allclose(oracle.rht(x, 12345, inverse=True), inv_ref, rtol=0,
                               atol=1e-12 * max(1.0, np.abs(x).sum()))


@pytest.mark.parametrize("k", [4, 12, 16])
def test_inverse_and_norm(k):
    n = 1 << k
    x = np.random.default_rng([162, k]).standard_normal(n)
    y = oracle.rht(x, 7)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)
    np.testing.assert_allclose(oracle.rht(y, 7, inverse=True), x, rtol=0, atol=1e-12 * np.linalg.norm(x))
    with pytest.raises(ValueError):
        oracle.rht(np.zeros(n + 1), 7)  # not a power of two


def test_signs_are_fair_and_seeded():
    n = 1 << 16
    d = oracle.rht_signs(n, 99)
    assert set(np.unique(d)) == {-1, 1}
    neg = int((d < 0).sum())
    assert abs(neg - n / 2) < 5 * math.sqrt(n / 4)
    assert not np.array_equal(d, oracle.rht_signs(n, 100))
    np.testing.assert_array_equal(d, oracle.rht_signs(n, 99))
    # the sign of element i is bit i mod 128 of its Philox block
    for i in (0, 1, 31, 32, 127, 128, 4000):
        r = oracle.philox4x32([i >> 7, 0, 0xFFFFFFFF, 0], [99, 0])
        bit = (int(r[(i >> 5) & 3]) >> (i & 31)) & 1
        assert d[i] == (-1 if bit else 1)


def test_one_hot_spreads_evenly():
    n = 1 << 10
    for k in (0, 5, 1023):
        x = np.zeros(n)
        x[k] = 3.0
        y = oracle.rht(x, 5)
        np.testing.assert_allclose(np.abs(y), 3.0 / math.sqrt(n), rtol=1e-14)


def test_coordinates_become_gaussian_and_p_fraction_outside():
    stats = pytest.importorskip("scipy.stats")
    n = 1 << 16
    x = workloads.student_t_f32(n, 3, 1.0, 7, 0).astype(np.float64)  # heavy tails
    y = oracle.rht(x, 2024)
    kurt_x = float(np.mean(x ** 4) / np.mean(x ** 2) ** 2)
    kurt_y = float(np.mean(y ** 4) / np.mean(y ** 2) ** 2)
    assert kurt_x > 6 and abs(kurt_y - 3.0) < 0.15
    for p in (1 / 32, 1 / 512):
        t_p = stats.norm.ppf(1 - p / 2)
        m, M = oracle.rht_norm_range([x], t_p)
        assert m == -M and abs(M - t_p / math.sqrt(n) * np.linalg.norm(x)) <= 1e-12 * M
        frac = float(np.mean(np.abs(y) > M))
        assert abs(frac - p) < 6 * math.sqrt(p * (1 - p) / n) + 0.1 * p


def test_norm_range_takes_the_largest_worker():
    xs = [np.random.default_rng([163, w]).standard_normal(256) * (w + 1) for w in range(4)]
    m, M = oracle.rht_norm_range(xs, 2.0)
    assert abs(M - 2.0 / 16 * max(np.linalg.norm(x) for x in xs)) < 1e-12


def test_rotation_commutes_with_averaging():
    n = 1 << 12
    xs = [np.random.default_rng([164, w]).standard_normal(n) for w in range(5)]
    lhs = np.mean([oracle.rht(x, 3) for x in xs], axis=0)
    rhs = oracle.rht(np.mean(xs, axis=0), 3)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
