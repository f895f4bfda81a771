"""Pins for the oracle's uniform THC path and NMSE (CPU only).

What fixes the oracle here, other than the oracle itself: the published
Philox4x32 known-answer vectors, the THC page's worked example of the
uniform table T0, inputs on grid points (no randomness left), the SQ
up-probability (binomial tests), unbiasedness (mean over seeds), an exact
expectation by enumerating all 2^P up/down outcomes on tiny inputs, the
closed-form USQ variance behind the expected NMSE, the hand-written packing
layout, and numpy's own min/max/sum/norm for the plain definitions.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_philox_known_answers(golden_dir):
    g = _golden(golden_dir, "philox4x32_kat.json")
    for v in g["vectors"]:
        ctr = [int(h, 16) for h in v["counter"]]
        key = [int(h, 16) for h in v["key"]]
        out = oracle.philox4x32(ctr, key, v["rounds"])
        assert [format(int(o), "08x") for o in out] == v["out"]


def test_grid_worked_example(golden_dir):
    g = _golden(golden_dir, "thc_usq_b2.json")
    b, m, M = g["b"], g["m"], g["M"]
    L = (1 << b) - 1
    T0 = [float(eval(s)) for s in g["T0"]]  # "-1/3" style fractions
    # one worker: the decoded value of index z is the grid point T0[z]
    vals = oracle.thc_decode(np.arange(L + 1, dtype=np.uint16), m, M, b, 1)
    np.testing.assert_allclose(vals, T0, rtol=0, atol=1e-15)
    # two workers whose indices sum to 3: the average is 0, so the value sum is 0
    for z, z2 in g["index_pairs_summing_to_3"]:
        avg = oracle.thc_decode(np.array([z + z2], np.uint16), m, M, b, 2)
        assert abs(avg[0] * 2 - g["value_sum_for_index_sum_3"]) < 1e-15
        assert abs((T0[z] + T0[z2]) - 2 * avg[0]) < 1e-15


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_grid_point_inputs_are_exact(b):
    # [m, M] = [0, L]: the scale is exactly 1, every integer input is a grid
    # point (f = 0) and its index is the input itself, whatever the seed
    L = (1 << b) - 1
    x = np.tile(np.arange(L + 1, dtype=np.float32), 3)
    for seed in (0, 1, 0xDEADBEEFCAFE):
        for worker in (0, 5):
            pk = oracle.thc_encode(x, 0.0, float(L), b, seed, worker)
            np.testing.assert_array_equal(oracle.thc_unpack(pk, x.size, b), x.astype(np.uint8))
    # the two ends of any range map to indices 0 and L
    x2 = np.array([-1.0, 1.0, -1.0], np.float32)
    np.testing.assert_array_equal(oracle.thc_unpack(oracle.thc_encode(x2, -1.0, 1.0, b, 3, 0), 3, b),
                                  [0, L, 0])


def test_degenerate_range():
    x = np.full(37, 0.75, np.float32)
    pk = oracle.thc_encode(x, 0.75, 0.75, 4, 9, 0)
    assert np.all(oracle.thc_unpack(pk, 37, 4) == 0)
    avg = oracle.thc_allreduce([x, x, x], 4, 9)
    assert np.all(avg == 0.75)


@pytest.mark.parametrize("b", [2, 4, 8])
def test_indices_are_floor_or_ceil(b):
    L = (1 << b) - 1
    x = np.random.default_rng(31).standard_normal(4000).astype(np.float32)
    m, M = float(x.min()), float(x.max())
    idx = oracle.thc_unpack(oracle.thc_encode(x, m, M, b, 77, 2), x.size, b)
    t = (x.astype(np.float64) - m) / (M - m) * L
    lo = np.floor(t - 1e-4)
    hi = np.ceil(t + 1e-4)
    assert np.all(idx >= np.maximum(lo, 0)) and np.all(idx <= np.minimum(hi, L))


@pytest.mark.parametrize("frac", [0.25, 0.5, 0.75, 0.1])
def test_up_probability_is_fraction(frac):
    # b = 2 on [0, 3]: x = 1 + frac has j = 1 and f = frac (fp32), so it goes
    # up with probability ~frac; count ups over many coordinates and workers
    n = 40000
    xv = np.float32(1.0 + frac)
    f = float(xv) - 1.0
    x = np.full(n, xv, np.float32)
    ups = 0
    for worker in range(3):
        idx = oracle.thc_unpack(oracle.thc_encode(x, 0.0, 3.0, 2, 1234, worker), n, 2)
        assert set(np.unique(idx)) <= {1, 2}
        ups += int((idx == 2).sum())
    total = 3 * n
    sigma = math.sqrt(total * f * (1 - f))
    assert abs(ups - total * f) < 5 * sigma


def test_workers_and_elements_draw_independently():
    n = 50000
    x = np.full(n, np.float32(1.5), np.float32)
    a = oracle.thc_unpack(oracle.thc_encode(x, 0.0, 3.0, 2, 99, 0), n, 2).astype(np.float64)
    bb = oracle.thc_unpack(oracle.thc_encode(x, 0.0, 3.0, 2, 99, 1), n, 2).astype(np.float64)
    c = oracle.thc_unpack(oracle.thc_encode(x, 0.0, 3.0, 2, 100, 0), n, 2).astype(np.float64)
    lim = 5 / math.sqrt(n)
    assert abs(np.corrcoef(a, bb)[0, 1]) < lim  # other worker
    assert abs(np.corrcoef(a, c)[0, 1]) < lim  # other seed
    assert abs(np.corrcoef(a[:-1], a[1:])[0, 1]) < lim  # neighbouring elements
    assert abs(np.corrcoef(a[:-4], a[4:])[0, 1]) < lim  # next Philox block


def _bias_bound(m, M, b):
    L = (1 << b) - 1
    step = (M - m) / L
    # p is f rounded up to 2^-23; the fp32 position carries about 4 roundings of t <= L
    return step * (2.0 ** -23 + 4 * L * 2.0 ** -24) + 1e-12


def _exact_moments(xs, m, M, b):
    """E and Var of the decoded average by enumerating all 2^P up/down outcomes."""
    P, N = len(xs), xs[0].size
    L = (1 << b) - 1
    step = (float(M) - float(m)) / L
    mean = np.zeros(N)
    second = np.zeros(N)
    for e in range(N):
        js, ps = [], []
        for w in range(P):
            t = float(oracle.thc_position(xs[w][e], m, M, b))
            j = math.floor(t)
            f = t - j
            js.append(j)
            ps.append(math.ceil(f * 2 ** 23) / 2 ** 23)  # P(u < f), u on the 2^-23 grid
        for mask in range(1 << P):
            prob, s = 1.0, sum(js)
            for w in range(P):
                up = (mask >> w) & 1
                prob *= ps[w] if up else 1 - ps[w]
                s += up
            val = float(m) + s / P * step
            mean[e] += prob * val
            second[e] += prob * val * val
    return mean, second - mean ** 2


@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("b", [2, 4])
def test_brute_force_expectation_is_unbiased(P, b):
    N = 64
    xs = [np.random.default_rng([41, P, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    mean, var = _exact_moments(xs, m, M, b)
    xbar = np.mean(np.stack(xs).astype(np.float64), axis=0)
    assert np.all(np.abs(mean - xbar) <= _bias_bound(m, M, b))
    # the closed-form USQ variance: (step / P)^2 sum_w p(1-p) <= step^2 / (4P)
    step = (float(M) - float(m)) / ((1 << b) - 1)
    assert np.all(var <= step ** 2 / (4 * P) * (1 + 1e-9))
    # the oracle's realised averages over many seeds agree with the exact moments
    K = 1500
    acc = np.zeros(N)
    for seed in range(K):
        acc += oracle.thc_allreduce(xs, b, seed, m, M)
    emp = acc / K
    sigma = np.sqrt(var / K) + 1e-15
    assert np.all(np.abs(emp - mean) <= 5.5 * sigma + 1e-12)


def test_unbiased_over_seeds_sweep_shape():
    # Student-t(3) gradients like the THC sweep, P = 16, b = 2
    P, N, b = 16, 256, 2
    xs = [workloads.student_t_f32(N, 3, 1e-3, 4, w) for w in range(P)]
    m, M = oracle.thc_range(xs)
    xbar = np.mean(np.stack(xs).astype(np.float64), axis=0)
    K = 400
    acc = np.zeros(N)
    for seed in range(K):
        acc += oracle.thc_allreduce(xs, b, 1000 + seed, m, M)
    step = (float(M) - float(m)) / 3
    sigma = math.sqrt(step ** 2 / (4 * P) / K)
    assert np.all(np.abs(acc / K - xbar) <= 5.5 * sigma + _bias_bound(m, M, b))


def test_decode_is_homomorphic():
    # decoding the index sum equals averaging the per-worker decoded values
    P, N, b = 5, 300, 4
    xs = [np.random.default_rng([43, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    avg, packed = oracle.thc_allreduce(xs, b, 5, m, M, want_packed=True)
    per = [oracle.thc_decode(oracle.thc_unpack(pk, N, b).astype(np.uint16), m, M, b, 1) for pk in packed]
    np.testing.assert_allclose(avg, np.mean(per, axis=0), rtol=0, atol=1e-12 * (float(M) - float(m)))


def test_nmse_matches_closed_form():
    P, N, b = 4, 1 << 16, 4
    xs = [workloads.student_t_f32(N, 3, 1e-3, 4, w) for w in range(P)]
    m, M = oracle.thc_range(xs)
    L = (1 << b) - 1
    step = (float(M) - float(m)) / L
    xbar = np.mean(np.stack(xs).astype(np.float64), axis=0)
    # expected squared error per coordinate: (step / P)^2 sum_w p(1 - p)
    var = np.zeros(N)
    for w in range(P):
        t = np.array([oracle.thc_position(v, m, M, b) for v in xs[w]], np.float64)
        f = t - np.floor(t)
        p = np.ceil(f * 2 ** 23) / 2 ** 23
        var += p * (1 - p)
    expect = (step / P) ** 2 * var.sum() / np.dot(xbar, xbar)
    got = oracle.nmse(xbar, oracle.thc_allreduce(xs, b, 2024, m, M))
    assert abs(got - expect) < 0.05 * expect
    assert got <= N * step ** 2 / (4 * P * np.dot(xbar, xbar))


def test_packing_layout(golden_dir):
    g = _golden(golden_dir, "thc_packing.json")
    for case in g["cases"]:
        b = case["b"]
        L = (1 << b) - 1
        x = np.array(case["indices"], np.float32)  # on-grid inputs: index == value on [0, L]
        words = oracle.thc_encode(x, 0.0, float(L), b, 0, 0)
        assert [format(int(w), "08x") for w in words] == case["words"]
        np.testing.assert_array_equal(oracle.thc_unpack(words, x.size, b), case["indices"])


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_aggregate_is_integer_sum(b):
    P, N = 7, 1001
    xs = [np.random.default_rng([47, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    packed = [oracle.thc_encode(x, m, M, b, 8, w) for w, x in enumerate(xs)]
    sums = oracle.thc_aggregate(packed, N, b)
    ref = np.sum([oracle.thc_unpack(pk, N, b).astype(np.int64) for pk in packed], axis=0)
    np.testing.assert_array_equal(sums, ref)


def test_aggregate_rejects_overflow():
    packed = [np.zeros(1, np.uint32)] * 258
    with pytest.raises(ValueError):
        oracle.thc_aggregate(packed, 4, 8)  # 258 * 255 > 65535


def test_range_is_global_min_max():
    xs = [np.random.default_rng([53, w]).standard_normal(999).astype(np.float32) * (w + 1) for w in range(6)]
    m, M = oracle.thc_range(xs)
    allv = np.concatenate(xs)
    assert m == allv.min() and M == allv.max()
    xs[2][5] = np.nan
    m2, M2 = oracle.thc_range(xs)
    assert m2 == np.nanmin(np.concatenate(xs)) and M2 == np.nanmax(np.concatenate(xs))


def test_nmse_definition():
    x = np.random.default_rng(59).standard_normal(1000).astype(np.float32)
    xh = (x + np.random.default_rng(60).standard_normal(1000).astype(np.float32) * 0.1).astype(np.float32)
    ref = np.linalg.norm(x.astype(np.float64) - xh.astype(np.float64)) ** 2 / np.linalg.norm(x.astype(np.float64)) ** 2
    assert abs(oracle.nmse(x, xh) - ref) <= 1e-12 * ref
    assert oracle.nmse(x, x) == 0.0
    assert oracle.nmse(x, np.zeros_like(x)) == 1.0
    assert abs(oracle.nmse(x, (2 * x).astype(np.float32)) - 1.0) < 1e-15
    assert math.isnan(oracle.nmse(np.zeros(4, np.float32), np.ones(4, np.float32)))


def test_masked_round_all_arrived_is_the_full_round():
    P, N, b = 6, 777, 4
    xs = [np.random.default_rng([151, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    full, pk_full = oracle.thc_allreduce(xs, b, 3, m, M, want_packed=True)
    masked, pk_m = oracle.thc_allreduce_masked(xs, (1 << P) - 1, b, 3, m, M, want_packed=True)
    np.testing.assert_array_equal(full, masked)
    for a, c in zip(pk_full, pk_m):
        np.testing.assert_array_equal(a, c)


def test_masked_round_keeps_worker_ids_and_divides_by_arrivals():
    # stragglers 1 and 4 dropped: the others are encoded with their own ids
    # (not renumbered) and the decode divides by the 4 that arrived
    P, N, b = 6, 500, 4
    xs = [np.random.default_rng([152, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    arrived = 0b101101
    avg, pk = oracle.thc_allreduce_masked(xs, arrived, b, 11, m, M, want_packed=True)
    ids = [w for w in range(P) if (arrived >> w) & 1]
    for w in ids:
        np.testing.assert_array_equal(pk[w], oracle.thc_encode(xs[w], m, M, b, 11, w))
    idx = np.sum([oracle.thc_unpack(pk[w], N, b).astype(np.int64) for w in ids], axis=0)
    np.testing.assert_allclose(avg, oracle.thc_decode(idx.astype(np.uint16), m, M, b, len(ids)), rtol=0, atol=0)
    # a single arrival decodes to that worker's own quantized values
    one = oracle.thc_allreduce_masked(xs, 1 << 3, b, 11, m, M)
    q = oracle.thc_unpack(oracle.thc_encode(xs[3], m, M, b, 11, 3), N, b)
    np.testing.assert_allclose(one, oracle.thc_decode(q.astype(np.uint16), m, M, b, 1), rtol=0, atol=0)


def test_masked_round_unbiased_for_the_arrived_mean():
    P, N, b = 5, 64, 2
    xs = [np.random.default_rng([153, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    arrived = 0b10110
    ids = [w for w in range(P) if (arrived >> w) & 1]
    target = np.mean(np.stack([xs[w] for w in ids]).astype(np.float64), axis=0)
    K = 1500
    acc = np.zeros(N)
    for seed in range(K):
        acc += oracle.thc_allreduce_masked(xs, arrived, b, seed, m, M)
    step = (float(M) - float(m)) / 3
    sigma = math.sqrt(step ** 2 / (4 * len(ids)) / K)
    assert np.all(np.abs(acc / K - target) <= 5.5 * sigma + _bias_bound(m, M, b))


def test_samples_match_full_round():
    P, N, b = 5, 3001, 4
    xs = [np.random.default_rng([73, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    m, M = oracle.thc_range(xs)
    avg, packed = oracle.thc_allreduce(xs, b, 17, m, M, want_packed=True)
    idx = np.array([0, 3, 4, 1500, 2999, 3000], np.int64)
    ind, savg = oracle.thc_allreduce_samples(np.stack([x[idx] for x in xs]), idx, b, 17, m, M)
    np.testing.assert_array_equal(savg, avg[idx])
    for w in range(P):
        np.testing.assert_array_equal(ind[w], oracle.thc_unpack(packed[w], N, b)[idx])
