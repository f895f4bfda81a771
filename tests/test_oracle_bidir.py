"""Pins for the oracle's bidirectional dual ring (ring tutorial section 11, exercise 1).

The exercise asks for two things this checks directly: every worker ends
with the exact ground-truth sum (integer inputs), and the two rings do not
interfere.  Plus: the literal two-ring schedule equals the closed-form fold
bit for bit on every P <= 4, N <= 64; 2(P-1) steps with the single ring's
per-worker volume 2(P-1)/P N; the hand-derived ordering example that tells
the counter-clockwise half from a clockwise one.
"""
import json
import os

import numpy as np
import pytest

import oracle


def test_order_example(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "bidir_order_p3.json")))
    xs = [np.full(d["N"], v, np.float32) for v in d["worker_values"]]
    np.testing.assert_array_equal(oracle.bidir_fold(xs, op=oracle.SUM), np.array(d["sum"], np.float32))
    bufs = [x.copy() for x in xs]
    steps, _ = oracle.bidir_schedule(bufs, op=oracle.SUM)
    assert steps == d["steps"]
    for b in bufs:
        np.testing.assert_array_equal(b, np.array(d["sum"], np.float32))
    assert d["sum"] != d["sum_if_both_clockwise"]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 7, 8, 16])
def test_exact_ground_truth_and_volume(P):
    N = 2 * P * 37
    g = np.random.default_rng([131, P])
    ints = g.integers(-1000, 1000, size=(P, N))
    bufs = [row.astype(np.float32) for row in ints]
    steps, sent = oracle.bidir_schedule(bufs, op=oracle.SUM)
    assert steps == 2 * (P - 1)
    assert all(int(s) * P == 2 * (P - 1) * N for s in sent)
    for b in bufs:
        np.testing.assert_array_equal(b, ints.sum(0).astype(np.float32))


def test_brute_force_schedule_equals_fold():
    for P in range(1, 5):
        for N in range(0, 65):
            xs = [np.random.default_rng([132, P, N, w]).standard_normal(N).astype(np.float32) * 10 ** w
                  for w in range(P)]
            for op in (oracle.SUM, oracle.AVG):
                bufs = [x.copy() for x in xs]
                oracle.bidir_schedule(bufs, op=op)
                fold = oracle.bidir_fold(xs, op=op)
                for b in bufs:
                    np.testing.assert_array_equal(b.view(np.uint32), fold.view(np.uint32))


def test_samples_match_full_fold():
    P, N = 6, 5003
    xs = [np.random.default_rng([134, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    full = oracle.bidir_fold(xs, op=oracle.AVG)
    idx = np.array([0, 1, 416, 417, 2501, 2502, 5002], np.int64)
    np.testing.assert_array_equal(oracle.bidir_fold_samples(np.stack([x[idx] for x in xs]), N, idx), full[idx])


def test_first_half_is_the_single_ring():
    # the clockwise half folds exactly like the single ring on the same sub-chunks
    P, N = 4, 64
    xs = [np.random.default_rng([133, w]).standard_normal(N).astype(np.float32) for w in range(P)]
    bi = oracle.bidir_fold(xs, op=oracle.SUM)
    half = N // 2  # sub-chunks of 8: the clockwise half is elements 0..31, chunk c = e // 8
    single = oracle.ring_fold([x[:half].copy() for x in xs], op=oracle.SUM)
    np.testing.assert_array_equal(bi[:half], single)
