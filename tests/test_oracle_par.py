"""The threaded helpers that run the oracle over full-size inputs give what
the oracle's whole-vector functions give, at sizes cut into many runs."""
import numpy as np

import oracle
from oracle_par import (bidir_fold_range_bf16, dbtree_fold_range, fusion_step, ring_fold_range, runs,
                        thc_range_parallel, thc_range_samples)


def _xs(P, N, seed):
    return [np.random.default_rng([seed, w]).standard_normal(N).astype(np.float32) for w in range(P)]


def test_runs_cover_exactly():
    for lo, hi, k in [(0, 10, 3), (5, 6, 4), (0, 1000, 64), (7, 7, 3)]:
        r = runs(lo, hi, k)
        assert sum(b - a for a, b in r) == hi - lo
        assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))


def test_folds_in_pieces_equal_whole_folds():
    P, N = 5, 10007
    xs = _xs(P, N, 1)
    whole = oracle.ring_fold(xs)
    lo = 3001
    np.testing.assert_array_equal(ring_fold_range(np.stack([x[lo:] for x in xs]), N, lo, threads=7), whole[lo:])
    tree = oracle.dbtree_fold(xs)
    np.testing.assert_array_equal(dbtree_fold_range(np.stack([x[:5000] for x in xs]), N, 0, threads=3), tree[:5000])
    bf = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in xs]
    wide = [(b.astype(np.uint32) << 16).view(np.float32) for b in bf]
    ref = oracle.f32_to_bf16_array(oracle.bidir_fold(wide))
    np.testing.assert_array_equal(bidir_fold_range_bf16(np.stack(bf), N, 0, threads=4), ref)


def test_thc_in_pieces_equals_whole_round():
    P, N, b, seed = 4, 4099, 4, 77
    xs = _xs(P, N, 2)
    m, M = oracle.thc_range(xs)
    assert thc_range_parallel(xs, threads=5) == (m, M)
    avg, packed = oracle.thc_allreduce(xs, b, seed, m, M, want_packed=True)
    lo = 32 * 17
    ind, got = thc_range_samples(np.stack([x[lo:] for x in xs]), lo, b, seed, m, M, threads=6)
    np.testing.assert_array_equal(got, avg[lo:])
    for w in range(P):
        np.testing.assert_array_equal(ind[w], oracle.thc_unpack(packed[w], N, b)[lo:])


def test_fusion_step_per_buffer():
    P, b, seed = 3, 4, 5
    sizes = np.array([100, 3000, 7, 2500, 999], np.int64)
    host = [[np.random.default_rng([3, w, i]).standard_normal(int(s)).astype(np.float32) for i, s in enumerate(sizes)]
            for w in range(P)]
    sb, so, bn, per = fusion_step(host, sizes, 16 << 10, 16, b, seed)
    assert len(per) == len(bn) > 1
    for k in range(len(bn)):
        bufs = [oracle.fusion_pack(host[w], sb, so, k, bn[k]) for w in range(P)]
        np.testing.assert_array_equal(per[k]["ring"], oracle.ring_fold(bufs))
        assert per[k]["mM"] == oracle.thc_range(bufs)
        np.testing.assert_array_equal(per[k]["thc"], oracle.thc_allreduce(bufs, b, seed, *per[k]["mM"]))
