"""The benchmark's all-cores oracle timing (host only).

``bench.py`` times the CPU oracle on every host core by cutting the tensor
list into contiguous runs, one spawned process per run, each running the
unchanged oracle step over its run; the processes start together at a
barrier.  Checked here: the runs cover the list exactly once and about
evenly, and a two-process step on a small sample completes and reports a
positive wall time.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_slice_bounds_cover_the_list():
    sizes = workloads.resnet_fusion_sizes().astype(np.int64)
    for k in (1, 2, 3, 8, 16, 64):
        runs = bench._slice_bounds(sizes, k)
        assert runs[0][0] == 0 and runs[-1][1] == sizes.size
        assert all(a < b for a, b in runs)
        assert all(runs[i][1] == runs[i + 1][0] for i in range(len(runs) - 1))
        assert len(runs) <= k
        if k <= 16:  # no run holds more than its share plus one tensor
            share = sizes.sum() / k
            assert max(sizes[a:b].sum() for a, b in runs) <= share + sizes.max()


def test_slice_bounds_more_runs_than_tensors():
    sizes = np.array([5, 7, 9], np.int64)
    runs = bench._slice_bounds(sizes, 8)
    assert runs == [(0, 1), (1, 2), (2, 3)]


def test_parallel_oracle_two_processes():
    sizes = workloads.resnet_fusion_sizes()[:12]
    po = bench.ParallelOracle(sizes, 2)
    try:
        assert len(po.procs) == 2
        assert po.params == int(sizes.sum())
        assert po.step(3) > 0.0
        assert po.step(4) > 0.0
    finally:
        po.close()
    assert not any(p.is_alive() for p in po.procs)
