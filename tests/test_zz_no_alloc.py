"""The allocation-free NMSE entry point against the workspace one and the oracle.

gar_nmse_noalloc serves callers that cannot give the library a workspace
because they may not allocate device memory (a plug-in whose host framework
owns all of the device's memory, or a latency-critical path that must not
pay cudaMalloc's device-wide synchronisation).  Its partial sums live in a
fixed array inside the library that every call shares and that keeps the
previous call's contents, so the checks run calls in a row on different
inputs and sizes: a later call must not see anything left by an earlier one.
It runs the same kernels, grid and summation order as gar_nmse, so the two
must agree bit for bit; both are held to the oracle's fp64 NMSE within 2e-6.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
from helpers import need_cuda, to_dev

pytestmark = pytest.mark.gpu


def _pair(N, call):
    rng = np.random.default_rng([101, call, N])
    x = rng.standard_normal(N).astype(np.float32)
    xh = (x + rng.standard_normal(N).astype(np.float32) * np.float32(0.03 * (call + 1))).astype(np.float32)
    return x, xh


def _both(torch, g, x, xh, stream=None):
    N = x.size
    xd, xhd = to_dev(x, torch), to_dev(xh, torch)
    ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8 + 1, dtype=torch.float64, device="cuda")
    ref = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    out = torch.full((1,), -2.0, dtype=torch.float64, device="cuda")
    torch.cuda.synchronize()
    g.gar_nmse(xd, xhd, ref, ws, stream=stream)
    g.gar_nmse_noalloc(xd, xhd, out, stream=stream)
    torch.cuda.synchronize()
    return out.item(), ref.item()


def test_nmse_noalloc_matches_workspace_entry_point():
    torch, g = need_cuda()
    # large first, so that the later calls run over stale partial sums
    for call, N in enumerate((1 << 22, 4099, 1 << 20, 1)):
        x, xh = _pair(N, call)
        o, r = _both(torch, g, x, xh)
        assert o == r, (call, N, o, r)  # the same kernels and order: the same bits
        want = oracle.nmse(x, xh)
        assert abs(o - want) <= 2e-6 * want, (call, N, o, want)


def test_nmse_noalloc_on_a_side_stream_and_empty():
    torch, g = need_cuda()
    side = torch.cuda.Stream()
    x, xh = _pair(300_001, 7)
    o, r = _both(torch, g, x, xh, stream=side)
    assert o == r
    assert abs(o - oracle.nmse(x, xh)) <= 2e-6 * oracle.nmse(x, xh)
    # N = 0: 0 / 0, NaN from both entry points
    e = np.zeros(0, np.float32)
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    g.gar_nmse_noalloc(torch.zeros(1, device="cuda")[:0], torch.zeros(1, device="cuda")[:0], out)
    torch.cuda.synchronize()
    assert np.isnan(out.item()) and np.isnan(oracle.nmse(e, e))
