"""The allocation-free NMSE entry point against the workspace one.

gar_nmse_noalloc serves callers that cannot give the library a workspace
because they may not allocate device memory (a plug-in whose host framework
owns all of the device's memory, or a latency-critical path that must not
pay cudaMalloc's device-wide synchronisation).  Its partial sums live in a
fixed array inside the library that every call shares and that keeps the
previous call's contents, so the check runs two calls in a row on different
inputs and sizes: the second must not see anything left by the first.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from helpers import need_cuda, to_dev

pytestmark = pytest.mark.gpu


def test_nmse_noalloc_matches_workspace_entry_point():
    torch, g = need_cuda()
    for call, N in enumerate((1 << 20, 4099)):  # large first, so the second reuses stale partials
        rng = np.random.default_rng([101, call])
        x = rng.standard_normal(N).astype(np.float32)
        xh = (x + rng.standard_normal(N).astype(np.float32) * np.float32(0.03 * (call + 1))).astype(np.float32)
        xd, xhd = to_dev(x, torch), to_dev(xh, torch)
        ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8, dtype=torch.float64, device="cuda")
        ref = torch.empty(1, dtype=torch.float64, device="cuda")
        g.gar_nmse(xd, xhd, ref, ws)
        out = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
        g.gar_nmse_noalloc(xd, xhd, out)
        torch.cuda.synchronize()
        r, o = ref.item(), out.item()
        assert np.isfinite(o)
        assert abs(o - r) <= 2e-6 * r, (call, N, o, r)
