"""Guard bands and the timeline.

Guard bands: every output a kernel writes lies inside a larger buffer whose
other words hold a canary pattern; after the call the canaries must be intact
(no kernel writes past either end of its outputs), across ragged sizes and
unaligned starts.  The timeline: with GAR_TIMELINE set, the library's device
calls are recorded as Chrome trace events named after the entry points.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads
from helpers import need_cuda

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CANARY = 0x7FC0DEAD  # a NaN pattern no kernel produces
G = 67               # guard words before and after each output


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _guarded(torch, n, dtype, off):
    """A view of n elements with G words of canary on each side, starting off
    elements into the storage (so it may be unaligned)."""
    es = torch.tensor([], dtype=dtype).element_size()
    words = ((G * 4 + off * es + n * es + G * 4) + 3) // 4
    store = torch.full((words,), CANARY, dtype=torch.int32, device="cuda")
    first = (G * 4) // es + off
    return store, store.view(dtype)[first:first + n]


def _intact(store, view, torch):
    """The canary words outside the view are unchanged."""
    es = view.element_size()
    base = store.data_ptr()
    lo = (view.data_ptr() - base) // 4
    hi = (view.data_ptr() - base + view.numel() * es + 3) // 4
    s = store.cpu().numpy()
    assert np.all(s[:lo] == CANARY), "written before the output"
    assert np.all(s[hi:] == CANARY), "written after the output"


@pytest.mark.parametrize("N,off", [(1, 0), (7, 1), (4099, 0), (4101, 3), (70001, 2)])
def test_guards_ring_thc_nmse(env, N, off):
    torch, g = env
    P = 5
    xs = [workloads.device_normal(N, 1.0, 900 + w, torch.float32, "cuda") for w in range(P)]
    # ring all-reduce into one output
    st, out = _guarded(torch, N, torch.float32, off)
    g.gar_ring_allreduce_sim_out(xs, [out])
    # THC range, encode, aggregate, decode, fused
    smM, mM = _guarded(torch, 2, torch.float32, 0)
    g.gar_thc_range(xs, mM)
    b = 4
    words = g.gar_thc_words(N, b)
    pk = [_guarded(torch, words, torch.int32, off) for _ in range(P)]
    for w in range(P):
        g.gar_thc_encode(xs[w], mM, b, 11, w, pk[w][1])
    ssum, sums = _guarded(torch, N, torch.int16, off)
    g.gar_thc_aggregate([p[1] for p in pk], N, b, sums)
    savg, avg = _guarded(torch, N, torch.float32, off)
    g.gar_thc_decode(sums, mM, b, P, avg)
    sfa, favg = _guarded(torch, N, torch.float32, off)
    fpk = [_guarded(torch, words, torch.int32, off) for _ in range(P)]
    g.gar_thc_allreduce_fused(xs, b, 11, mM, favg, [p[1] for p in fpk])
    snm, nm = _guarded(torch, 1, torch.float64, 0)
    ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8 + 1, dtype=torch.float64, device="cuda")
    g.gar_nmse(out, favg, nm, ws)
    torch.cuda.synchronize()
    for s_, v_ in [(st, out), (smM, mM), (ssum, sums), (savg, avg), (sfa, favg), (snm, nm)] + pk + fpk:
        _intact(s_, v_, torch)


def test_guards_fused_plan_paths(env):
    """Fused all-reduce and plan-driven THC writing into guarded tensors of
    ragged sizes, some unaligned: nothing outside any tensor changes."""
    torch, g = env
    P, b = 3, 4
    sizes = np.array([1, 5, 4099, 3, 1000, 2, 7001], np.int64)
    dt = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, 16 << 10, 4)
    src = [[workloads.device_normal(int(n), 1.0, 950 + 10 * w + i, torch.float32, "cuda")
            for i, n in enumerate(sizes)] for w in range(P)]
    dst_g = [[_guarded(torch, int(n), torch.float32, i % 3) for i, n in enumerate(sizes)] for _ in range(P)]
    g.gar_fused_allreduce(src, [[v for _, v in row] for row in dst_g], plan)
    mM = torch.empty((plan.n_buffers, 2), device="cuda")
    ring_g = [[_guarded(torch, int(n), torch.float32, 0) for n in sizes] for _ in range(P)]
    g.gar_fused_allreduce_range(src, [[v for _, v in row] for row in ring_g], plan, mM)
    out_g = [_guarded(torch, int(n), torch.float32, (i + 1) % 3) for i, n in enumerate(sizes)]
    pk_g = [[_guarded(torch, g.gar_thc_words(int(n), b), torch.int32, 0) for n in plan.buf_numel] for _ in range(P)]
    g.gar_thc_allreduce_fused_plan(src, plan, b, 3, mM, [v for _, v in out_g], [[v for _, v in row] for row in pk_g])
    torch.cuda.synchronize()
    for row in dst_g + ring_g + pk_g:
        for s_, v_ in row:
            _intact(s_, v_, torch)
    for s_, v_ in out_g:
        _intact(s_, v_, torch)


def test_timeline_records_device_calls(tmp_path):
    path = tmp_path / "trace.json"
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import torch, gradient_allreduce_homomorphic_gb300 as g\n"
        "x = [torch.randn(100000, device='cuda') for _ in range(4)]\n"
        "out = torch.empty(100000, device='cuda')\n"
        "mM = torch.empty(2, device='cuda')\n"
        "s = torch.cuda.Stream()\n"
        "g.gar_ring_allreduce_sim_out(x, [out])\n"
        "g.gar_thc_range(x, mM, stream=s)\n"
        "g.gar_thc_words(100000, 4)\n"
        "assert g.timeline() is not None\n" % ROOT)
    env = dict(os.environ, GAR_TIMELINE=str(path))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    ev = json.load(open(path))["traceEvents"]
    assert [e["name"] for e in ev] == ["gar_ring_allreduce_sim_out", "gar_thc_range"]
    assert all(e["ph"] == "X" and e["dur"] > 0 for e in ev)
    assert ev[0]["tid"] != ev[1]["tid"]  # two streams, two tracks
