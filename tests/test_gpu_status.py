"""The device status word (gar_sync_status): non-finite inputs seen by a THC
range pass raise GAR_STATUS_NONFINITE; finite inputs leave the word at 0; the
word clears on request.  Covered: gar_thc_range, gar_fusion_pack_all with a
range and gar_fused_allreduce_range, NaN and infinities, vector and
element-by-element paths; the range results themselves are unchanged (NaN
skipped, infinities taken in)."""
import numpy as np
import pytest

import oracle
from helpers import need_cuda, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch, g = need_cuda()
    g.gar_sync_status()  # start from a clear word
    return torch, g


def _xs(P, N, seed):
    return [np.random.default_rng([seed, P, N, w]).standard_normal(N).astype(np.float32) for w in range(P)]


def test_finite_inputs_leave_status_clear(env):
    torch, g = env
    xs = [to_dev(x, torch) for x in _xs(4, 100003, 1)]
    mM = torch.empty(2, device="cuda")
    g.gar_thc_range(xs, mM)
    assert g.gar_sync_status() == 0


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
@pytest.mark.parametrize("where", [0, 77, 100002])
def test_thc_range_flags_nonfinite(env, bad, where):
    torch, g = env
    hx = _xs(3, 100003, 2)
    hx[1][where] = bad
    mM = torch.empty(2, device="cuda")
    g.gar_thc_range([to_dev(x, torch) for x in hx], mM)
    assert g.gar_sync_status() & g.GAR_STATUS_NONFINITE
    m, M = oracle.thc_range(hx)  # the range itself as before: NaN skipped, infinities in
    hm = to_host(mM)
    assert hm[0] == m and hm[1] == M
    assert g.gar_sync_status() == 0  # cleared by the first read


def test_status_unaligned_path_and_no_clear(env):
    torch, g = env
    hx = _xs(2, 5001, 3)
    hx[0][4999] = np.nan
    bases = [to_dev(np.concatenate([[0.0], x]).astype(np.float32), torch) for x in hx]
    mM = torch.empty(2, device="cuda")
    g.gar_thc_range([b[1:] for b in bases], mM)  # 4-byte offset: element by element
    assert g.gar_sync_status(clear=False) & g.GAR_STATUS_NONFINITE
    assert g.gar_sync_status(clear=True) & g.GAR_STATUS_NONFINITE
    assert g.gar_sync_status() == 0


def _plan(g, sizes):
    return g.gar_fusion_plan(np.asarray(sizes, np.int64), np.zeros(len(sizes), np.int32), 1 << 16, 16)


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_fusion_range_passes_flag_nonfinite(env, bad):
    torch, g = env
    P = 4
    sizes = [1000, 3, 40000, 17, 9000]
    rng = np.random.default_rng(4)
    host = [[rng.standard_normal(s).astype(np.float32) for s in sizes] for _ in range(P)]
    plan = _plan(g, sizes)
    for which in ("pack_all", "fused_range"):
        for poison in (False, True):
            hx = [[t.copy() for t in w] for w in host]
            if poison:
                hx[2][2][123] = bad
            src = [[to_dev(t, torch) for t in w] for w in hx]
            mM = torch.empty(2 * plan.n_buffers, device="cuda")
            if which == "pack_all":
                fbs = [[torch.empty(int(n), device="cuda") for n in plan.buf_numel] for _ in range(P)]
                g.gar_fusion_pack_all(src, plan, fbs, d_mM=mM)
            else:
                dst = [[torch.empty_like(t) for t in w] for w in src]
                g.gar_fused_allreduce_range(src, dst, plan, mM)
            got = g.gar_sync_status()
            assert bool(got & g.GAR_STATUS_NONFINITE) == poison, (which, poison, got)
