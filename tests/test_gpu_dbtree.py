"""GPU parity of the double-binary-tree all-reduce against the oracle (bit-exact).

fp32 and bf16 against the oracle's two-tree fold (itself equal to its literal
reduce + broadcast schedule), the hand-derived P=4 fold expressions, every P
from 1 to 64, ragged sizes (the group that straddles the two halves, the
ragged last group), unaligned buffers (the element-wise path), and the
full-size bf16 bucket (P=16, 2^28 elements per worker) on every element.
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle_par import dbtree_fold_range
from helpers import bf16_bits, need_cuda, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _xs(P, N, seed):
    """Values over several binades, so that the association order shows."""
    out = []
    for w in range(P):
        r = np.random.default_rng([seed, P, N, w])
        out.append((r.standard_normal(N) * 10.0 ** r.uniform(-3, 3, N)).astype(np.float32))
    return out


def _run(g, torch, xs, op):
    bufs = [to_dev(x, torch) for x in xs]
    g.gar_dbtree_allreduce(bufs, op=op)
    return [to_host(b) for b in bufs]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 31, 33, 63, 64])
@pytest.mark.parametrize("N", [0, 1, 2, 7, 130, 4099, 65541])
def test_dbtree_f32(env, P, N):
    torch, g = env
    xs = _xs(P, N, 151)
    for op in (g.GAR_SUM, g.GAR_AVG):
        ref = oracle.dbtree_fold(xs, op=op)
        for h in _run(g, torch, xs, op):
            same_bits(h, ref)


def test_dbtree_every_p_and_small_n(env):
    torch, g = env
    for P in range(1, 65):
        for N in (3, 8, 9, 33):
            xs = _xs(P, N, 152)
            ref = oracle.dbtree_fold(xs, op=oracle.AVG)
            for h in _run(g, torch, xs, g.GAR_AVG):
                same_bits(h, ref)


def test_dbtree_p4_hand_expressions(env):
    """Tree 1: rank 3 on top of rank 1 (children 0, 2); tree 2 (the mirror):
    rank 0 on top of rank 2 (children 3, 1); written out by hand."""
    torch, g = env
    N = 10001
    x = _xs(4, N, 153)
    h = (N + 1) // 2
    t1 = x[3] + ((x[1] + x[0]) + x[2])
    t2 = x[0] + ((x[2] + x[3]) + x[1])
    want = np.concatenate([t1[:h], t2[h:]])
    for out in _run(g, torch, x, g.GAR_SUM):
        same_bits(out, want)


@pytest.mark.parametrize("P,N,off", [(3, 1001, 1), (8, 4099, 3), (16, 257, 2), (64, 515, 1)])
def test_dbtree_unaligned(env, P, N, off):
    """Buffers that start off a 16-byte boundary take the element-wise path."""
    torch, g = env
    xs = _xs(P, N, 154)
    bases = [torch.zeros(N + 8, dtype=torch.float32, device="cuda") for _ in range(P)]
    views = [b[off:off + N] for b in bases]
    for v, x in zip(views, xs):
        v.copy_(torch.from_numpy(x).cuda())
    g.gar_dbtree_allreduce(views, op=g.GAR_AVG)
    ref = oracle.dbtree_fold(xs, op=oracle.AVG)
    for b in bases:
        hb = to_host(b)
        same_bits(hb[off:off + N], ref)
        assert not hb[:off].any() and not hb[off + N:].any()  # nothing written outside


@pytest.mark.parametrize("P,N", [(1, 17), (3, 50), (8, 10001), (16, 70003), (64, 4097)])
def test_dbtree_bf16(env, P, N):
    torch, g = env
    hs = [bf16_bits((x * 0.01).astype(np.float32), torch) for x in _xs(P, N, 155)]
    for op in (g.GAR_SUM, g.GAR_AVG):
        ref = oracle.dbtree_fold(hs, op=op)
        bufs = [to_dev(h, torch) for h in hs]
        g.gar_dbtree_allreduce(bufs, op=op)
        for b in bufs:
            same_bits(to_host(b), ref)


def test_dbtree_f32_mid_size(env):
    torch, g = env
    P, N = 8, (1 << 22) + 5
    xs = _xs(P, N, 156)
    ref = oracle.dbtree_fold(xs, op=oracle.AVG)
    out = _run(g, torch, xs, g.GAR_AVG)
    for w in (0, 3, 7):
        same_bits(out[w], ref)


def test_dbtree_large_bf16_full_size(env):
    """P=16, N = 2^28 bf16 per worker, in place (the launch the benchmark
    times): every element against the oracle's two-tree fold (worker 0 on
    the host, every other worker equal to worker 0 on the device)."""
    torch, g = env
    P, N = 16, 1 << 28
    bufs = [workloads.device_normal(N, 1e-2, 6100 + w, torch.bfloat16, "cuda") for w in range(P)]
    host = [to_host(b) for b in bufs]
    g.gar_dbtree_allreduce(bufs, op=g.GAR_AVG)
    torch.cuda.synchronize()
    for w in range(1, P):
        assert torch.equal(bufs[w].view(torch.int16), bufs[0].view(torch.int16)), f"worker {w} differs from 0"
    chunk = 1 << 24
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        ref = dbtree_fold_range(np.stack([h[lo:hi] for h in host]), N, lo, op=oracle.AVG)
        same_bits(to_host(bufs[0][lo:hi]), ref)
    del bufs
    torch.cuda.empty_cache()


def test_dbtree_differs_from_ring(env):
    """The fold order is really another one: for these inputs the tree and
    the ring round differently somewhere."""
    torch, g = env
    xs = _xs(8, 4096, 158)
    tree = _run(g, torch, xs, g.GAR_SUM)[0]
    bufs = [to_dev(x, torch) for x in xs]
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_SUM)
    assert np.any(tree != to_host(bufs[0]))
