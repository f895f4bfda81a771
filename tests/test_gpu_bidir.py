"""GPU parity of the bidirectional dual ring against the oracle (bit-exact).

fp32 against the oracle's two-ring fold (itself equal to its literal
schedule), bf16 against the same fold on the exactly widened inputs rounded
to bf16, the hand-derived ordering example, ragged and degenerate sizes,
P up to 64 (128 sub-chunks), and the full-size bf16 bucket (P=16, 2^28
elements per worker) on every element.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from oracle_par import bidir_fold_range_bf16
from helpers import bf16_bits, need_cuda, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _xs(P, N, seed):
    return [(np.random.default_rng([seed, P, N, w]).standard_normal(N) * 10.0 ** (w % 3)).astype(np.float32)
            for w in range(P)]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 33, 64])
@pytest.mark.parametrize("N", [0, 1, 7, 130, 4099, 65541])
def test_bidir_f32(env, P, N):
    torch, g = env
    xs = _xs(P, N, 141)
    for op in (g.GAR_SUM, g.GAR_AVG):
        bufs = [to_dev(x, torch) for x in xs]
        g.gar_ring_allreduce_bidir(bufs, op=op)
        ref = oracle.bidir_fold(xs, op=op)
        for b in bufs:
            same_bits(to_host(b), ref)


def test_bidir_brute_force_small(env):
    torch, g = env
    for P in range(1, 5):
        for N in range(0, 65):
            xs = _xs(P, N, 142)
            bufs = [to_dev(x, torch) for x in xs]
            g.gar_ring_allreduce_bidir(bufs, op=g.GAR_AVG)
            ref = oracle.bidir_fold(xs, op=oracle.AVG)
            for b in bufs:
                same_bits(to_host(b), ref)


@pytest.mark.parametrize("P,N", [(3, 50), (8, 10001), (16, 70003)])
def test_bidir_bf16(env, P, N):
    torch, g = env
    hs = [bf16_bits((x * 0.01).astype(np.float32), torch) for x in _xs(P, N, 143)]
    wide = [(h.astype(np.uint32) << 16).view(np.float32) for h in hs]  # exact widening
    ref32 = oracle.bidir_fold(wide, op=oracle.AVG)
    ref = np.array([oracle.f32_to_bf16(v) for v in ref32], np.uint16)
    bufs = [to_dev(h, torch) for h in hs]
    g.gar_ring_allreduce_bidir(bufs, op=g.GAR_AVG)
    for b in bufs:
        same_bits(to_host(b), ref)


def test_bidir_order_golden(env, golden_dir):
    torch, g = env
    d = json.load(open(os.path.join(golden_dir, "bidir_order_p3.json")))
    bufs = [torch.full((d["N"],), v, dtype=torch.float32, device="cuda") for v in d["worker_values"]]
    g.gar_ring_allreduce_bidir(bufs, op=g.GAR_SUM)
    for b in bufs:
        assert to_host(b).tolist() == d["sum"]


def test_bidir_large_bf16_full_size(env):
    # P=16, N = 2^28 bf16 per worker, in place: every element against the
    # oracle's two-ring fold (worker 0 on the host, every other worker equal
    # to worker 0 on the device)
    torch, g = env
    P, N = 16, 1 << 28
    bufs = [workloads.device_normal(N, 1e-2, 6000 + w, torch.bfloat16, "cuda") for w in range(P)]
    host = [to_host(b) for b in bufs]
    g.gar_ring_allreduce_bidir(bufs, op=g.GAR_AVG)
    torch.cuda.synchronize()
    for w in range(1, P):
        assert torch.equal(bufs[w].view(torch.int16), bufs[0].view(torch.int16)), f"worker {w} differs from 0"
    chunk = 1 << 24
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        ref = bidir_fold_range_bf16(np.stack([h[lo:hi] for h in host]), N, lo, op=oracle.AVG)
        same_bits(to_host(bufs[0][lo:hi]), ref)
    del bufs
    torch.cuda.empty_cache()
