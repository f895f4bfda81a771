"""GPU parity of the ring all-reduce against the oracle (bit-exact).

Through the C ABI: in-place (all-gather to every worker), out-of-place (one
or P outputs), the literal 2(P-1)-step schedule, fp32 and bf16, ragged and
degenerate sizes, unaligned buffers, and the full-size configurations
(P=4 x 2^20 fp32; P=16 x 2^28 bf16), every element against the oracle.
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle_par import ring_fold_range
from helpers import bf16_bits, need_cuda, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _inputs(P, N, seed, scale=1.0):
    return [(np.random.default_rng([seed, P, N, w]).standard_normal(N).astype(np.float32) * scale *
             np.float32(10.0 ** (w % 3))) for w in range(P)]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 64])
@pytest.mark.parametrize("N", [0, 1, 7, 64, 1000, 4099, 65539])
def test_ring_f32_in_place(env, P, N):
    torch, g = env
    xs = _inputs(P, N, 1)
    for op in (g.GAR_SUM, g.GAR_AVG):
        bufs = [to_dev(x, torch) for x in xs]
        g.gar_ring_allreduce_sim(bufs, op=op)
        ref = oracle.ring_fold(xs, op=op)
        for b in bufs:
            same_bits(to_host(b), ref)


def test_ring_f32_brute_force_small(env):
    torch, g = env
    for P in range(1, 5):
        for N in range(0, 65):
            xs = _inputs(P, N, 2)
            bufs = [to_dev(x, torch) for x in xs]
            g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
            ref = oracle.ring_fold(xs, op=oracle.AVG)
            for b in bufs:
                same_bits(to_host(b), ref)


@pytest.mark.parametrize("P,N", [(2, 17), (3, 1000), (4, 4101), (16, 70001), (64, 9999), (5, 1 << 16)])
def test_ring_bf16(env, P, N):
    torch, g = env
    xs = [bf16_bits(x, torch) for x in _inputs(P, N, 3, 0.1)]
    for op in (g.GAR_SUM, g.GAR_AVG):
        bufs = [to_dev(x, torch) for x in xs]
        g.gar_ring_allreduce_sim(bufs, op=op)
        ref = oracle.ring_fold(xs, op=op)
        for b in bufs:
            same_bits(to_host(b), ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_out", [1, "P"])
def test_ring_out_of_place(env, dtype, n_out):
    torch, g = env
    P, N = 6, 12345
    xs = _inputs(P, N, 4)
    if dtype == "bf16":
        xs = [bf16_bits(x, torch) for x in xs]
    bufs = [to_dev(x, torch) for x in xs]
    k = P if n_out == "P" else 1
    outs = [torch.empty_like(bufs[0]) for _ in range(k)]
    g.gar_ring_allreduce_sim_out(bufs, outs, op=g.GAR_AVG)
    ref = oracle.ring_fold(xs, op=oracle.AVG)
    for o in outs:
        same_bits(to_host(o), ref)
    for b, x in zip(bufs, xs):  # inputs untouched
        same_bits(to_host(b), x)


@pytest.mark.parametrize("P,N", [(1, 10), (2, 9), (3, 3), (4, 8), (4, 10), (5, 3), (7, 1001), (16, 4096)])
def test_literal_schedule(env, P, N):
    torch, g = env
    xs = _inputs(P, N, 5)
    for op in (g.GAR_SUM, g.GAR_AVG):
        bufs = [to_dev(x, torch) for x in xs]
        steps, sent = g.gar_ring_allreduce_steps(bufs, op=op)
        host = [x.copy() for x in xs]
        ref_steps, ref_sent = oracle.ring_schedule(host, op=op)
        assert steps == ref_steps == 2 * (P - 1)
        np.testing.assert_array_equal(sent, ref_sent)
        for b, h in zip(bufs, host):
            same_bits(to_host(b), h)
        # the one-pass fold gives the same bits as the literal schedule
        fold = [to_dev(x, torch) for x in xs]
        g.gar_ring_allreduce_sim(fold, op=op)
        same_bits(to_host(fold[0]), to_host(bufs[0]))


def test_demo_golden(env, golden_dir):
    import json
    import os

    torch, g = env
    d = json.load(open(os.path.join(golden_dir, "ring_demo_p4_k8.json")))
    bufs = [torch.tensor(r, dtype=torch.float32, device="cuda") for r in d["inputs"]]
    steps, sent = g.gar_ring_allreduce_steps(bufs, op=g.GAR_SUM)
    assert steps == d["steps"] and all(int(s) * d["elem_bytes"] == d["bytes_sent_per_worker"] for s in sent)
    for b in bufs:
        assert to_host(b).tolist() == d["sum"]
    bufs = [torch.tensor(r, dtype=torch.float32, device="cuda") for r in d["inputs"]]
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
    for b in bufs:
        assert to_host(b).tolist() == d["avg"]


def test_order_golden(env, golden_dir):
    import json
    import os

    torch, g = env
    d = json.load(open(os.path.join(golden_dir, "ring_order_p3.json")))
    bufs = [torch.full((3,), v, dtype=torch.float32, device="cuda") for v in d["worker_values"]]
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_SUM)
    for b in bufs:
        assert to_host(b).tolist() == d["sum"]


def test_unaligned_buffers(env):
    torch, g = env
    P, N = 5, 10007
    xs = _inputs(P, N + 3, 6)
    for shift in (1, 2, 3):
        bases = [to_dev(x, torch) for x in xs]
        bufs = [b[shift:shift + N] for b in bases]  # 4-byte but not 16-byte aligned
        g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
        ref = oracle.ring_fold([x[shift:shift + N].copy() for x in xs], op=oracle.AVG)
        for b in bufs:
            same_bits(to_host(b), ref)
    hb = [bf16_bits(x, torch) for x in xs]
    bases = [to_dev(h, torch) for h in hb]
    bufs = [b[1:1 + N] for b in bases]
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
    same_bits(to_host(bufs[0]), oracle.ring_fold([h[1:1 + N].copy() for h in hb], op=oracle.AVG))


def test_special_values(env):
    torch, g = env
    P, N = 3, 64
    xs = _inputs(P, N, 7)
    xs[0][3] = np.inf
    xs[1][5] = -np.inf
    xs[2][5] = np.inf      # inf + -inf = NaN
    xs[1][9] = np.nan
    xs[0][11] = -0.0
    xs[1][11] = -0.0
    xs[2][11] = -0.0
    xs[0][13] = 3e38
    xs[1][13] = 3e38       # overflow to inf
    xs[2][20] = 1e-45      # subnormals
    xs[1][20] = 1e-45
    for op in (g.GAR_SUM, g.GAR_AVG):
        bufs = [to_dev(x, torch) for x in xs]
        g.gar_ring_allreduce_sim(bufs, op=op)
        same_bits(to_host(bufs[0]), oracle.ring_fold(xs, op=op))


def test_partition_4mb_full(env):
    # P=4 workers, one 4 MB partition each (N = 2^20 fp32), N(0, 1)
    torch, g = env
    P, N = 4, 1 << 20
    xs = workloads.workers_normal(P, N, 1.0, workloads.CONFIG_IDS["partition_4mb"])
    ref = oracle.ring_fold(xs, op=oracle.AVG)
    bufs = [to_dev(x, torch) for x in xs]
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
    for b in bufs:
        same_bits(to_host(b), ref)
    out = [torch.empty(N, dtype=torch.float32, device="cuda")]
    g.gar_ring_allreduce_sim_out([to_dev(x, torch) for x in xs], out, op=g.GAR_AVG)
    same_bits(to_host(out[0]), ref)


def test_large_bf16_full_size(env):
    # P=16 workers, N = 2^28 bf16 N(0, 1e-2) each (8 GiB): fp32 fold in ring
    # order, bf16 average out, in place (the launch the benchmark times);
    # every element against the oracle (worker 0 on the host, every other
    # worker equal to worker 0 on the device)
    torch, g = env
    P, N = 16, 1 << 28
    bufs = [workloads.device_normal(N, 1e-2, 5000 + w, torch.bfloat16, "cuda") for w in range(P)]
    host = [to_host(b) for b in bufs]  # the inputs, before the in-place call
    g.gar_ring_allreduce_sim(bufs, op=g.GAR_AVG)
    torch.cuda.synchronize()
    for w in range(1, P):
        assert torch.equal(bufs[w].view(torch.int16), bufs[0].view(torch.int16)), f"worker {w} differs from 0"
    chunk = 1 << 24
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        ref = ring_fold_range(np.stack([h[lo:hi] for h in host]), N, lo, op=oracle.AVG)
        same_bits(to_host(bufs[0][lo:hi]), ref)
    del bufs
    torch.cuda.empty_cache()
