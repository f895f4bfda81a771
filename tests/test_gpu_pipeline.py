"""The benchmarked step itself against the oracle, element by element.

The bucketed averaging step (gradient_allreduce_homomorphic_gb300.pipeline)
runs the ResNet-101-like Tensor Fusion workload -- P = 8 workers, 300 fp32
tensors, 45M parameters each, 64 MB fusion buffers, THC b = 4 -- in the
schedule the benchmark times: the ring all-reduce of each fusion buffer on
one stream, THC of buffer b on a second stream behind an event on the ring
of buffer b, the NMSE after both ([R] "8. Compute-Communication Overlapping
& Gradient Bucketing"; [H] "Tensor Fusion").

Two steps run back to back with no host synchronisation between them; the
inputs change between the steps (copied in on the caller's stream), and
each step's results are snapshotted on the caller's stream right behind
it.  A missing or misplaced event -- THC reading a stale range, the NMSE
reading a half-written average, a step's ring overwriting what the previous
step's THC still reads -- changes a snapshot, which is compared with the
oracle for every tensor of every worker:

* the ring averages, bit for bit (pack -> ring fold -> unpack, [R] section 7);
* each fusion buffer's [m, M], exactly;
* every worker's wire words, bit for bit ([T] section 4, Algorithm 1);
* the THC average, within 1e-6 * max(|m|, |M|) of the oracle's fp64 decode;
* the NMSE, within 2e-6 of the oracle's fp64 NMSE of the same averages.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, to_host
from oracle_par import fusion_step

pytestmark = pytest.mark.gpu

P, B, CAP, ALIGN = 8, 4, 64 << 20, 16


def _inputs(torch, offs, seed_base):
    return [workloads.device_normal(int(offs[-1]), 0.01, seed_base + w, torch.float32, "cuda") for w in range(P)]


def _snapshot(st):
    return {"ring": [f.clone() for f in st.ring_flat], "thc": st.thc_flat.clone(), "mM": st.mM.clone(),
            "packed": [[t.clone() for t in row] for row in st.packed], "nmse": st.nmse.clone()}


@pytest.fixture(scope="module")
def steps():
    torch, g = need_cuda()
    from gradient_allreduce_homomorphic_gb300 import pipeline

    sizes = workloads.resnet_fusion_sizes()
    offs = pipeline.flat_offsets(sizes)
    cfg = workloads.CONFIG_IDS["resnet_fusion"]
    first = _inputs(torch, offs, 1000 * cfg)
    second = _inputs(torch, offs, 1000 * cfg + 500)
    grads = [t.clone() for t in first]
    seeds = (workloads.THC_SEED, workloads.THC_SEED + 1)
    out = {}
    for mode in ("separate", "fused"):
        st = pipeline.AveragingStep(grads, sizes, offs, b=B, capacity_bytes=CAP, align_bytes=ALIGN, nmse=mode)
        for w in range(P):
            grads[w].copy_(first[w])
        st.run(seeds[0])
        snap1 = _snapshot(st)
        for w in range(P):  # new gradients, on the caller's stream, before the next step
            grads[w].copy_(second[w])
        st.run(seeds[1])
        snap2 = _snapshot(st)
        torch.cuda.synchronize()
        out[mode] = (st, snap1, snap2)
    hosts = []
    for inp in (first, second):
        flat = [to_host(t) for t in inp]
        hosts.append([[f[int(offs[i]):int(offs[i]) + int(s)] for i, s in enumerate(sizes)] for f in flat])
    refs = [fusion_step(h, sizes, CAP, ALIGN, B, s) for h, s in zip(hosts, seeds)]
    return torch, sizes, offs, out, refs


def _check(sizes, offs, snap, ref, workers=P):
    sb, so, bn, per = ref
    flat_len = int(offs[-1])
    ring = np.zeros(flat_len, np.float32)
    for k in range(len(bn)):
        outs = oracle.fusion_unpack(per[k]["ring"], sb, so, sizes, k)
        for i, o in enumerate(outs):
            if o is not None:
                ring[int(offs[i]):int(offs[i]) + int(sizes[i])] = o
    for w in range(workers):  # every worker's copy of the exact average, bit for bit
        got = to_host(snap["ring"][w])
        bad = np.nonzero(got.view(np.uint32) != ring.view(np.uint32))[0]
        assert bad.size == 0, f"worker {w}: {bad.size} ring values differ, first at flat {bad[0]}"
    mM = to_host(snap["mM"])
    thc = to_host(snap["thc"]).astype(np.float64)
    for k in range(len(bn)):
        m, M = per[k]["mM"]
        assert (mM[k, 0], mM[k, 1]) == (m, M), f"buffer {k} range"
        for w in range(workers):
            words = to_host(snap["packed"][w][k])[: per[k]["packed"][w].size]
            np.testing.assert_array_equal(words, per[k]["packed"][w], err_msg=f"buffer {k} worker {w} wire words")
        tol = 1e-6 * max(abs(float(m)), abs(float(M)))
        for i in np.nonzero(sb == k)[0]:
            lo = int(offs[i])
            ref = per[k]["thc"][int(so[i]):int(so[i]) + int(sizes[i])]
            err = np.max(np.abs(thc[lo:lo + int(sizes[i])] - ref), initial=0.0)
            assert err <= tol, f"tensor {i} (buffer {k}): THC average off by {err} > {tol}"
    # the NMSE the step reports, against the oracle's NMSE of the same two
    # averages (flat buffers, padding zero in both)
    ref_nmse = oracle.nmse(ring, to_host(snap["thc"]))
    got = float(to_host(snap["nmse"])[0])
    assert abs(got - ref_nmse) <= 2e-6 * ref_nmse, (got, ref_nmse)
    # and close to the NMSE of the oracle's own compressed average
    own = np.zeros(flat_len, np.float32)
    for k in range(len(bn)):
        for i in np.nonzero(sb == k)[0]:
            own[int(offs[i]):int(offs[i]) + int(sizes[i])] = per[k]["thc"][int(so[i]):int(so[i]) + int(sizes[i])]
    assert abs(oracle.nmse(ring, own) - ref_nmse) <= 1e-4 * ref_nmse


@pytest.mark.parametrize("mode", ["separate", "fused"])
@pytest.mark.parametrize("step", [0, 1])
def test_bench_step_matches_oracle(steps, mode, step):
    torch, sizes, offs, out, refs = steps
    st, snap1, snap2 = out[mode]
    _check(sizes, offs, (snap1, snap2)[step], refs[step])


def test_bench_step_launch_count(steps):
    """One step launches, per fusion buffer, a range reset, a ring fold and a
    THC kernel, then the NMSE's two kernels (separate mode)."""
    torch, sizes, offs, out, refs = steps
    import gradient_allreduce_homomorphic_gb300 as g

    st = out["separate"][0]
    n0 = g.gar_launch_count()
    st.run(123)
    torch.cuda.synchronize()
    assert g.gar_launch_count() - n0 == 3 * st.nb + 2


def test_bench_step_from_host(steps):
    """The end-to-end form of the step (pinned host gradients in, both
    averages and the NMSE out, pipelined by bucket on copy streams) gives the
    device-resident step's results."""
    torch, sizes, offs, out, refs = steps
    st, snap1, snap2 = out["separate"]
    host_in = [torch.empty(st.flat_len, dtype=torch.float32, pin_memory=True) for _ in range(P)]
    for w in range(P):
        host_in[w].copy_(st.flat[w])  # the second step's gradients
    host_ring = torch.zeros(st.flat_len, dtype=torch.float32, pin_memory=True)
    host_thc = torch.zeros(st.flat_len, dtype=torch.float32, pin_memory=True)
    host_nmse = torch.zeros(1, dtype=torch.float64, pin_memory=True)
    for w in range(P):  # the device copies must come from the host
        st.flat[w].zero_()
    st.setup_host()
    st.host_begin()
    st.run_from_host(workloads.THC_SEED + 7, host_in, host_ring, host_thc, host_nmse)
    st.run_from_host(workloads.THC_SEED + 1, host_in, host_ring, host_thc, host_nmse)
    st.host_end()
    torch.cuda.synchronize()
    assert np.array_equal(host_ring.numpy().view(np.uint32), to_host(snap2["ring"][0]).view(np.uint32))
    assert np.array_equal(host_thc.numpy().view(np.uint32), to_host(snap2["thc"]).view(np.uint32))
    assert host_nmse.numpy()[0] == float(to_host(snap2["nmse"])[0])


@pytest.mark.parametrize("P_,b,mode", [(3, 2, "separate"), (5, 8, "fused"), (1, 4, "fused")])
def test_small_step_other_worker_counts(P_, b, mode):
    """The bucketed step with worker counts that take the any-P kernel builds
    (and one worker), small fusion buffers (many buckets), against the oracle."""
    torch, g = need_cuda()
    from gradient_allreduce_homomorphic_gb300 import pipeline

    sizes = np.array([1, 4096, 77, 3000, 5, 20000, 12345, 2], np.int64)
    offs = pipeline.flat_offsets(sizes)
    host_flat = [np.random.default_rng([211, P_, w]).standard_normal(int(offs[-1])).astype(np.float32)
                 for w in range(P_)]
    grads = [torch.from_numpy(f).cuda() for f in host_flat]
    cap = 32 << 10
    st = pipeline.AveragingStep(grads, sizes, offs, b=b, capacity_bytes=cap, align_bytes=16, nmse=mode)
    assert st.nb > 2
    seed = 0x5EED + P_
    st.run(seed)
    st.run(seed)  # twice: the second step must give the same results
    torch.cuda.synchronize()
    host = [[f[int(offs[i]):int(offs[i]) + int(s)] for i, s in enumerate(sizes)] for f in host_flat]
    ref = fusion_step(host, sizes, cap, 16, b, seed)
    _check(sizes, offs, _snapshot(st), ref, workers=P_)
