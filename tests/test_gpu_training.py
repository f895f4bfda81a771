"""THC's training step ([T] section 5) as gradient_allreduce_homomorphic_gb300
.training.TrainingStep runs it: the workers' error-feedback rotations and
updates spread over side streams.

* Any stream count gives the one-stream step's results bit for bit, over two
  steps in a row (the error vectors carry over): the rotated vectors, the
  range, every wire word, the average, its inverse rotation and every e.
* The step against the oracle: the rotated vectors within the rotation's
  bound of the oracle's fp64 rotation of grad + e; the range within 1e-6 of
  the oracle's norm-based range; every wire word bit-exact and the average
  within 1e-6 * M against the oracle's THC round over the GPU's own rotated
  vectors and range; the estimate within the rotation's bound of the
  oracle's inverse rotation of the GPU's average; each e against the
  oracle's fp32 update with the oracle's inverse rotation of the worker's
  own decoded vector.
Uniform (b = 2) and non-uniform (b = 4, g = 36) THC; n = 2^21 (2-CTA cluster
passes) and 2^16 (strided passes).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, to_host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
P = 4


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _table(b, g):
    return np.rint(np.linspace(0, g, (1 << b))).astype(np.uint16)


def _inputs(torch, n, k):
    grads = [torch.from_numpy(workloads.student_t_f32(n, 4, 1e-2, 601, k * 16 + w)).cuda() for w in range(P)]
    errs = [torch.from_numpy(workloads.normal_f32(n, 1e-6, 602, k * 16 + w)).cuda() for w in range(P)]
    return grads, errs


def _snapshot(st):
    ts = [st.mM, st.avg, st.est] + st.ys + st.packed + st.errs
    return [to_host(t).copy() for t in ts]


CASES = [(21, 4, 36), (21, 2, None), (16, 4, 36)]


@pytest.mark.parametrize("k,b,g", CASES)
def test_stream_counts_agree(env, k, b, g):
    torch, gar = env
    from gradient_allreduce_homomorphic_gb300.training import TrainingStep

    n = 1 << k
    table = _table(b, g) if g else None
    gar.gar_sync_status(clear=True)  # earlier tests may have left a bit set
    snaps = {}
    for streams in (1, 2, 3):
        grads, errs = _inputs(torch, n, k)
        st = TrainingStep(grads, errs, b=b, table=table, t_p=2.15, rht_seed=0xD1A6, streams=streams)
        out = []
        for seed in (0x5EED, 0x5EEE):
            st.run(seed)
            torch.cuda.synchronize()
            out.append(_snapshot(st))
        snaps[streams] = out
    for streams in (2, 3):
        for a, c in zip(snaps[1], snaps[streams]):
            for x, y in zip(a, c):
                assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), streams
    assert gar.gar_sync_status() == 0


@pytest.mark.parametrize("k,b,g", CASES)
def test_step_against_oracle(env, k, b, g):
    torch, gar = env
    from gradient_allreduce_homomorphic_gb300.training import TrainingStep

    n = 1 << k
    table = _table(b, g) if g else None
    steps = g if g else (1 << b) - 1
    grads, errs = _inputs(torch, n, k)
    gh = [to_host(t).copy() for t in grads]
    eh = [to_host(t).copy() for t in errs]
    st = TrainingStep(grads, errs, b=b, table=table, t_p=2.15, rht_seed=0xD1A6, streams=2)
    seed = 0x5EED
    st.run(seed)
    torch.cuda.synchronize()
    xs = [oracle.ef_apply(a, c) for a, c in zip(gh, eh)]
    bound = lambda v: (k + 2) * U * float(np.linalg.norm(np.asarray(v, np.float64))) * 1.0001 + 1e-30  # noqa: E731
    ys = [to_host(y).copy() for y in st.ys]
    for w in range(P):
        ref = oracle.rht(xs[w], 0xD1A6)
        assert np.linalg.norm(ys[w].astype(np.float64) - ref) <= bound(xs[w]), w
    m, M = (float(v) for v in to_host(st.mM))
    rm, rM = oracle.rht_norm_range(xs, 2.15)
    assert m == -M and abs(M - rM) <= 1e-6 * rM
    if table is None:
        ref_avg, ref_pk = oracle.thc_allreduce(ys, b, seed, np.float32(m), np.float32(M), want_packed=True)
    else:
        ref_avg, ref_pk = oracle.nuhc_allreduce(ys, b, g, table, seed, np.float32(m), np.float32(M),
                                                want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(st.packed[w])[:ref_pk[w].size], ref_pk[w])
    avg = to_host(st.avg).astype(np.float64)
    assert np.max(np.abs(avg - ref_avg)) <= 1e-6 * max(abs(m), abs(M))
    est_ref = oracle.rht(to_host(st.avg), 0xD1A6, inverse=True)
    assert np.linalg.norm(to_host(st.est).astype(np.float64) - est_ref) <= bound(to_host(st.avg))
    for w in range(P):
        # the worker's own vector decoded on the grid (P = 1), rotated back by the oracle
        if table is None:
            own = oracle.thc_decode(oracle.thc_aggregate([ref_pk[w]], n, b), np.float32(m), np.float32(M), b, 1)
        else:
            own = oracle.nuhc_decode(oracle.nuhc_aggregate([ref_pk[w]], n, b, table), np.float32(m),
                                     np.float32(M), steps, 1)
        xhat = oracle.rht(own.astype(np.float32), 0xD1A6, inverse=True)
        ref_e = xs[w].astype(np.float64) - xhat
        err = np.linalg.norm(to_host(st.errs[w]).astype(np.float64) - ref_e)
        # the rotation's bound, the update's two fp32 roundings, and the GPU's
        # fp32 decode against the oracle's fp64 one (1e-6 * M an element,
        # kept in norm by the orthogonal rotation)
        decode = np.sqrt(n) * 1e-6 * max(abs(m), abs(M))
        assert err <= bound(own) + 2 * U * float(np.linalg.norm(xs[w].astype(np.float64))) + decode, w


def test_rejects_bad_shapes(env):
    torch, gar = env
    from gradient_allreduce_homomorphic_gb300.training import TrainingStep

    g3 = [torch.zeros(3000, device="cuda") for _ in range(2)]
    with pytest.raises(ValueError):
        TrainingStep(g3, [t.clone() for t in g3])
    g4 = [torch.zeros(4096, device="cuda") for _ in range(2)]
    with pytest.raises(ValueError):
        TrainingStep(g4, [g4[0].clone()])
    with pytest.raises(ValueError):
        TrainingStep(g4, [t.clone() for t in g4], streams=0)


def test_two_stream_step_captured(env):
    """The step with its workers' chains on two side streams captured as one
    CUDA graph (the side streams fork from and join the capturing stream):
    replays from the same error vectors give the eager steps bit for bit."""
    torch, gar = env
    from gradient_allreduce_homomorphic_gb300.training import TrainingStep

    n = 1 << 21
    grads, errs = _inputs(torch, n, 21)
    e0 = [t.clone() for t in errs]
    st = TrainingStep(grads, errs, b=4, table=_table(4, 36), t_p=2.15, rht_seed=0xD1A6, streams=2)
    st.run(0x5EED)
    torch.cuda.synchronize()
    eager1 = _snapshot(st)
    st.run(0x5EED)
    torch.cuda.synchronize()
    eager2 = _snapshot(st)
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            st.run(0x5EED)
    torch.cuda.synchronize()
    for e, e_init in zip(st.errs, e0):
        e.copy_(e_init)
    for t in [st.avg, st.est, st.mM] + st.ys:
        t.zero_()
    torch.cuda.synchronize()
    n0 = gar.gar_launch_count()
    for ref in (eager1, eager2):
        graph.replay()
        torch.cuda.synchronize()
        for x, y in zip(_snapshot(st), ref):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert gar.gar_launch_count() == n0
