"""The averaging step captured in a CUDA graph: every call of the path is
asynchronous on the caller's stream, allocates nothing and waits for nothing,
so one step (the ring with each fusion buffer's THC range, THC b=4 over the
plan, the wire-vector checksum and the NMSE) can be captured once and replayed.
A replay must give the eager step's results bit for bit, and a replay after
the inputs were overwritten in place must follow the new values."""
import numpy as np
import pytest

import workloads
from helpers import need_cuda

pytestmark = pytest.mark.gpu

P, B_THC, SEED = 8, 4, 0x5EED


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _setup(torch, g):
    sizes = workloads.log_uniform_sizes(40, 256, 200_000, 1_000_000, [11, 999]).astype(np.int64)
    dt = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, capacity_bytes=1 << 20, align_bytes=16)
    n = int(sizes.sum())
    flat_src = [torch.empty(n, device="cuda") for _ in range(P)]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    src = [[f[offs[i]:offs[i + 1]] for i in range(sizes.size)] for f in flat_src]
    flat_ring = [torch.empty(n, device="cuda") for _ in range(P)]
    ring = [[f[offs[i]:offs[i + 1]] for i in range(sizes.size)] for f in flat_ring]
    flat_thc = torch.empty(n, device="cuda")
    thc = [flat_thc[offs[i]:offs[i + 1]] for i in range(sizes.size)]
    st = dict(plan=plan, n=n, flat_src=flat_src, src=src, flat_ring=flat_ring, ring=ring, flat_thc=flat_thc, thc=thc)
    st["mM"] = torch.empty((plan.n_buffers, 2), device="cuda")
    st["ws"] = torch.empty(g.gar_nmse_workspace_bytes(n) // 8 + 1, dtype=torch.float64, device="cuda")
    st["nmse"] = torch.empty(1, dtype=torch.float64, device="cuda")
    st["ck"] = torch.empty(1, dtype=torch.int64, device="cuda")
    return st


def _fill(torch, st, seed):
    for w, f in enumerate(st["flat_src"]):
        f.copy_(torch.from_numpy(workloads.normal_f32(st["n"], 0.01, seed, w)))


def _step(g, st):
    g.gar_fused_allreduce_range(st["src"], st["ring"], st["plan"], st["mM"])
    g.gar_thc_allreduce_fused_plan(st["src"], st["plan"], B_THC, SEED, st["mM"], st["thc"])
    g.gar_checksum(st["flat_thc"], st["ck"])
    g.gar_nmse(st["flat_ring"][0], st["flat_thc"], st["nmse"], st["ws"])


def _results(st):
    return ([f.cpu().numpy().view(np.uint32).copy() for f in st["flat_ring"]],
            st["flat_thc"].cpu().numpy().view(np.uint32).copy(), st["mM"].cpu().numpy().view(np.uint32).copy(),
            int(st["ck"].cpu().numpy()[0]), st["nmse"].cpu().numpy().view(np.uint64).copy())


def _same(a, b):
    for x, y in zip(a[0], b[0]):
        assert np.array_equal(x, y), "ring average"
    assert np.array_equal(a[1], b[1]), "THC average"
    assert np.array_equal(a[2], b[2]), "THC range"
    assert a[3] == b[3], "checksum"
    assert np.array_equal(a[4], b[4]), "NMSE"


def test_graph_replay_equals_eager(env):
    torch, g = env
    st = _setup(torch, g)
    _fill(torch, st, 301)
    _step(g, st)  # eager, also warms the library up before the capture
    torch.cuda.synchronize()
    eager = _results(st)

    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            _step(g, st)
    torch.cuda.synchronize()
    for f in st["flat_ring"]:
        f.zero_()
    st["flat_thc"].zero_()
    st["nmse"].zero_()
    launches0 = g.gar_launch_count()
    graph.replay()
    torch.cuda.synchronize()
    assert g.gar_launch_count() == launches0  # a replay issues no library call
    _same(_results(st), eager)

    # new gradients written into the same buffers: the replay reads them
    _fill(torch, st, 302)
    _step(g, st)
    torch.cuda.synchronize()
    eager2 = _results(st)
    assert not np.array_equal(eager2[1], eager[1])
    _fill(torch, st, 302)
    graph.replay()
    torch.cuda.synchronize()
    _same(_results(st), eager2)


def test_two_stream_step_captured(env):
    """The bucketed step the benchmark times (gradient_allreduce_homomorphic_gb300
    .pipeline: ring of each fusion buffer on one stream, THC of buffer b on a
    second stream behind an event, NMSE after both) captured as one graph:
    the side streams fork from and join the capturing stream, and a replay
    gives the eager step's results bit for bit, following new inputs."""
    torch, g = env
    from gradient_allreduce_homomorphic_gb300 import pipeline

    sizes = workloads.log_uniform_sizes(60, 256, 300_000, 2_000_000, [12, 999]).astype(np.int64)
    offs = pipeline.flat_offsets(sizes)
    grads = [torch.empty(int(offs[-1]), device="cuda") for _ in range(P)]

    def fill(seed):
        for w, f in enumerate(grads):
            f.copy_(torch.from_numpy(workloads.normal_f32(int(offs[-1]), 0.01, seed, w)))

    st = pipeline.AveragingStep(grads, sizes, offs, b=B_THC, capacity_bytes=1 << 20, align_bytes=16)
    assert st.nb > 2

    def results():
        return ([f.cpu().numpy().view(np.uint32).copy() for f in st.ring_flat],
                st.thc_flat.cpu().numpy().view(np.uint32).copy(), st.mM.cpu().numpy().view(np.uint32).copy(),
                [[t.cpu().numpy().copy() for t in row] for row in st.packed], st.nmse.cpu().numpy().view(np.uint64))

    def same(a, b):
        for x, y in zip(a[0], b[0]):
            assert np.array_equal(x, y), "ring average"
        assert np.array_equal(a[1], b[1]), "THC average"
        assert np.array_equal(a[2], b[2]), "ranges"
        for ra, rb in zip(a[3], b[3]):
            for x, y in zip(ra, rb):
                assert np.array_equal(x, y), "wire words"
        assert np.array_equal(a[4], b[4]), "NMSE"

    fill(401)
    st.run(SEED)
    torch.cuda.synchronize()
    eager = results()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            st.run(SEED)
    torch.cuda.synchronize()
    for f in st.ring_flat:
        f.zero_()
    st.thc_flat.zero_()
    graph.replay()
    torch.cuda.synchronize()
    same(results(), eager)
    fill(402)
    st.run(SEED)
    torch.cuda.synchronize()
    eager2 = results()
    assert not np.array_equal(eager2[1], eager[1])
    fill(402)
    graph.replay()
    torch.cuda.synchronize()
    same(results(), eager2)


def test_training_step_captured(env):
    """THC's section 5 training step through the fused calls -- per worker the
    error feedback applied inside the forward rotation with the norm's sums,
    the norm-based range, non-uniform THC (b = 4, g = 36), the inverse
    rotation of the average, per worker the error-feedback update from its own
    wire vector -- captured as one graph (cluster launches included; n = 2^21
    takes the 2-CTA cluster pass, 2^22 the 4-CTA one).  Replays from the same
    error vectors give the eager step's results bit for bit, two replays in a
    row the two eager steps'."""
    torch, g = env
    g.gar_sync_status(clear=True)  # earlier tests may have left a bit set
    P_, b, gr, t_p = 4, 4, 36, 2.15
    tab = np.rint(np.linspace(0, gr, 16)).astype(np.uint16)
    for k in (21, 22):
        n = 1 << k
        grads = [torch.from_numpy(workloads.student_t_f32(n, 4, 1e-2, 401, w)).cuda() for w in range(P_)]
        e0 = [torch.from_numpy(workloads.normal_f32(n, 1e-6, 402, w)).cuda() for w in range(P_)]
        e = [t.clone() for t in e0]
        ys = [torch.empty(n, device="cuda") for _ in range(P_)]
        packed = [torch.empty(g.gar_thc_words(n, b), dtype=torch.int32, device="cuda") for _ in range(P_)]
        sums = [torch.empty(g.gar_rht_tiles(n), dtype=torch.float64, device="cuda") for _ in range(P_)]
        yt, pt, st = g.pointer_table(ys), g.pointer_table(packed), g.pointer_table(sums)
        mM = torch.empty(2, device="cuda")
        avg, est, tmp = (torch.empty(n, device="cuda") for _ in range(3))

        def step():
            for w in range(P_):
                g.gar_rht_ef_forward(grads[w], e[w], ys[w], 11, sums[w])
            g.gar_rht_norm_range_from_sums(st, n, t_p, mM)
            g.gar_nuhc_allreduce_fused(yt, b, gr, tab, 5, mM, avg, pt)
            g.gar_rht(avg, est, 11, inverse=True)
            for w in range(P_):
                g.gar_rht_ef_update(packed[w], b, gr, tab, mM, grads[w], e[w], tmp, 11)

        def reset():
            for w in range(P_):
                e[w].copy_(e0[w])

        def results():
            out = [mM, avg, est] + ys + packed + e
            return [t.cpu().numpy().view(np.uint32 if t.dtype != torch.int32 else np.int32).copy() for t in out]

        def same(a, c):
            for x, y in zip(a, c):
                assert np.array_equal(x, y)

        reset()
        step()
        torch.cuda.synchronize()
        eager1 = results()
        step()
        torch.cuda.synchronize()
        eager2 = results()

        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                step()
        torch.cuda.synchronize()
        for t in [avg, est, mM] + ys:
            t.zero_()
        reset()
        launches0 = g.gar_launch_count()
        graph.replay()
        torch.cuda.synchronize()
        assert g.gar_launch_count() == launches0
        same(results(), eager1)
        graph.replay()
        torch.cuda.synchronize()
        same(results(), eager2)
        assert g.gar_sync_status() == 0
