"""GPU parity of the plan-driven paths that skip the packed buffers.

gar_fused_allreduce_range must give the same per-buffer [m, M] as
gar_fusion_pack_all's range (bit for bit, zero padding included) and the
same averages as gar_fused_allreduce, leaving its inputs untouched.
gar_thc_allreduce_fused_plan must equal pack -> gar_thc_allreduce_fused per
buffer -> unpack bit for bit: the output tensors and every worker's packed
index words.  Plans cover ragged tensor ends, empty tensors, one-element
tensors packed tight (many tensors in one packed word), unaligned tensor
pointers, several launches per buffer (P=64), and the full-size ResNet-like
plan; one small case is checked against the oracle directly.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, same_bits, to_dev, to_host
from oracle_par import fusion_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _plan_inputs(trial, P, torch, tiny=False, offset=0):
    g = np.random.default_rng([141, trial])
    count = int(g.integers(1, 60))
    if tiny:
        sizes = g.integers(0, 3, size=count).astype(np.int64)
    else:
        sizes = g.integers(0, 3000, size=count).astype(np.int64)
        sizes[g.integers(0, count)] = int(g.integers(5000, 20000))
    src = []
    for w in range(P):
        row = []
        for i in range(count):
            x = np.random.default_rng([142, trial, w, i]).standard_normal(int(sizes[i])).astype(np.float32)
            if offset:  # a view starting `offset` elements into its storage: not 16-byte aligned
                t = torch.zeros(int(sizes[i]) + offset, device="cuda")
                t[offset:] = to_dev(x, torch)
                row.append(t[offset:])
            else:
                row.append(to_dev(x, torch))
        src.append(row)
    return sizes, src


def _reference(g, torch, src, plan, b, seed):
    """pack_all (+ range) -> THC per buffer -> unpack of the average."""
    P = len(src)
    fbs = [[torch.zeros(max(int(n), 1), device="cuda")[: int(n)] for n in plan.buf_numel] for _ in range(P)]
    mM = torch.empty((plan.n_buffers, 2), device="cuda")
    g.gar_fusion_pack_all(src, plan, fbs, mM)
    out = [torch.full_like(t, 1234.5) for t in src[0]]
    packed = [[None] * plan.n_buffers for _ in range(P)]
    bufs = plan.buffers()
    for bf in range(plan.n_buffers):
        members = [i for i in range(plan.count) if bufs[i] == bf]
        if not members:
            continue
        n = int(plan.buf_numel[bf])
        avg = torch.empty(n, device="cuda")
        pk = [torch.zeros(max(g.gar_thc_words(n, b), 1), dtype=torch.int32, device="cuda") for _ in range(P)]
        g.gar_thc_allreduce_fused([fbs[w][bf] for w in range(P)], b, seed, mM[bf], avg, pk)
        g.gar_fusion_unpack(avg, plan, bf, out)
        for w in range(P):
            packed[w][bf] = pk[w]
    return mM, out, packed


def _plan_run(g, torch, src, plan, b, seed, mM):
    P = len(src)
    out = [torch.full_like(t, 1234.5) for t in src[0]]
    packed = [[torch.zeros(max(g.gar_thc_words(int(n), b), 1), dtype=torch.int32, device="cuda")
               for n in plan.buf_numel] for _ in range(P)]
    g.gar_thc_allreduce_fused_plan(src, plan, b, seed, mM, out, packed)
    return out, packed


def _compare(g, plan, ref, got, P):
    _, ref_out, ref_pk = ref
    out, pk = got
    for i in range(plan.count):
        same_bits(to_host(out[i]), to_host(ref_out[i]))
    bufs = plan.buffers()
    for bf in range(plan.n_buffers):
        if not any(bufs[i] == bf for i in range(plan.count)):
            continue
        for w in range(P):
            np.testing.assert_array_equal(to_host(pk[w][bf]), to_host(ref_pk[w][bf]))


@pytest.mark.parametrize("trial", range(6))
@pytest.mark.parametrize("P", [1, 3, 8])
@pytest.mark.parametrize("align", [16, 4])
def test_fused_allreduce_range(env, trial, P, align):
    torch, g = env
    sizes, src = _plan_inputs(trial, P, torch)
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, align)
    keep = [[to_host(t).copy() for t in row] for row in src]
    fbs = [[torch.empty(max(int(n), 1), device="cuda")[: int(n)] for n in plan.buf_numel] for _ in range(P)]
    ref_mM = torch.full((plan.n_buffers, 2), 99.0, device="cuda")
    g.gar_fusion_pack_all(src, plan, fbs, ref_mM)
    mM = torch.full((plan.n_buffers, 2), 99.0, device="cuda")
    dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce_range(src, dst, plan, mM)
    same_bits(to_host(mM), to_host(ref_mM))
    ref_dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce(src, ref_dst, plan)
    for w in range(P):
        for i in range(len(sizes)):
            same_bits(to_host(dst[w][i]), to_host(ref_dst[w][i]))
            same_bits(to_host(src[w][i]), keep[w][i])  # inputs untouched


def test_fused_allreduce_range_slices_and_errors(env):
    torch, g = env
    sizes, src = _plan_inputs(3, 4, torch)
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, 16)
    fbs = [[torch.empty(max(int(n), 1), device="cuda")[: int(n)] for n in plan.buf_numel] for _ in range(4)]
    ref = torch.empty((plan.n_buffers, 2), device="cuda")
    g.gar_fusion_pack_all(src, plan, fbs, ref)
    bufs = plan.buffers()
    mM = torch.full((plan.n_buffers, 2), 7.0, device="cuda")
    for bf in range(plan.n_buffers):  # one call per buffer, as a pipelined schedule makes them
        idx = [i for i in range(plan.count) if bufs[i] == bf]
        if not idx:
            continue
        sub = plan.subplan(idx[0], len(idx))
        dst = [[torch.empty_like(src[w][i]) for i in idx] for w in range(4)]
        g.gar_fused_allreduce_range([[src[w][i] for i in idx] for w in range(4)], dst, sub, mM)
    same_bits(to_host(mM), to_host(ref))
    bf16 = [[t.to(torch.bfloat16) for t in row] for row in src]
    plan16 = g.gar_fusion_plan(sizes, np.ones(len(sizes), np.int32), 16 << 10, 16)
    with pytest.raises(g.GarError) as e:
        g.gar_fused_allreduce_range(bf16, bf16, plan16, mM)
    assert e.value.status == g.GAR_EDTYPE


@pytest.mark.parametrize("trial", range(5))
@pytest.mark.parametrize("P", [1, 3, 4, 8, 16])
@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_thc_plan_equals_pack_thc_unpack(env, trial, P, b):
    torch, g = env
    if P * ((1 << b) - 1) > 65535:
        pytest.skip("overflow")
    sizes, src = _plan_inputs(trial, P, torch)
    align = 16 if trial % 2 == 0 else 4
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, align)
    seed = 0x5EED + trial
    ref = _reference(g, torch, src, plan, b, seed)
    _compare(g, plan, ref, _plan_run(g, torch, src, plan, b, seed, ref[0]), P)


@pytest.mark.parametrize("b", [1, 4, 8])
def test_thc_plan_tiny_tensors_many_launches(env, b):
    """P=64: at most 32 tensors per launch; one-element tensors packed tight
    put up to 32 tensors in one packed word."""
    torch, g = env
    P = 64 if b < 8 else 16
    sizes, src = _plan_inputs(7, P, torch, tiny=True)
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 1 << 10, 4)
    ref = _reference(g, torch, src, plan, b, 99)
    _compare(g, plan, ref, _plan_run(g, torch, src, plan, b, 99, ref[0]), P)
    sizes, src = _plan_inputs(8, P, torch)  # larger tensors, several launches per buffer
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 64 << 10, 16)
    ref = _reference(g, torch, src, plan, b, 98)
    _compare(g, plan, ref, _plan_run(g, torch, src, plan, b, 98, ref[0]), P)


def test_thc_plan_unaligned_pointers(env):
    torch, g = env
    sizes, src = _plan_inputs(4, 5, torch, offset=1)
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, 16)
    ref = _reference(g, torch, src, plan, 4, 5)
    _compare(g, plan, ref, _plan_run(g, torch, src, plan, 4, 5, ref[0]), 5)


def test_thc_plan_against_oracle(env):
    torch, g = env
    P, b, seed = 3, 4, 0x5EED
    sizes, src = _plan_inputs(11, P, torch)
    dt = np.zeros(len(sizes), np.int32)
    plan = g.gar_fusion_plan(sizes, dt, 16 << 10, 16)
    host = [[to_host(t) for t in row] for row in src]
    sb, so, bn = oracle.fusion_plan(sizes, dt, 16 << 10, 16)
    mM = torch.empty((plan.n_buffers, 2), device="cuda")
    g.gar_fused_allreduce_range(src, [[torch.empty_like(t) for t in row] for row in src], plan, mM)
    out, pk = _plan_run(g, torch, src, plan, b, seed, mM)
    for bf in range(len(bn)):
        members = [i for i in range(len(sizes)) if sb[i] == bf]
        if not members:
            continue
        bufs = [oracle.fusion_pack(host[w], sb, so, bf, bn[bf]) for w in range(P)]
        m, M = oracle.thc_range(bufs)
        assert (float(m), float(M)) == tuple(float(v) for v in to_host(mM[bf]))
        avg, ref_pk = oracle.thc_allreduce(bufs, b, seed, m, M, want_packed=True)
        for w in range(P):
            np.testing.assert_array_equal(to_host(pk[w][bf])[: ref_pk[w].size], ref_pk[w])
        tol = 1e-6 * max(abs(float(m)), abs(float(M)))
        for i in members:
            ref = avg[so[i]: so[i] + sizes[i]]
            assert np.max(np.abs(to_host(out[i]).astype(np.float64) - ref), initial=0.0) <= tol


def test_resnet_plan_full_size(env):
    """The bench's workload and kernel builds (the ring fold with the range,
    the plan THC kernel built for 8 workers): P=8, 300 tensors (45M
    parameters), b=4, against the oracle's pack -> ring fold / range / THC
    round -> unpack over every value of every worker, and against the GPU's
    own pack -> THC -> unpack composition."""
    torch, g = env
    P, b, seed = 8, 4, workloads.THC_SEED
    sizes = workloads.resnet_fusion_sizes()
    dt = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, 64 << 20, 16)
    src = [[workloads.device_normal(int(s), 0.01, 5000 * w + i, torch.float32, "cuda") for i, s in enumerate(sizes)]
           for w in range(P)]
    mM = torch.empty((plan.n_buffers, 2), device="cuda")
    dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce_range(src, dst, plan, mM)
    out, pk = _plan_run(g, torch, src, plan, b, seed, mM)
    torch.cuda.synchronize()
    host = [[to_host(t) for t in row] for row in src]
    sb, so, bn, per = fusion_step(host, sizes, 64 << 20, 16, b, seed)
    assert np.array_equal(sb, plan.buffers()) and np.array_equal(so, plan.offsets())
    got_mM = to_host(mM)
    for k in range(len(bn)):
        m, M = per[k]["mM"]
        assert (got_mM[k, 0], got_mM[k, 1]) == (m, M)
        ring = oracle.fusion_unpack(per[k]["ring"], sb, so, sizes, k)
        tol = 1e-6 * max(abs(float(m)), abs(float(M)))
        for i in np.nonzero(sb == k)[0]:
            for w in range(P):
                same_bits(to_host(dst[w][i]), ring[i])
            ref = per[k]["thc"][int(so[i]):int(so[i]) + int(sizes[i])]
            assert np.max(np.abs(to_host(out[i]).astype(np.float64) - ref), initial=0.0) <= tol
        for w in range(P):
            np.testing.assert_array_equal(to_host(pk[w][k])[: per[k]["packed"][w].size], per[k]["packed"][w])
    ref = _reference(g, torch, src, plan, b, seed)
    same_bits(got_mM, to_host(ref[0]))
    for i in range(plan.count):
        assert torch.equal(out[i].view(torch.int32), ref[1][i].view(torch.int32))


def _nmse_run(g, torch, src, plan, b, seed, mM, refs):
    P = len(src)
    out = [torch.full_like(t, 1234.5) for t in src[0]]
    packed = [[torch.zeros(max(g.gar_thc_words(int(n), b), 1), dtype=torch.int32, device="cuda")
               for n in plan.buf_numel] for _ in range(P)]
    ws = torch.empty(g.gar_thc_plan_nmse_workspace_bytes(plan, b) // 8 + 1, dtype=torch.float64, device="cuda")
    pair = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    g.gar_thc_allreduce_fused_plan_nmse(src, plan, b, seed, mM, out, refs, pair, ws, packed)
    return out, packed, pair


@pytest.mark.parametrize("trial", range(4))
@pytest.mark.parametrize("P", [1, 3, 8, 16])
@pytest.mark.parametrize("b", [2, 4, 8])
def test_thc_plan_nmse(env, trial, P, b):
    """The NMSE variant gives the plain call's outputs and wire words bit for
    bit, and sums of (ref - avg)^2 and ref^2 within 2e-6 of fp64 sums over
    the tensors (gap elements excluded), the same on a second call."""
    torch, g = env
    sizes, src = _plan_inputs(trial, P, torch, offset=1 if trial == 3 else 0)
    align = 16 if trial % 2 == 0 else 4
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, align)
    seed = 0x5EED + 7 * trial
    ref = _reference(g, torch, src, plan, b, seed)
    refs = [torch.from_numpy(np.random.default_rng([143, trial, i]).standard_normal(int(n)).astype(np.float32)).cuda()
            for i, n in enumerate(sizes)]
    out, packed, pair = _nmse_run(g, torch, src, plan, b, seed, ref[0], refs)
    _compare(g, plan, ref, (out, packed), P)
    num = sum(float(np.sum((to_host(r).astype(np.float64) - to_host(o).astype(np.float64)) ** 2))
              for r, o in zip(refs, out))
    den = sum(float(np.sum(to_host(r).astype(np.float64) ** 2)) for r in refs)
    got = pair.cpu().numpy()
    assert abs(got[0] - num) <= 2e-6 * num + 1e-30 and abs(got[1] - den) <= 2e-6 * den + 1e-30
    _, _, pair2 = _nmse_run(g, torch, src, plan, b, seed, ref[0], refs)
    assert pair2.cpu().numpy().tobytes() == got.tobytes()


def test_thc_plan_nmse_resnet_combined(env):
    """The ResNet-like plan, one call per fusion buffer with the ring average
    as reference, pairs combined: the NMSE of the oracle over the whole model."""
    torch, g = env
    P, b, seed = 8, 4, 0x5EED
    cfg = workloads.CONFIG_IDS["resnet_fusion"]
    sizes = workloads.resnet_fusion_sizes()
    dt = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, 64 << 20, 16)
    src = [[workloads.device_normal(int(s), 0.01, 7000 + 1000 * w + i, torch.float32, "cuda")
            for i, s in enumerate(sizes)] for w in range(P)]
    ring = [[torch.empty_like(t) for t in row] for row in src]
    mM = torch.empty((plan.n_buffers, 2), device="cuda")
    g.gar_fused_allreduce_range(src, ring, plan, mM)
    out = [torch.empty_like(t) for t in src[0]]
    pairs = torch.empty((plan.n_buffers, 2), dtype=torch.float64, device="cuda")
    ws = torch.empty(g.gar_thc_plan_nmse_workspace_bytes(plan, b) // 8 + 1, dtype=torch.float64, device="cuda")
    for bf in range(plan.n_buffers):
        first, cnt = plan.buffer_tensors(bf)
        sub = plan.subplan(first, cnt)
        rows = slice(first, first + cnt)
        g.gar_thc_allreduce_fused_plan_nmse([row[rows] for row in src], sub, b, seed, mM, out[rows], ring[0][rows],
                                            pairs[bf], ws)
    nm = torch.empty(1, dtype=torch.float64, device="cuda")
    g.gar_nmse_combine(pairs, nm)
    ref = oracle.nmse(np.concatenate([to_host(t) for t in ring[0]]), np.concatenate([to_host(t) for t in out]))
    assert abs(nm.item() - ref) <= 2e-6 * ref


def test_thc_plan_nmse_edges(env):
    import ctypes

    torch, g = env
    lib = g.load()
    pair = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    ws = torch.empty(16, dtype=torch.float64, device="cuda")
    no_refs = (ctypes.c_void_p * 1)()
    # no tensors: the pair is (0, 0)
    rc = lib.gar_thc_allreduce_fused_plan_nmse(None, 3, None, None, 0, None, 0, 4, 1, None, None, None, no_refs,
                                               pair.data_ptr(), ws.data_ptr(), 128, None)
    assert rc == 0
    assert pair.cpu().numpy().tolist() == [0.0, 0.0]
    sizes, src = _plan_inputs(0, 3, torch)
    plan = g.gar_fusion_plan(sizes, np.zeros(len(sizes), np.int32), 16 << 10, 16)
    refs = [torch.zeros_like(t) for t in src[0]]
    out = [torch.empty_like(t) for t in src[0]]
    mM = torch.zeros((plan.n_buffers, 2), device="cuda")
    with pytest.raises(g.GarError):  # workspace too small
        g.gar_thc_allreduce_fused_plan_nmse(src, plan, 4, 1, mM, out, refs, pair, ws[:1])


@pytest.mark.parametrize("P,b,k", [(4, 4, 64), (8, 2, 40), (64, 4, 9), (3, 8, 70)])
def test_partition_stream(env, P, b, k):
    """A stream of THC partitions ([T] section 2: the model cut into 4 MB
    partitions, each with its own range), small here: k partitions per
    worker, each its own fusion buffer, averaged by the ring with the range
    and by THC over the plan -- several buffers per launch -- against the
    oracle partition by partition."""
    torch, g = env
    rng = np.random.default_rng([151, P, b, k])
    n = 4096
    sizes = np.full(k, n, np.int64)
    sizes[rng.integers(0, k, 3)] = [1, 4093, 777]  # a few ragged partitions
    dt = np.zeros(k, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, n * 4, 16)
    assert plan.n_buffers == k
    host = [[(rng.standard_normal(int(s)) * rng.uniform(0.1, 10)).astype(np.float32) for s in sizes]
            for _ in range(P)]
    src = [[to_dev(x, torch) for x in row] for row in host]
    ring = [[torch.empty_like(t) for t in row] for row in src]
    mM = torch.full((k, 2), 7.0, device="cuda")
    g.gar_fused_allreduce_range(src, ring, plan, mM)
    seed = 0x5EED + k
    out, pk = _plan_run(g, torch, src, plan, b, seed, mM)
    torch.cuda.synchronize()
    got_mM = to_host(mM)
    for i in range(k):
        xs = [host[w][i] for w in range(P)]
        m, M = oracle.thc_range(xs)
        assert (got_mM[i, 0], got_mM[i, 1]) == (m, M), i
        for w in range(P):
            same_bits(to_host(ring[w][i]), oracle.ring_fold(xs, op=oracle.AVG))
        avg, ref_pk = oracle.thc_allreduce(xs, b, seed, m, M, want_packed=True)
        for w in range(P):
            np.testing.assert_array_equal(to_host(pk[w][i])[: ref_pk[w].size], ref_pk[w], err_msg=f"{i} {w}")
        tol = 1e-6 * max(abs(float(m)), abs(float(M)))
        assert np.max(np.abs(to_host(out[i]).astype(np.float64) - avg)) <= tol
