"""GPU parity of Tensor Fusion (pack, unpack, plan-driven fused all-reduce).

Bit-exact against the oracle: pack reproduces the oracle's fusion buffer
(zero padding included), unpack restores the tensors, and the one-pass
fused all-reduce equals the oracle's pack -> ring fold -> unpack and the
library's own pack -> ring -> unpack pipeline.  Full-size ResNet-like plan
(300 tensors, P=8) and VGG-like plan (P=8, 138M parameters) compared on
every element of every worker.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import bf16_bits, need_cuda, same_bits, to_dev, to_host
from oracle_par import ring_fold_range

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _random_plan_inputs(trial, P, mixed):
    g = np.random.default_rng([91, trial])
    count = int(g.integers(1, 40))
    sizes = g.integers(0, 3000, size=count).astype(np.int64)
    sizes[g.integers(0, count)] = int(g.integers(5000, 20000))  # one bigger than the capacity
    dtype = (g.integers(0, 2, size=count) if mixed else np.zeros(count)).astype(np.int32)
    host = []
    for w in range(P):
        row = []
        for i in range(count):
            x = np.random.default_rng([92, trial, w, i]).standard_normal(int(sizes[i])).astype(np.float32)
            row.append(x)
        host.append(row)
    return sizes, dtype, host


def _as_dtype(x, dt, torch):
    return bf16_bits(x, torch) if dt == 1 else x


@pytest.mark.parametrize("trial", range(8))
@pytest.mark.parametrize("align", [16, 4])
def test_pack_unpack(env, trial, align):
    torch, g = env
    sizes, dtype, host32 = _random_plan_inputs(trial, 1, mixed=trial % 2 == 1)
    host = [_as_dtype(x, int(d), torch) for x, d in zip(host32[0], dtype)]
    cap = 16 << 10
    plan = g.gar_fusion_plan(sizes, dtype, cap, align)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, cap, align)
    src = [to_dev(h, torch) for h in host]
    for b in range(plan.n_buffers):
        members = [i for i in range(len(sizes)) if sb[i] == b]
        ref = oracle.fusion_pack([host[i] for i in range(len(sizes))], sb, so, b, bn[b]) if members else None
        tdt = torch.bfloat16 if (members and dtype[members[0]] == 1) else torch.float32
        fb = torch.full((int(bn[b]),), 7.0, dtype=tdt, device="cuda")  # garbage that padding must clear
        g.gar_fusion_pack(src, plan, b, fb)
        if members:
            same_bits(to_host(fb), ref)
        dst = [torch.empty_like(t) for t in src]
        g.gar_fusion_unpack(fb, plan, b, dst)
        for i in members:
            same_bits(to_host(dst[i]), host[i])


def _oracle_fused(host, sizes, dtype, sb, so, bn, op):
    """pack -> ring fold -> unpack with the oracle, per worker."""
    P = len(host)
    out = [[None] * len(sizes) for _ in range(P)]
    for b in range(len(bn)):
        members = [i for i in range(len(sizes)) if sb[i] == b]
        if not members:
            continue
        packed = [oracle.fusion_pack(host[w], sb, so, b, bn[b]) for w in range(P)]
        red = oracle.ring_fold(packed, op=op)
        pieces = oracle.fusion_unpack(red, sb, so, sizes, b)
        for i in members:
            for w in range(P):
                out[w][i] = pieces[i]
    return out


@pytest.mark.parametrize("trial", range(10))
@pytest.mark.parametrize("P", [2, 3, 8])
def test_fused_allreduce(env, trial, P):
    torch, g = env
    sizes, dtype, host32 = _random_plan_inputs(trial, P, mixed=trial % 2 == 1)
    host = [[_as_dtype(x, int(d), torch) for x, d in zip(row, dtype)] for row in host32]
    cap, align = 16 << 10, 16
    plan = g.gar_fusion_plan(sizes, dtype, cap, align)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, cap, align)
    op = g.GAR_AVG if trial % 3 else g.GAR_SUM
    ref = _oracle_fused(host, sizes, dtype, sb, so, bn, op)
    src = [[to_dev(h, torch) for h in row] for row in host]
    dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce(src, dst, plan, op=op)
    for w in range(P):
        for i in range(len(sizes)):
            same_bits(to_host(dst[w][i]), ref[w][i])
    # in place gives the same bits
    g.gar_fused_allreduce(src, src, plan, op=op)
    for w in range(P):
        for i in range(len(sizes)):
            same_bits(to_host(src[w][i]), ref[w][i])


def test_fused_equals_pack_ring_unpack_on_gpu(env):
    torch, g = env
    P = 4
    sizes, dtype, host = _random_plan_inputs(3, P, mixed=False)
    plan = g.gar_fusion_plan(sizes, dtype, 16 << 10, 16)
    src = [[to_dev(h, torch) for h in row] for row in host]
    fused = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce(src, fused, plan, op=g.GAR_AVG)
    staged = [[torch.empty_like(t) for t in row] for row in src]
    for b in range(plan.n_buffers):
        fbs = [torch.empty(int(plan.buf_numel[b]), dtype=torch.float32, device="cuda") for _ in range(P)]
        for w in range(P):
            g.gar_fusion_pack(src[w], plan, b, fbs[w])
        g.gar_ring_allreduce_sim(fbs, op=g.GAR_AVG)
        for w in range(P):
            g.gar_fusion_unpack(fbs[w], plan, b, staged[w])
    for w in range(P):
        for i in range(len(sizes)):
            same_bits(to_host(fused[w][i]), to_host(staged[w][i]))


def test_fused_unaligned_tensors(env):
    torch, g = env
    P = 3
    sizes = np.array([101, 7, 2000, 33], np.int64)
    dtype = np.zeros(4, np.int32)
    plan = g.gar_fusion_plan(sizes, dtype, 1 << 20, 16)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, 1 << 20, 16)
    host = [[np.random.default_rng([93, w, i]).standard_normal(int(s)).astype(np.float32)
             for i, s in enumerate(sizes)] for w in range(P)]
    bases = [[to_dev(np.concatenate([[0.0], h]).astype(np.float32), torch) for h in row] for row in host]
    src = [[b[1:] for b in row] for row in bases]  # 4-byte aligned views
    dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce(src, dst, plan, op=g.GAR_AVG)
    ref = _oracle_fused(host, sizes, dtype, sb, so, bn, oracle.AVG)
    for w in range(P):
        for i in range(len(sizes)):
            same_bits(to_host(dst[w][i]), ref[w][i])


@pytest.mark.parametrize("inplace", [False, True])
def test_fused_common_phase_views(env, inplace):
    """Unpadded views of one flat buffer per worker (tensor i starts at the sum
    of the sizes before it): the tensors are not 16-byte aligned, but all of a
    tensor's pointers share one phase, so the fold runs in 16-byte vectors
    after a short scalar head -- with the same sums as the oracle."""
    torch, g = env
    P = 8
    sizes = np.array([5, 1, 4099, 3, 70001, 2, 9, 40000, 7, 123457], np.int64)
    dtype = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dtype, 256 << 10, 16)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, 256 << 10, 16)
    host = [workloads.tensors_normal(sizes, 1.0, 94, w) for w in range(P)]
    offs = np.concatenate([[0], np.cumsum(sizes)])

    def views(flat):
        return [flat[int(offs[i]):int(offs[i + 1])] for i in range(sizes.size)]

    src_flat = [to_dev(np.concatenate(row), torch) for row in host]
    src = [views(f) for f in src_flat]
    if inplace:
        dst = src
    else:
        dst_flat = [torch.zeros(int(offs[-1]), device="cuda") for _ in range(P)]
        dst = [views(f) for f in dst_flat]
    g.gar_fused_allreduce(src, dst, plan, op=g.GAR_AVG)
    ref = _oracle_fused(host, sizes, dtype, sb, so, bn, oracle.AVG)
    for w in range(P):
        for i in range(sizes.size):
            same_bits(to_host(dst[w][i]), ref[w][i])


def test_resnet_fusion_full_size(env):
    # 300 fp32 tensors (~45M parameters), P=8, N(0, 0.01), 64 MB fusion buffers
    torch, g = env
    P = 8
    cfg = workloads.CONFIG_IDS["resnet_fusion"]
    sizes = workloads.resnet_fusion_sizes()
    dtype = np.zeros(sizes.size, np.int32)
    host = [workloads.tensors_normal(sizes, 0.01, cfg, w) for w in range(P)]
    plan = g.gar_fusion_plan(sizes, dtype, 64 << 20, 16)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, 64 << 20, 16)
    assert plan.n_buffers == len(bn) == 3
    src = [[to_dev(h, torch) for h in row] for row in host]
    dst = [[torch.empty_like(t) for t in row] for row in src]
    g.gar_fused_allreduce(src, dst, plan, op=g.GAR_AVG)
    ref = _oracle_fused(host, sizes, dtype, sb, so, bn, oracle.AVG)
    for w in (0, 3, 7):
        for i in range(len(sizes)):
            same_bits(to_host(dst[w][i]), ref[w][i])


def test_vgg_fusion_full_size(env):
    # 16 fp32 tensors, 138M parameters (largest 102,760,448), P=8, N(0, 1e-3),
    # fused pack + ring + unpack in place (the launch the benchmark times):
    # every element of every tensor of every worker against the oracle's
    # ring fold at that element's position in its fusion buffer
    torch, g = env
    P = 8
    sizes = workloads.vgg_fusion_sizes()
    dtype = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dtype, 64 << 20, 16)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, 64 << 20, 16)
    assert np.array_equal(sb, plan.buffers()) and np.array_equal(so, plan.offsets())
    src = [[workloads.device_normal(int(s), 1e-3, 7000 + 100 * w + i, torch.float32, "cuda")
            for i, s in enumerate(sizes)] for w in range(P)]
    host = [[to_host(t) for t in row] for row in src]  # the inputs, before the in-place call
    g.gar_fused_allreduce(src, src, plan, op=g.GAR_AVG)
    torch.cuda.synchronize()
    chunk = 1 << 23
    for i, s in enumerate(sizes):
        k = int(sb[i])
        got = [to_host(src[w][i]) for w in range(P)]
        for lo in range(0, int(s), chunk):
            hi = min(int(s), lo + chunk)
            ref = ring_fold_range(np.stack([host[w][i][lo:hi] for w in range(P)]), int(bn[k]), int(so[i]) + lo,
                                  op=oracle.AVG)
            for w in range(P):
                same_bits(got[w][lo:hi], ref)
    del src
    torch.cuda.empty_cache()


@pytest.mark.parametrize("trial", range(8))
@pytest.mark.parametrize("P", [1, 3, 8])
def test_pack_all(env, trial, P):
    # every worker, every buffer in one pass: the same bytes as per-worker packs;
    # with a range, the min/max of the packed buffers (padding zeros included)
    torch, g = env
    mixed = trial % 4 == 3
    sizes, dtype, host32 = _random_plan_inputs(trial, P, mixed=mixed)
    host = [[_as_dtype(x, int(d), torch) for x, d in zip(row, dtype)] for row in host32]
    cap, align = 16 << 10, (16 if trial % 2 == 0 else 4)
    plan = g.gar_fusion_plan(sizes, dtype, cap, align)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, cap, align)
    src = [[to_dev(h, torch) for h in row] for row in host]
    fbs = []
    for w in range(P):
        row = []
        for b in range(len(bn)):
            members = [i for i in range(len(sizes)) if sb[i] == b]
            tdt = torch.bfloat16 if (members and dtype[members[0]] == 1) else torch.float32
            row.append(torch.full((int(bn[b]),), 9.0, dtype=tdt, device="cuda"))
        fbs.append(row)
    want_range = not mixed
    mM = torch.empty((len(bn), 2), dtype=torch.float32, device="cuda") if want_range else None
    g.gar_fusion_pack_all(src, plan, fbs, mM)
    for b in range(len(bn)):
        packed = [oracle.fusion_pack(host[w], sb, so, b, bn[b]) for w in range(P)]
        for w in range(P):
            same_bits(to_host(fbs[w][b]), packed[w])
        if want_range and bn[b] > 0:
            m, M = oracle.thc_range(packed)
            assert to_host(mM[b]).tolist() == [m, M]


def test_pack_all_unaligned_and_leading_gap(env):
    torch, g = env
    P = 3
    sizes = np.array([5, 17, 0, 40], np.int64)
    dtype = np.zeros(4, np.int32)
    plan = g.gar_fusion_plan(sizes, dtype, 1 << 20, 16)
    # a hand-made plan: the first tensor starts at offset 3 (zeros before it)
    for s, off in zip(plan.segs, (3, 12, 32, 32)):
        s.offset = off
    plan.buf_numel[0] = 75
    host = [[np.random.default_rng([96, w, i]).standard_normal(int(k)).astype(np.float32) for i, k in enumerate(sizes)]
            for w in range(P)]
    bases = [[to_dev(np.concatenate([[1.0], h]).astype(np.float32), torch) for h in row] for row in host]
    src = [[b[1:] for b in row] for row in bases]  # 4-byte aligned views
    fbs = [[torch.full((75,), 5.0, device="cuda")] for _ in range(P)]
    mM = torch.empty((1, 2), device="cuda")
    g.gar_fusion_pack_all(src, plan, fbs, mM)
    for w in range(P):
        ref = np.zeros(75, np.float32)
        for k, off in zip(range(4), (3, 12, 32, 32)):
            ref[off:off + sizes[k]] = host[w][k]
        same_bits(to_host(fbs[w][0]), ref)
    allv = np.concatenate([np.concatenate(r) for r in host] + [np.zeros(1, np.float32)])
    assert to_host(mM[0]).tolist() == [allv.min(), allv.max()]


def test_plan_slices(env):
    # a slice of the plan (one buffer's tensors) packs, ranges and reduces only
    # that buffer; every other buffer and range entry is left untouched
    torch, g = env
    P = 4
    sizes, dtype, host = _random_plan_inputs(5, P, mixed=False)
    plan = g.gar_fusion_plan(sizes, dtype, 16 << 10, 16)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, 16 << 10, 16)
    assert plan.n_buffers >= 2
    src = [[to_dev(h, torch) for h in row] for row in host]
    fbs = [[torch.full((int(k),), 3.0, device="cuda") for k in bn] for _ in range(P)]
    mM = torch.full((len(bn), 2), 7.0, device="cuda")
    b = 1
    first, cnt = plan.buffer_tensors(b)
    assert list(range(first, first + cnt)) == [i for i in range(len(sizes)) if sb[i] == b]
    sub = plan.subplan(first, cnt)
    g.gar_fusion_pack_all([row[first:first + cnt] for row in src], sub, fbs, mM)
    packed = [oracle.fusion_pack(host[w], sb, so, b, bn[b]) for w in range(P)]
    m, M = oracle.thc_range(packed)
    assert to_host(mM[b]).tolist() == [m, M]
    for bb in range(len(bn)):
        if bb != b:
            assert np.all(to_host(mM[bb]) == 7.0)
        for w in range(P):
            if bb == b:
                same_bits(to_host(fbs[w][bb]), packed[w])
            else:
                assert np.all(to_host(fbs[w][bb]) == 3.0)
    # the fused all-reduce of the slice touches only that buffer's tensors
    dst = [[torch.full_like(t, 5.0) for t in row] for row in src]
    g.gar_fused_allreduce([row[first:first + cnt] for row in src], [row[first:first + cnt] for row in dst], sub)
    ref = _oracle_fused(host, sizes, dtype, sb, so, bn, oracle.AVG)
    for w in range(P):
        for i in range(len(sizes)):
            if first <= i < first + cnt:
                same_bits(to_host(dst[w][i]), ref[w][i])
            else:
                assert np.all(to_host(dst[w][i]) == 5.0)
