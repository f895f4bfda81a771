"""Pins for the oracle's Tensor Fusion plan, pack and unpack (CPU only).

The plan is checked against properties that together single out the
next-fit rule the Horovod page's fusion steps describe (ready order, same
dtype, fits in the room left, oversize tensors alone), not against a second
copy of the rule.  Pack and unpack are byte copies: round trip identity and
zero padding.
"""
import numpy as np
import pytest

import oracle
import workloads

ES = {oracle.F32: 4, oracle.BF16: 2}


def check_plan(numel, dtype, cap, align, plan):
    seg_buf, seg_off, buf_numel = plan
    count = len(numel)
    if count == 0:
        assert len(buf_numel) == 0
        return
    assert seg_buf[0] == 0
    ends = {}
    for i in range(count):
        es = ES[int(dtype[i])]
        nbytes = int(numel[i]) * es
        if i > 0:
            step = int(seg_buf[i]) - int(seg_buf[i - 1])
            assert step in (0, 1), "buffers are opened in list order"
        b = int(seg_buf[i])
        if i == 0 or seg_buf[i] != seg_buf[i - 1]:
            assert seg_off[i] == 0, "a new buffer starts at offset 0"
            if i > 0:
                # closed only for a dtype change or because tensor i does not fit
                pes = ES[int(dtype[i - 1])]
                prev_end = (int(seg_off[i - 1]) + int(numel[i - 1])) * pes
                start = -(-prev_end // align) * align
                assert dtype[i] != dtype[i - 1] or start + nbytes > cap
        else:
            assert dtype[i] == dtype[i - 1], "one dtype per buffer"
            prev_end = (int(seg_off[i - 1]) + int(numel[i - 1])) * es
            start = -(-prev_end // align) * align
            assert int(seg_off[i]) * es == start, "the next aligned position, no gap beyond alignment"
            assert start + nbytes <= cap, "a tensor joins a buffer only if it fits"
        ends[b] = int(seg_off[i]) + int(numel[i])
    assert len(buf_numel) == max(ends) + 1
    for b, e in ends.items():
        assert buf_numel[b] == e
    for b in range(len(buf_numel)):
        members = [i for i in range(count) if seg_buf[i] == b]
        es = ES[int(dtype[members[0]])]
        if buf_numel[b] * es > cap:
            assert len(members) == 1, "only a lone oversize tensor exceeds the capacity"


def test_resnet_like_plan():
    sizes = workloads.resnet_fusion_sizes()
    dt = np.zeros(sizes.size, np.int32)
    plan = oracle.fusion_plan(sizes, dt, 64 << 20, 16)
    check_plan(sizes, dt, 64 << 20, 16, plan)
    assert len(plan[2]) == 3
    assert int(np.sum(sizes)) <= int(np.sum(plan[2]))


def test_vgg_like_plan_big_tensor_alone():
    sizes = workloads.vgg_fusion_sizes()
    dt = np.zeros(sizes.size, np.int32)
    plan = oracle.fusion_plan(sizes, dt, 64 << 20, 16)
    check_plan(sizes, dt, 64 << 20, 16, plan)
    big = int(np.argmax(sizes))
    assert sum(1 for b in plan[0] if b == plan[0][big]) == 1
    assert plan[2][plan[0][big]] == sizes[big]


@pytest.mark.parametrize("trial", range(40))
def test_random_plans(trial):
    g = np.random.default_rng([61, trial])
    count = int(g.integers(0, 40))
    numel = g.integers(0, 3000, size=count).astype(np.int64)
    mixed = trial % 2 == 1
    dtype = (g.integers(0, 2, size=count) if mixed else np.zeros(count)).astype(np.int32)
    cap = int(g.choice([64, 1000, 4096, 20000]))
    align = int(g.choice([4, 16, 64]))
    plan = oracle.fusion_plan(numel, dtype, cap, align)
    check_plan(numel, dtype, cap, align, plan)


def test_tight_alignment_is_contiguous():
    numel = np.array([3, 5, 7, 1], np.int64)
    dt = np.zeros(4, np.int32)
    sb, so, bn = oracle.fusion_plan(numel, dt, 1 << 20, 4)
    assert list(so) == [0, 3, 8, 15] and list(bn) == [16]


def test_dtype_change_closes_buffer():
    numel = np.array([10, 10, 10, 10], np.int64)
    dt = np.array([0, 0, 1, 0], np.int32)
    sb, so, bn = oracle.fusion_plan(numel, dt, 1 << 20, 16)
    assert list(sb) == [0, 0, 1, 2]


def test_bad_alignment_rejected():
    with pytest.raises(ValueError):
        oracle.fusion_plan(np.array([4], np.int64), np.array([0], np.int32), 1024, 6)


@pytest.mark.parametrize("dtype,np_t", [(oracle.F32, np.float32), (oracle.BF16, np.uint16)])
def test_pack_unpack_roundtrip(dtype, np_t):
    g = np.random.default_rng(67)
    numel = g.integers(1, 500, size=25).astype(np.int64)
    dt = np.full(25, dtype, np.int32)
    sb, so, bn = oracle.fusion_plan(numel, dt, 2048, 16)
    if np_t is np.float32:
        tensors = [g.standard_normal(int(k)).astype(np.float32) for k in numel]
    else:
        tensors = [g.integers(0, 65536, size=int(k)).astype(np.uint16) for k in numel]
    restored = [None] * 25
    for b in range(len(bn)):
        buf = oracle.fusion_pack(tensors, sb, so, b, bn[b])
        # every element outside the tensors' slots is zero padding
        covered = np.zeros(int(bn[b]), bool)
        for i in range(25):
            if sb[i] == b:
                covered[so[i]:so[i] + numel[i]] = True
                np.testing.assert_array_equal(buf[so[i]:so[i] + numel[i]], tensors[i])
        assert np.all(buf[~covered] == 0)
        outs = oracle.fusion_unpack(buf, sb, so, numel, b)
        for i, o in enumerate(outs):
            if o is not None:
                restored[i] = o
    for t, r in zip(tensors, restored):
        np.testing.assert_array_equal(t, r)
