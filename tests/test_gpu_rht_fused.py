"""GPU parity of the fused worker steps of THC's training process (THC section 5).

gar_rht_ef_forward (error feedback applied while the transform reads its
input, the norm's sums of squares taken in the same pass) and
gar_rht_ef_update (the worker's own indices decoded while the inverse
transform reads them, e updated while it writes) must give bit for bit what
the separate calls give: gar_ef_apply -> gar_rht, and aggregate([own]) ->
decode(P = 1) -> gar_rht(inverse) -> gar_ef_update.  The separate calls are
themselves held to the oracle (tests/test_gpu_rht.py); here the fused
results are also checked against the oracle directly: the rotation within
(log2 n + 2) 2^-24 ||x||, the range within 1e-6 relative, and e against the
oracle's fp32 update of the fp64 inverse rotation within the same bound.
Sizes cover the one-CTA kernel, the tile kernel alone, one strided pass,
cluster passes of 2 to 16 CTAs and two strided passes.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
SIZES = [0, 5, 11, 12, 13, 17, 20, 21, 22, 23, 24, 25]


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _bound(n, norm):
    k = max(int(n).bit_length() - 1, 1)
    return (k + 2) * U * norm * 1.0001 + 1e-30


def _table(b, g):
    L = (1 << b) - 1
    return np.rint(np.linspace(0, g, L + 1)).astype(np.uint16)


@pytest.mark.parametrize("k", SIZES)
def test_forward_equals_apply_then_rht(env, k):
    torch, gar = env
    n, seed = 1 << k, 0xD1A6 + k
    g = workloads.student_t_f32(n, 4, 1e-2, 191, k)
    e = workloads.normal_f32(n, 1e-6, 192, k)
    gd, ed = to_dev(g, torch), to_dev(e, torch)
    x = torch.empty(n, device="cuda")
    ref_y = torch.empty(n, device="cuda")
    gar.gar_ef_apply(gd, ed, x)
    gar.gar_rht(x, ref_y, seed)
    y = torch.full((n,), 7.0, device="cuda")
    sums = torch.full((gar.gar_rht_tiles(n),), -1.0, dtype=torch.float64, device="cuda")
    gar.gar_rht_ef_forward(gd, ed, y, seed, sums)
    same_bits(to_host(y), to_host(ref_y))
    same_bits(to_host(gd), g)  # inputs untouched
    same_bits(to_host(ed), e)
    xs = oracle.ef_apply(g, e)
    ref = oracle.rht(xs, seed)
    assert np.linalg.norm(to_host(y).astype(np.float64) - ref) <= _bound(n, np.linalg.norm(xs.astype(np.float64)))
    # the per-tile sums add up to ||x||^2
    s = to_host(sums)
    assert s.size == max(1, n // 4096) and np.all(s >= 0)
    exact = float(np.sum(xs.astype(np.float64) ** 2))
    assert abs(float(np.sum(s)) - exact) <= 1e-6 * exact
    # without sums: the same y
    y2 = torch.empty(n, device="cuda")
    gar.gar_rht_ef_forward(gd, ed, y2, seed)
    same_bits(to_host(y2), to_host(y))


@pytest.mark.parametrize("P,k", [(1, 5), (3, 12), (8, 16), (4, 21)])
def test_range_from_sums(env, P, k):
    torch, gar = env
    n, t_p = 1 << k, 2.15
    gs = [workloads.student_t_f32(n, 4, 1e-2, 193, w) for w in range(P)]
    es = [workloads.normal_f32(n, 1e-6, 194, w) for w in range(P)]
    sums = []
    for w in range(P):
        y = torch.empty(n, device="cuda")
        s = torch.empty(gar.gar_rht_tiles(n), dtype=torch.float64, device="cuda")
        gar.gar_rht_ef_forward(to_dev(gs[w], torch), to_dev(es[w], torch), y, 3, s)
        sums.append(s)
    mM = torch.empty(2, device="cuda")
    gar.gar_rht_norm_range_from_sums(sums, n, t_p, mM)
    m, M = (float(v) for v in to_host(mM))
    rm, rM = oracle.rht_norm_range([oracle.ef_apply(a, b) for a, b in zip(gs, es)], t_p)
    assert m == -M and abs(M - rM) <= 1e-6 * rM
    with pytest.raises(gar.GarError):
        gar.gar_rht_norm_range_from_sums(sums, n, -1.0, mM)


def _own_chain(torch, gar, packed, b, steps, table, mM, gd, e_old, seed):
    """The separate calls the fused update must equal."""
    n = gd.numel()
    own = torch.empty(n + 1, dtype=torch.int16, device="cuda")[:n]
    y_hat = torch.empty(n, device="cuda")
    if table is None:
        gar.gar_thc_aggregate([packed], n, b, own)
        gar.gar_thc_decode(own, mM, b, 1, y_hat)
    else:
        gar.gar_nuhc_aggregate([packed], n, b, table, own)
        gar.gar_nuhc_decode(own, mM, steps, 1, y_hat)
    x_hat = torch.empty(n, device="cuda")
    gar.gar_rht(y_hat, x_hat, seed, inverse=True)
    x = torch.empty(n, device="cuda")
    gar.gar_ef_apply(gd, e_old, x)
    e = e_old.clone()
    gar.gar_ef_update(e, x, x_hat)
    return e, y_hat, x


@pytest.mark.parametrize("k", SIZES)
@pytest.mark.parametrize("b,g", [(4, 36), (2, None), (8, 300), (1, None)])
def test_update_equals_separate_chain(env, k, b, g):
    torch, gar = env
    n, seed, q_seed = 1 << k, 0xD1A6 + k, 0x5EED + k
    L = (1 << b) - 1
    table = _table(b, g) if g is not None else None
    steps = g if g is not None else L
    gs = workloads.student_t_f32(n, 4, 1e-2, 195, k)
    es = workloads.normal_f32(n, 1e-6, 196, k)
    gd, ed = to_dev(gs, torch), to_dev(es, torch)
    y = torch.empty(n, device="cuda")
    gar.gar_rht_ef_forward(gd, ed, y, seed)
    mM = torch.empty(2, device="cuda")
    gar.gar_thc_range([y], mM)
    packed = torch.zeros(max(gar.gar_thc_words(n, b), 1), dtype=torch.int32, device="cuda")
    if table is None:
        gar.gar_thc_encode(y, mM, b, q_seed, 0, packed)
    else:
        gar.gar_nuhc_encode(y, mM, b, g, table, q_seed, 0, packed)
    ref_e, y_hat, x = _own_chain(torch, gar, packed, b, steps, table, mM, gd, ed, seed)
    e = ed.clone()
    tmp = torch.full((n,), 5.0, device="cuda")
    gar.gar_rht_ef_update(packed, b, steps, table, mM, gd, e, tmp, seed)
    same_bits(to_host(e), to_host(ref_e))
    same_bits(to_host(gd), gs)
    # against the oracle: x - rht^-1(y_hat) in fp64, rounded like the fp32 update
    xs = oracle.ef_apply(gs, es)
    ref_xhat = oracle.rht(to_host(y_hat), seed, inverse=True)
    err = np.linalg.norm(to_host(e).astype(np.float64) - (xs.astype(np.float64) - ref_xhat))
    bound = _bound(n, np.linalg.norm(to_host(y_hat).astype(np.float64))) + 2 * U * np.linalg.norm(xs) + 1e-30
    assert err <= bound


@pytest.mark.parametrize("k", [13, 21, 24])
def test_update_scratch_alignment(env, k):
    """Where tmp is 128-byte aligned the update's last pass drops the scratch
    lines from L2 once read; where it is only 16-byte aligned it does not.
    Both must give the same e, bit for bit, and both equal the separate chain."""
    torch, gar = env
    n, b, g, seed, q_seed = 1 << k, 4, 36, 0xA11 + k, 0xB22 + k
    table = _table(b, g)
    gs = workloads.student_t_f32(n, 4, 1e-2, 197, k)
    es = workloads.normal_f32(n, 1e-6, 198, k)
    gd, ed = to_dev(gs, torch), to_dev(es, torch)
    y = torch.empty(n, device="cuda")
    gar.gar_rht_ef_forward(gd, ed, y, seed)
    mM = torch.empty(2, device="cuda")
    gar.gar_thc_range([y], mM)
    packed = torch.zeros(gar.gar_thc_words(n, b), dtype=torch.int32, device="cuda")
    gar.gar_nuhc_encode(y, mM, b, g, table, q_seed, 0, packed)
    ref_e, _, _ = _own_chain(torch, gar, packed, b, g, table, mM, gd, ed, seed)
    base = torch.full((n + 64,), 3.0, device="cuda")
    assert base.data_ptr() % 128 == 0
    outs = []
    for off in (0, 4):  # 0 B and 16 B past a 128-byte boundary
        e = ed.clone()
        gar.gar_rht_ef_update(packed, b, g, table, mM, gd, e, base[off:off + n], seed)
        outs.append(to_host(e))
    same_bits(outs[0], outs[1])
    same_bits(outs[0], to_host(ref_e))


def test_update_rejects_bad_tables(env):
    torch, gar = env
    n = 64
    packed = torch.zeros(gar.gar_thc_words(n, 4), dtype=torch.int32, device="cuda")
    mM = torch.tensor([-1.0, 1.0], device="cuda")
    gd, e, tmp = (torch.zeros(n, device="cuda") for _ in range(3))
    with pytest.raises(gar.GarError):  # no table: the grid has 2^b - 1 steps
        gar.gar_rht_ef_update(packed, 4, 20, None, mM, gd, e, tmp, 1)
    bad = _table(4, 36)
    bad[5] = bad[4]
    with pytest.raises(gar.GarError):
        gar.gar_rht_ef_update(packed, 4, 36, bad, mM, gd, e, tmp, 1)
    with pytest.raises(gar.GarError):  # tmp overlaps e
        gar.gar_rht_ef_update(packed, 4, 15, None, mM, gd, e, e, 1)


@pytest.mark.parametrize("P,k,b,g,p", [(4, 16, 4, 36, 1 / 32), (3, 12, 2, 5, 1 / 32), (8, 22, 4, 36, 1 / 64)])
def test_fused_training_step_equals_separate_steps(env, P, k, b, g, p):
    """One step of THC's training process through the fused calls: every
    worker's rotated vector, the range, the wire words, the average, its
    inverse rotation and every worker's new e equal the separate calls' (the
    range within 1e-6: its sums are ordered differently, so the THC round of
    the fused chain runs on the fused range in both chains)."""
    from statistics import NormalDist

    torch, gar = env
    n = 1 << k
    rht_seed, q_seed = 0xD1A6, workloads.THC_SEED
    t_p = NormalDist().inv_cdf(1 - p / 2)
    T = _table(b, g)
    grads = [to_dev(workloads.student_t_f32(n, 4, 1e-2, 197, w), torch) for w in range(P)]
    errs = [to_dev(workloads.normal_f32(n, 1e-6, 198, w), torch) for w in range(P)]
    # fused
    ys, sums = [], []
    for w in range(P):
        y = torch.empty(n, device="cuda")
        s = torch.empty(gar.gar_rht_tiles(n), dtype=torch.float64, device="cuda")
        gar.gar_rht_ef_forward(grads[w], errs[w], y, rht_seed, s)
        ys.append(y)
        sums.append(s)
    mM = torch.empty(2, device="cuda")
    gar.gar_rht_norm_range_from_sums(sums, n, t_p, mM)
    avg = torch.empty(n, device="cuda")
    packed = [torch.empty(gar.gar_thc_words(n, b), dtype=torch.int32, device="cuda") for _ in range(P)]
    gar.gar_nuhc_allreduce_fused(ys, b, g, T, q_seed, mM, avg, packed)
    est = torch.empty(n, device="cuda")
    gar.gar_rht(avg, est, rht_seed, inverse=True)
    new_e = [e.clone() for e in errs]
    tmp = torch.empty(n, device="cuda")
    for w in range(P):
        gar.gar_rht_ef_update(packed[w], b, g, T, mM, grads[w], new_e[w], tmp, rht_seed)
    # separate calls
    xs = []
    for w in range(P):
        x = torch.empty(n, device="cuda")
        gar.gar_ef_apply(grads[w], errs[w], x)
        xs.append(x)
        y = torch.empty(n, device="cuda")
        gar.gar_rht(x, y, rht_seed)
        same_bits(to_host(y), to_host(ys[w]))
    ws = torch.empty(gar.gar_rht_norm_range_workspace_bytes(P, n) // 8, dtype=torch.float64, device="cuda")
    mM2 = torch.empty(2, device="cuda")
    gar.gar_rht_norm_range(xs, t_p, mM2, ws)
    assert abs(float(to_host(mM2)[1]) - float(to_host(mM)[1])) <= 1e-6 * float(to_host(mM)[1])
    avg2 = torch.empty(n, device="cuda")
    packed2 = [torch.empty(gar.gar_thc_words(n, b), dtype=torch.int32, device="cuda") for _ in range(P)]
    gar.gar_nuhc_allreduce_fused(ys, b, g, T, q_seed, mM, avg2, packed2)
    same_bits(to_host(avg2), to_host(avg))
    for w in range(P):
        assert torch.equal(packed2[w], packed[w])
        ref_e, _, _ = _own_chain(torch, gar, packed[w], b, g, T, mM, grads[w], errs[w], rht_seed)
        same_bits(to_host(new_e[w]), to_host(ref_e))
    # and the oracle's round on the same range and rotated vectors
    m, M = (float(v) for v in to_host(mM))
    ref_avg, ref_pk = oracle.nuhc_allreduce([to_host(y) for y in ys], b, g, T, q_seed, m, M, want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(packed[w])[: ref_pk[w].size], ref_pk[w])
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= 1e-6 * M
