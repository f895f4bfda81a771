"""GPU parity of THC's pre/post-processing (THC section 5) against the oracle.

The randomized Hadamard transform runs in fp32 on the GPU and in fp64 in the
oracle.  Each butterfly stage adds at most one rounding (relative 2^-24) to
each element, and the map is orthogonal up to the final 1/sqrt(n), so the
error vector has norm at most (log2 n + 2) * 2^-24 * ||x||_2 (first order);
the tests hold the GPU to that bound.  A wrong sign or index moves the
result by O(||x||), far outside it.  The norm-based range is within 1e-6
relative of the oracle's fp64 value; the error-feedback updates are one fp32
addition or subtraction and must match numpy's IEEE fp32 bit for bit.  The
composite test runs one step of the page's THC training process (error
feedback, norm exchange in parallel with the rotation, non-uniform THC,
inverse rotation, error-feedback update) and checks every stage.
"""
import math
from statistics import NormalDist

import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def t_of_p(p):
    """Threshold with a p fraction of a standard normal outside [-t, t]."""
    return NormalDist().inv_cdf(1 - p / 2)


def rht_bound(n, norm):
    k = max(int(n).bit_length() - 1, 1)
    return (k + 2) * U * norm * 1.0001 + 1e-30


def check_rht(got, x, seed, inverse):
    ref = oracle.rht(x, seed, inverse=inverse)
    err = np.linalg.norm(got.astype(np.float64) - ref)
    bound = rht_bound(x.size, np.linalg.norm(x.astype(np.float64)))
    assert err <= bound, f"n={x.size} inverse={inverse}: error norm {err:.3e} > {bound:.3e}"


# k = 0..11 use the one-CTA kernel, 12 the tile kernel alone, 13..20 one strided
# pass (moved down below bit 12 when fewer than eight bits remain), 21..24 one
# cluster pass of 2, 4, 8 or 16 CTAs (bits 12..k-1), 25 two strided passes
@pytest.mark.parametrize("k", [0, 1, 2, 5, 7, 11, 12, 13, 15, 16, 17, 19, 20, 21, 22, 23, 24, 25])
@pytest.mark.parametrize("inverse", [False, True])
def test_rht_matches_oracle(env, k, inverse):
    torch, gar = env
    n = 1 << k
    x = workloads.normal_f32(n, 1.0, 171, k)
    out = torch.empty(n, device="cuda")
    gar.gar_rht(to_dev(x, torch), out, 0xC0FFEE + k, inverse=inverse)
    check_rht(to_host(out), x, 0xC0FFEE + k, inverse)


@pytest.mark.parametrize("k", [12, 18, 22, 24])
def test_rht_heavy_tailed_and_round_trip(env, k):
    torch, gar = env
    n = 1 << k
    x = workloads.student_t_f32(n, 3, 1e-3, 172, k)
    xd = to_dev(x, torch)
    y = torch.empty(n, device="cuda")
    gar.gar_rht(xd, y, 99)
    check_rht(to_host(y), x, 99, False)
    back = torch.empty(n, device="cuda")
    gar.gar_rht(y, back, 99, inverse=True)
    err = np.linalg.norm(to_host(back).astype(np.float64) - x)
    assert err <= 2 * rht_bound(n, np.linalg.norm(x.astype(np.float64)))
    # the rotation spreads the heavy tail: kurtosis close to a normal's
    yy = to_host(y).astype(np.float64)
    assert abs(np.mean(yy ** 4) / np.mean(yy ** 2) ** 2 - 3.0) < 0.3


@pytest.mark.parametrize("k", [3, 12, 16, 21, 24])
def test_rht_in_place_equals_out_of_place(env, k):
    torch, gar = env
    n = 1 << k
    x = to_dev(workloads.normal_f32(n, 1.0, 173, k), torch)
    for inverse in (False, True):
        out = torch.empty(n, device="cuda")
        gar.gar_rht(x, out, 5, inverse=inverse)
        y = x.clone()
        gar.gar_rht(y, y, 5, inverse=inverse)
        same_bits(to_host(y), to_host(out))


def test_rht_one_hot_and_seed_sharing(env):
    torch, gar = env
    n = 1 << 20
    for pos in (0, 1, 4095, 4096, 123457, n - 1):
        x = torch.zeros(n, device="cuda")
        x[pos] = 2.0
        y = torch.empty(n, device="cuda")
        gar.gar_rht(x, y, 11)
        # (1/sqrt n) H D e_pos = d_pos / sqrt(n) * column pos of H: every entry 2^-9 in size
        yy = to_host(y)
        assert np.all(np.abs(yy) == np.float32(2.0 / 1024))
        d = oracle.rht_signs(n, 11)
        j = np.array([0, 1, 77, 4097, n - 1])
        col = np.array([(-1) ** bin(int(jj) & pos).count("1") for jj in j])
        np.testing.assert_array_equal(np.sign(yy[j]), d[pos] * col)


def test_rht_full_size_sparse_and_round_trip(env):
    """n = 2^30 (4 GiB): three kernels.  A sparse input has an exact closed
    form at every output, checked on sampled outputs; the round trip and the
    norm hold for a dense input at the same size."""
    torch, gar = env
    n = 1 << 30
    seed = 0x5EED
    rng = np.random.default_rng(174)
    pos = np.sort(rng.choice(n, 6, replace=False))
    val = rng.standard_normal(6).astype(np.float32)
    x = torch.zeros(n, device="cuda")
    x[torch.from_numpy(pos).cuda()] = torch.from_numpy(val).cuda()
    gar.gar_rht(x, x, seed)  # in place
    j = np.concatenate([rng.choice(n, 4000, replace=False), [0, n - 1]])
    got = x[torch.from_numpy(j).cuda()].cpu().numpy().astype(np.float64)
    # signs d at the nonzeros, from the oracle's Philox: bit i mod 128 of block i / 128
    def sign_at(i):
        r = oracle.philox4x32([i >> 7, 0, 0xFFFFFFFF, 0], [seed & 0xFFFFFFFF, seed >> 32])
        return -1.0 if (int(r[(i >> 5) & 3]) >> (i & 31)) & 1 else 1.0
    assert [sign_at(i) for i in range(300)] == list(oracle.rht_signs(300, seed).astype(float))
    d = np.array([sign_at(int(q)) for q in pos])
    parity = np.array([[bin(int(jj) & int(p)).count("1") & 1 for p in pos] for jj in j])
    ref = ((1 - 2 * parity) * (d * val.astype(np.float64))).sum(axis=1) / math.sqrt(n)
    tol = (30 + 2) * U * np.linalg.norm(val.astype(np.float64)) * 1.0001
    assert np.max(np.abs(got - ref)) <= tol
    del x
    torch.cuda.empty_cache()
    xd = workloads.device_normal(n, 1.0, 175, torch.float32, "cuda")
    norm = torch.linalg.vector_norm(xd.double()).item()
    y = torch.empty_like(xd)
    gar.gar_rht(xd, y, seed)
    assert abs(torch.linalg.vector_norm(y.double()).item() - norm) <= rht_bound(n, norm)
    gar.gar_rht(y, y, seed, inverse=True)
    err = torch.linalg.vector_norm((y - xd).double()).item()
    assert err <= 2 * rht_bound(n, norm)


def test_rht_rejects_bad_arguments(env):
    torch, gar = env
    x = torch.zeros(4097, device="cuda")
    with pytest.raises(gar.GarError) as e:
        gar.gar_rht(x, torch.empty_like(x), 1)
    assert e.value.status == gar.GAR_EINVAL
    buf = torch.zeros(8192 + 4, device="cuda")
    with pytest.raises(gar.GarError) as e:
        gar.gar_rht(buf[1:4097], buf[4100:8196], 1)  # 4-byte offset
    assert e.value.status == gar.GAR_EALIGN
    with pytest.raises(gar.GarError) as e:
        gar.gar_rht(buf[:4096], buf[4:4100], 1)  # partial overlap
    assert e.value.status == gar.GAR_EINVAL


@pytest.mark.parametrize("P,n,off", [(1, 1, 0), (2, 1000, 0), (3, 4097, 1), (8, 1 << 16, 0), (64, 3001, 3),
                                     (4, (1 << 22) + 5, 0)])
def test_norm_range_matches_oracle(env, P, n, off):
    torch, gar = env
    xs = [workloads.normal_f32(n, float(w + 1), 176, w) for w in range(P)]
    store = [torch.zeros(n + off, device="cuda") for _ in range(P)]
    views = []
    for s, x in zip(store, xs):
        s[off:] = to_dev(x, torch)
        views.append(s[off:])  # off = 1, 3: not 16-byte aligned (scalar path)
    ws = torch.empty(gar.gar_rht_norm_range_workspace_bytes(P, n) // 8 + 1, dtype=torch.float64, device="cuda")
    mM = torch.empty(2, device="cuda")
    t_p = t_of_p(1 / 32)
    gar.gar_rht_norm_range(views, t_p, mM, ws)
    m, M = to_host(mM).astype(np.float64)
    rm, rM = oracle.rht_norm_range(xs, t_p)
    assert m == -M
    assert abs(M - rM) <= 1e-6 * rM


def test_norm_range_is_deterministic(env):
    torch, gar = env
    n = (1 << 20) + 3
    xs = [workloads.device_normal(n, 1.0, 177 + w, torch.float32, "cuda") for w in range(4)]
    ws = torch.empty(gar.gar_rht_norm_range_workspace_bytes(4, n) // 8, dtype=torch.float64, device="cuda")
    outs = []
    for _ in range(3):
        mM = torch.empty(2, device="cuda")
        gar.gar_rht_norm_range(xs, 2.0, mM, ws)
        outs.append(to_host(mM))
    same_bits(outs[0], outs[1])
    same_bits(outs[0], outs[2])


@pytest.mark.parametrize("n,off", [(0, 0), (1, 0), (7, 1), (4096, 0), (100003, 2), (1 << 22, 0)])
def test_error_feedback_bit_exact(env, n, off):
    torch, gar = env
    g = workloads.normal_f32(n, 1.0, 178, 0)
    e = workloads.normal_f32(n, 1e-4, 178, 1)
    xh = workloads.normal_f32(n, 1.0, 178, 2)
    def dev(a):
        s = torch.zeros(n + off, device="cuda")
        s[off:] = to_dev(a, torch)
        return s[off:]
    gd, ed, xhd = dev(g), dev(e), dev(xh)
    x = dev(np.zeros(n, np.float32))
    gar.gar_ef_apply(gd, ed, x)
    ref_x = oracle.ef_apply(g, e)
    same_bits(to_host(x), ref_x)
    gar.gar_ef_update(ed, x, xhd)  # e overwritten with x - x_hat
    ref_e = oracle.ef_update(ref_x, xh)
    same_bits(to_host(ed), ref_e)
    gar.gar_ef_apply(gd, ed, gd)  # in place on the gradient
    same_bits(to_host(gd), oracle.ef_apply(g, ref_e))


@pytest.mark.parametrize("P,k,b,g,p", [(4, 16, 4, 36, 1 / 32), (10, 18, 4, 20, 1 / 512), (3, 12, 2, 5, 1 / 32)])
def test_thc_training_step(env, P, k, b, g, p):
    """One step of THC's training process, every stage against the oracle."""
    torch, gar = env
    n = 1 << k
    rht_seed, q_seed = 0xD1A6, workloads.THC_SEED
    t_p = t_of_p(p)
    L = (1 << b) - 1
    T = np.rint(np.linspace(0, g, L + 1)).astype(np.uint16)  # evenly spread table (the pages give none)
    assert oracle.nuhc_table_ok(T, b, g)
    grads = [workloads.student_t_f32(n, 4, 1e-2, 179, w) for w in range(P)]
    errs = [workloads.normal_f32(n, 1e-6, 180, w) for w in range(P)]
    gd = [to_dev(a, torch) for a in grads]
    ed = [to_dev(a, torch) for a in errs]
    # learning step 1: x = grad + e
    xd = [torch.empty(n, device="cuda") for _ in range(P)]
    for w in range(P):
        gar.gar_ef_apply(gd[w], ed[w], xd[w])
    xs = [to_host(t) for t in xd]
    for w in range(P):
        same_bits(xs[w], grads[w] + errs[w])
    # preliminary stage (norms) alongside the rotation
    ws = torch.empty(gar.gar_rht_norm_range_workspace_bytes(P, n) // 8, dtype=torch.float64, device="cuda")
    mM = torch.empty(2, device="cuda")
    gar.gar_rht_norm_range(xd, t_p, mM, ws)
    yd = [torch.empty(n, device="cuda") for _ in range(P)]
    for w in range(P):
        gar.gar_rht(xd[w], yd[w], rht_seed)
    m, M = (float(v) for v in to_host(mM))
    rm, rM = oracle.rht_norm_range(xs, t_p)
    assert abs(M - rM) <= 1e-6 * rM and m == -M
    ys = [to_host(t) for t in yd]
    for w in range(P):
        check_rht(ys[w], xs[w], rht_seed, False)
    # about a p fraction of rotated coordinates land outside [-M, M] (truncated)
    out_frac = np.mean([np.mean(np.abs(y) > M) for y in ys])
    assert out_frac < 4 * p + 5 * math.sqrt(p / (n * P))
    # main stage: non-uniform THC on the rotated vectors (indices exact given the same inputs)
    avg = torch.empty(n, device="cuda")
    packed = [torch.empty(gar.gar_thc_words(n, b), dtype=torch.int32, device="cuda") for _ in range(P)]
    gar.gar_nuhc_allreduce_fused(yd, b, g, T, q_seed, mM, avg, packed)
    ref_avg, ref_packed = oracle.nuhc_allreduce(ys, b, g, T, q_seed, m, M, want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(packed[w])[:ref_packed[w].size], ref_packed[w])
    avg_h = to_host(avg).astype(np.float64)
    assert np.max(np.abs(avg_h - ref_avg)) <= 1e-6 * M
    # the estimate is unbiased up to the truncation: E||avg - mean y||^2 <= ||mean of the
    # clamping offsets||^2 + n * (widest grid interval)^2 / (4P)
    ys64 = np.stack(ys).astype(np.float64)
    bias = np.mean(np.clip(ys64, m, M) - ys64, axis=0)
    delta = (M - m) / g * int(np.max(np.diff(T.astype(np.int64))))
    expect = float(np.sum(bias ** 2)) + n * delta ** 2 / (4 * P)
    assert float(np.sum((avg_h - ys64.mean(axis=0)) ** 2)) <= 1.2 * expect
    # post-processing: inverse rotation of the estimate
    est = torch.empty(n, device="cuda")
    gar.gar_rht(avg, est, rht_seed, inverse=True)
    check_rht(to_host(est), to_host(avg), rht_seed, True)
    # learning step 2: e = x - x_hat, x_hat this worker's own decoded, inverse-rotated vector
    for w in range(P):
        own = torch.empty(n + 1, dtype=torch.int16, device="cuda")[:n]
        gar.gar_nuhc_aggregate([packed[w]], n, b, T, own)
        own_y = torch.empty(n, device="cuda")
        gar.gar_nuhc_decode(own, mM, g, 1, own_y)
        x_hat = torch.empty(n, device="cuda")
        gar.gar_rht(own_y, x_hat, rht_seed, inverse=True)
        ref_own = oracle.nuhc_decode(oracle.nuhc_aggregate([ref_packed[w]], n, b, T), m, M, g, 1)
        assert np.max(np.abs(to_host(own_y).astype(np.float64) - ref_own)) <= 1e-6 * M
        check_rht(to_host(x_hat), to_host(own_y), rht_seed, True)
        gar.gar_ef_update(ed[w], xd[w], x_hat)
        same_bits(to_host(ed[w]), xs[w] - to_host(x_hat))
