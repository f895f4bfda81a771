"""GPU parity of uniform THC and NMSE against the oracle.

Integer outputs (range, packed indices, index sums) are bit-exact; decoded
averages are within 1e-6 * max(|m|, |M|) of the oracle's fp64 decode (the
fp32 decode takes four roundings of at most 2^-24 of the range each); the
fused kernel equals decode(aggregate(encode)) bit for bit; NMSE is within
2e-6 relative of the oracle's fp64 sum.  Full-size THC sweep (N = 2^24,
P in {4, 16, 64}, b in {2, 4, 8}) checked on every element.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, to_dev, to_host
from oracle_par import thc_range_parallel, thc_range_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _xs(P, N, seed, scale=1.0):
    return [(np.random.default_rng([seed, P, N, w]).standard_normal(N) * scale).astype(np.float32) for w in range(P)]


def _run_range(torch, g, xd):
    mM = torch.empty(2, dtype=torch.float32, device="cuda")
    g.gar_thc_range(xd, mM)
    return mM


def _words(g, N, b, P, torch):
    return [torch.empty(max(g.gar_thc_words(N, b), 1), dtype=torch.int32, device="cuda") for _ in range(P)]


@pytest.mark.parametrize("P,N", [(1, 1), (2, 3), (4, 1000), (7, 4099), (64, 1025), (3, 1 << 18)])
def test_range(env, P, N):
    torch, g = env
    xs = _xs(P, N, 1)
    if N > 10:
        xs[P - 1][N // 2] = np.nan
    mM = to_host(_run_range(torch, g, [to_dev(x, torch) for x in xs]))
    m, M = oracle.thc_range(xs)
    assert mM[0] == m and mM[1] == M


def test_range_empty_and_unaligned(env):
    torch, g = env
    mM = to_host(_run_range(torch, g, [torch.empty(0, device="cuda")]))
    assert mM[0] == np.inf and mM[1] == -np.inf
    xs = _xs(3, 1001, 2)
    bases = [to_dev(np.concatenate([[100.0], x]).astype(np.float32), torch) for x in xs]
    mM = to_host(_run_range(torch, g, [b[1:] for b in bases]))
    m, M = oracle.thc_range(xs)
    assert mM[0] == m and mM[1] == M


@pytest.mark.parametrize("b", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [1, 5, 31, 33, 1000, 4097, 65537])
def test_encode(env, b, N):
    torch, g = env
    xs = _xs(2, N, 3)
    m, M = oracle.thc_range(xs)
    mM = torch.tensor([m, M], dtype=torch.float32, device="cuda")
    for worker, seed in ((0, 0x5EED), (1, 7), (63, (1 << 40) + 5)):
        out = _words(g, N, b, 1, torch)[0]
        g.gar_thc_encode(to_dev(xs[worker % 2], torch), mM, b, seed, worker, out)
        ref = oracle.thc_encode(xs[worker % 2], m, M, b, seed, worker)
        np.testing.assert_array_equal(to_host(out)[:ref.size], ref)


@pytest.mark.parametrize("b", [1, 2, 4, 8])
@pytest.mark.parametrize("P,N", [(1, 77), (3, 1000), (4, 4096), (8, 3001), (16, 5003), (64, 1027)])
def test_aggregate_decode_fused(env, b, P, N):
    torch, g = env
    seed = 0x5EED + P
    xs = _xs(P, N, 4)
    m, M = oracle.thc_range(xs)
    xd = [to_dev(x, torch) for x in xs]
    mM = _run_range(torch, g, xd)
    packed = _words(g, N, b, P, torch)
    for w in range(P):
        g.gar_thc_encode(xd[w], mM, b, seed, w, packed[w])
    sums = torch.empty(N, dtype=torch.int16, device="cuda")
    g.gar_thc_aggregate(packed, N, b, sums)
    avg = torch.empty(N, dtype=torch.float32, device="cuda")
    g.gar_thc_decode(sums, mM, b, P, avg)
    ref_avg, ref_packed = oracle.thc_allreduce(xs, b, seed, m, M, want_packed=True)
    ref_sums = oracle.thc_aggregate(ref_packed, N, b)
    np.testing.assert_array_equal(to_host(sums), ref_sums)
    tol = 1e-6 * max(abs(float(m)), abs(float(M)))
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= tol
    # fused: same packed words, the same avg bits as the three-kernel path
    favg = torch.empty(N, dtype=torch.float32, device="cuda")
    fpacked = _words(g, N, b, P, torch)
    g.gar_thc_allreduce_fused(xd, b, seed, mM, favg, fpacked)
    for w in range(P):
        np.testing.assert_array_equal(to_host(fpacked[w])[:ref_packed[w].size], ref_packed[w])
    np.testing.assert_array_equal(to_host(favg).view(np.uint32), to_host(avg).view(np.uint32))
    favg2 = torch.empty(N, dtype=torch.float32, device="cuda")
    g.gar_thc_allreduce_fused(xd, b, seed, mM, favg2)  # without the wire vectors
    np.testing.assert_array_equal(to_host(favg2).view(np.uint32), to_host(avg).view(np.uint32))


def test_worked_example_and_degenerate(env):
    torch, g = env
    # b = 2 on [-1, 1]: T0 = {-1, -1/3, 1/3, 1}; index sum 3 over 2 workers -> 0
    mM = torch.tensor([-1.0, 1.0], device="cuda")
    sums = torch.tensor([0, 1, 2, 3], dtype=torch.int16, device="cuda")
    avg = torch.empty(4, device="cuda")
    g.gar_thc_decode(sums, mM, 2, 1, avg)
    np.testing.assert_allclose(to_host(avg), [-1, -1 / 3, 1 / 3, 1], rtol=0, atol=2e-7)
    # (exactly 0 in real arithmetic; the fp32 decode fma(3, (2/3)/2, -1) is
    # within its stated bound of 1e-6 * max(|m|, |M|))
    g.gar_thc_decode(torch.tensor([3, 3], dtype=torch.int16, device="cuda"), mM, 2, 2, avg[:2])
    assert np.all(np.abs(to_host(avg[:2])) <= 1e-6)
    # on-grid inputs: index == value on [0, L], whatever the seed
    for b in (1, 2, 4, 8):
        L = (1 << b) - 1
        x = np.tile(np.arange(L + 1, dtype=np.float32), 5)
        out = _words(g, x.size, b, 1, torch)[0]
        g.gar_thc_encode(to_dev(x, torch), torch.tensor([0.0, float(L)], device="cuda"), b, 99, 3, out)
        np.testing.assert_array_equal(oracle.thc_unpack(to_host(out), x.size, b), x.astype(np.uint8))
    # M == m: every index 0, the average is m
    x = np.full(100, 0.5, np.float32)
    xd = [to_dev(x, torch) for _ in range(3)]
    mM = _run_range(torch, g, xd)
    favg = torch.empty(100, device="cuda")
    pk = _words(g, 100, 4, 3, torch)
    g.gar_thc_allreduce_fused(xd, 4, 1, mM, favg, pk)
    assert np.all(to_host(favg) == 0.5)
    assert all(np.all(to_host(p) == 0) for p in pk)


def test_unaligned_inputs(env):
    torch, g = env
    P, N, b, seed = 3, 3001, 4, 11
    xs = _xs(P, N, 5)
    m, M = oracle.thc_range(xs)
    bases = [to_dev(np.concatenate([[0.0], x]).astype(np.float32), torch) for x in xs]
    xd = [t[1:] for t in bases]
    mM = torch.tensor([m, M], device="cuda")
    favg_base = torch.empty(N + 1, device="cuda")
    favg = favg_base[1:]
    pk = _words(g, N, b, P, torch)
    g.gar_thc_allreduce_fused(xd, b, seed, mM, favg, pk)
    ref_avg, ref_packed = oracle.thc_allreduce(xs, b, seed, m, M, want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(pk[w])[:ref_packed[w].size], ref_packed[w])
    assert np.max(np.abs(to_host(favg).astype(np.float64) - ref_avg)) <= 1e-6 * max(abs(m), abs(M))


def test_partition_4mb_full(env):
    # P=4, N = 2^20 fp32 N(0, 1), b = 4 on the global [min, max]: full compare
    torch, g = env
    P, N, b, seed = 4, 1 << 20, 4, workloads.THC_SEED
    xs = workloads.workers_normal(P, N, 1.0, workloads.CONFIG_IDS["partition_4mb"])
    m, M = oracle.thc_range(xs)
    xd = [to_dev(x, torch) for x in xs]
    mM = _run_range(torch, g, xd)
    assert to_host(mM).tolist() == [m, M]
    avg = torch.empty(N, device="cuda")
    pk = _words(g, N, b, P, torch)
    g.gar_thc_allreduce_fused(xd, b, seed, mM, avg, pk)
    ref_avg, ref_packed = oracle.thc_allreduce(xs, b, seed, m, M, want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(pk[w]), ref_packed[w])
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= 1e-6 * max(abs(m), abs(M))
    # NMSE of the estimate against the exact average
    exact = np.mean(np.stack(xs).astype(np.float64), axis=0)
    ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8, dtype=torch.float64, device="cuda")
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    ex32 = exact.astype(np.float32)
    g.gar_nmse(to_dev(ex32, torch), avg, out, ws)
    ref = oracle.nmse(ex32, to_host(avg))
    assert abs(out.item() - ref) <= 2e-6 * ref


@pytest.fixture(scope="module")
def sweep_inputs(env):
    """The THC sweep's gradients for one worker count at a time: N = 2^24
    fp32 Student-t(3) x 1e-3 per worker, on the device and on the host."""
    torch, g = env
    cache = {}

    def get(P):
        if P not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            xd = [workloads.device_student_t(1 << 24, 3, 1e-3, 40_000 + 100 * P + w, "cuda") for w in range(P)]
            cache[P] = (xd, [to_host(x) for x in xd])
        return cache[P]

    yield get
    cache.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("P", [4, 16, 64])
def test_thc_sweep_full_size(env, sweep_inputs, P, b):
    # N = 2^24 per worker, shared [m, M]: the range, every worker's every
    # index (through its wire words) and every averaged value against the
    # oracle, in the launches the benchmark times
    torch, g = env
    N, seed = 1 << 24, workloads.THC_SEED
    xd, xh = sweep_inputs(P)
    mM = _run_range(torch, g, xd)
    m, M = thc_range_parallel(xh)
    assert to_host(mM).tolist() == [m, M]
    avg = torch.empty(N, device="cuda")
    pk = _words(g, N, b, P, torch)
    g.gar_thc_allreduce_fused(xd, b, seed, mM, avg, pk)
    got_avg = to_host(avg).astype(np.float64)
    got_pk = [to_host(t) for t in pk]
    tol = 1e-6 * max(abs(float(m)), abs(float(M)))
    chunk = 1 << 21
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        ref_idx, ref_avg = thc_range_samples(np.stack([x[lo:hi] for x in xh]), lo, b, seed, m, M)
        w0, w1 = lo * b // 32, hi * b // 32
        for w in range(P):
            np.testing.assert_array_equal(oracle.thc_unpack(got_pk[w][w0:w1], hi - lo, b), ref_idx[w],
                                          err_msg=f"worker {w}, elements {lo}..{hi}")
        err = np.max(np.abs(got_avg[lo:hi] - ref_avg))
        assert err <= tol, (lo, err, tol)
    # separate kernels agree with the fused one everywhere
    sums = torch.empty(N, dtype=torch.int16, device="cuda")
    g.gar_thc_aggregate(pk, N, b, sums)
    avg2 = torch.empty(N, device="cuda")
    g.gar_thc_decode(sums, mM, b, P, avg2)
    assert torch.equal(avg2.view(torch.int32), avg.view(torch.int32))
    enc = torch.empty_like(pk[P - 1])
    g.gar_thc_encode(xd[P - 1], mM, b, seed, P - 1, enc)
    assert torch.equal(enc, pk[P - 1])
    del pk
    torch.cuda.empty_cache()


@pytest.mark.parametrize("arrived", [0b11111111, 0b10110101, 0b00001000, 0b11111110])
@pytest.mark.parametrize("b", [2, 4, 8])
def test_straggler_masked(env, arrived, b):
    # stragglers dropped: only arrived workers encode (own ids) and sum, decode by their count
    torch, g = env
    P, N, seed = 8, 20011, 4242
    xs = _xs(P, N, 9)
    ids = [w for w in range(P) if (arrived >> w) & 1]
    m, M = oracle.thc_range([xs[w] for w in ids])
    mM = torch.tensor([m, M], device="cuda")
    xd = [to_dev(x, torch) if w in ids else None for w, x in enumerate(xs)]
    pk = [torch.zeros(g.gar_thc_words(N, b), dtype=torch.int32, device="cuda") if w in ids else None for w in range(P)]
    avg = torch.empty(N, device="cuda")
    g.gar_thc_allreduce_fused_masked(xd, arrived, b, seed, mM, avg, pk)
    ref_avg, ref_pk = oracle.thc_allreduce_masked(xs, arrived, b, seed, m, M, want_packed=True)
    for w in ids:
        np.testing.assert_array_equal(to_host(pk[w]), ref_pk[w])
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= 1e-6 * max(abs(m), abs(M))
    # the same as the separate kernels over the arrived workers' vectors
    sums = torch.empty(N, dtype=torch.int16, device="cuda")
    g.gar_thc_aggregate([pk[w] for w in ids], N, b, sums)
    avg2 = torch.empty(N, device="cuda")
    g.gar_thc_decode(sums, mM, b, len(ids), avg2)
    assert torch.equal(avg.view(torch.int32), avg2.view(torch.int32))
    if arrived == (1 << P) - 1:  # everyone arrived: the unmasked kernel, bit for bit
        avg3 = torch.empty(N, device="cuda")
        g.gar_thc_allreduce_fused(xd, b, seed, mM, avg3)
        assert torch.equal(avg.view(torch.int32), avg3.view(torch.int32))


def test_straggler_mask_rejects_no_arrivals(env):
    torch, g = env
    x = [torch.zeros(8, device="cuda")]
    with pytest.raises(g.GarError):
        g.gar_thc_allreduce_fused_masked(x, 0, 4, 1, torch.zeros(2, device="cuda"), torch.empty(8, device="cuda"))


@pytest.mark.parametrize("N", [1, 3, 4, 1000, 4097, 1 << 20])
def test_nmse(env, N):
    torch, g = env
    x = _xs(1, N, 6)[0]
    xh = (x + _xs(1, N, 7, 0.05)[0]).astype(np.float32)
    ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8, dtype=torch.float64, device="cuda")
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    g.gar_nmse(to_dev(x, torch), to_dev(xh, torch), out, ws)
    ref = oracle.nmse(x, xh)
    assert abs(out.item() - ref) <= 2e-6 * ref
    g.gar_nmse(to_dev(np.zeros(N, np.float32), torch), to_dev(xh, torch), out, ws)
    assert np.isnan(out.item())
    with pytest.raises(g.GarError):
        g.gar_nmse(to_dev(x, torch), to_dev(xh, torch), out, ws[:0])


@pytest.mark.parametrize("cuts", [(0, 1000), (0, 1, 4097, 4100, 70001), (0, 3, 4, 65536, 65537, 100000)])
def test_nmse_sums_over_ranges(env, cuts):
    """NMSE of a vector held in several ranges (one per fusion buffer, or per
    device): the ranges' pairs of sums, combined, match the oracle's NMSE of
    the whole vector; one range combined alone equals gar_nmse bit for bit."""
    torch, g = env
    N = cuts[-1]
    x = _xs(1, N, 8)[0]
    xh = (x + _xs(1, N, 9, 0.05)[0]).astype(np.float32)
    xd, hd = to_dev(x, torch), to_dev(xh, torch)
    ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8, dtype=torch.float64, device="cuda")
    pairs = torch.full((len(cuts) - 1, 2), float("nan"), dtype=torch.float64, device="cuda")
    for k in range(len(cuts) - 1):
        lo, hi = cuts[k], cuts[k + 1]
        g.gar_nmse_sums(xd[lo:hi], hd[lo:hi], pairs[k], ws)
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    g.gar_nmse_combine(pairs, out)
    ref = oracle.nmse(x, xh)
    assert abs(out.item() - ref) <= 2e-6 * ref
    # each pair's sums against fp64 sums of the same range
    p = pairs.cpu().numpy()
    for k in range(len(cuts) - 1):
        lo, hi = cuts[k], cuts[k + 1]
        d = x[lo:hi].astype(np.float64) - xh[lo:hi].astype(np.float64)
        assert abs(p[k, 0] - np.sum(d * d)) <= 2e-6 * np.sum(d * d) + 1e-300
        assert abs(p[k, 1] - np.sum(x[lo:hi].astype(np.float64) ** 2)) <= 2e-6 * np.sum(x[lo:hi].astype(np.float64) ** 2)
    # a single range, combined, is gar_nmse's result exactly
    whole = torch.empty(1, dtype=torch.float64, device="cuda")
    g.gar_nmse(xd, hd, whole, ws)
    one = torch.empty((1, 2), dtype=torch.float64, device="cuda")
    g.gar_nmse_sums(xd, hd, one[0], ws)
    g.gar_nmse_combine(one, out)
    assert out.item() == whole.item()
    with pytest.raises(g.GarError):
        g.gar_nmse_combine(pairs[:0], out)
