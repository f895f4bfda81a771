"""GPU parity of non-uniform THC (THC section 5, Algorithm 2) against the oracle.

Indices and table-value sums bit-exact; decoded averages within
1e-6 * max(|m|, |M|) of the oracle's fp64 decode; the fused kernel equals
decode(aggregate(encode)) bit for bit; the identity table with g = 2^b - 1
equals the uniform THC kernels bit for bit; the page's T2 example; a
full-size run with the page's simulation setting (b = 4, g = 36), every
element against the oracle.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle_par import pmap, runs, thc_range_parallel
from helpers import need_cuda, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def s_curve_table(b, g):
    """A valid table (strictly increasing, 0 .. g) denser near the middle."""
    L = (1 << b) - 1
    z = np.arange(L + 1) / L * 2 - 1
    raw = np.rint(g / 2 + g / 2 * np.sign(z) * np.abs(z) ** 1.6).astype(np.int64)
    raw[0], raw[-1] = 0, g
    for i in range(1, L):  # repair ties from rounding; the ends stay 0 and g
        raw[i] = max(raw[i], raw[i - 1] + 1)
    for i in range(L - 1, -1, -1):
        raw[i] = min(raw[i], raw[i + 1] - 1)
    assert oracle.nuhc_table_ok(raw, b, g)
    return raw.astype(np.uint16)


def _xs(P, N, seed):
    return [np.random.default_rng([seed, P, N, w]).standard_normal(N).astype(np.float32) for w in range(P)]


def _words(g, N, b, P, torch):
    return [torch.empty(max(g.gar_thc_words(N, b), 1), dtype=torch.int32, device="cuda") for _ in range(P)]


CASES = [(1, 1), (1, 5), (2, 3), (2, 4), (2, 17), (4, 15), (4, 36), (4, 51), (4, 4000), (8, 255), (8, 1000),
         (8, 1023), (8, 1024)]


@pytest.mark.parametrize("b,g", CASES)
@pytest.mark.parametrize("P,N", [(1, 77), (3, 1001), (8, 4096), (16, 2049)])
def test_encode_aggregate_decode_fused(env, b, g, P, N):
    torch, gar = env
    if P * g > 65535:
        pytest.skip("sum would overflow 16 bits")
    T = s_curve_table(b, g)
    seed = 0x5EED + g
    xs = _xs(P, N, 121)
    m, M = oracle.thc_range(xs)
    xd = [to_dev(x, torch) for x in xs]
    mM = torch.tensor([m, M], dtype=torch.float32, device="cuda")
    packed = _words(gar, N, b, P, torch)
    for w in range(P):
        gar.gar_nuhc_encode(xd[w], mM, b, g, T, seed, w, packed[w])
    sums = torch.empty(N + 1, dtype=torch.int16, device="cuda")[:N]
    gar.gar_nuhc_aggregate(packed, N, b, T, sums)
    avg = torch.empty(N, device="cuda")
    gar.gar_nuhc_decode(sums, mM, g, P, avg)
    ref_avg, ref_packed = oracle.nuhc_allreduce(xs, b, g, T, seed, m, M, want_packed=True)
    for w in range(P):
        np.testing.assert_array_equal(to_host(packed[w])[:ref_packed[w].size], ref_packed[w])
    np.testing.assert_array_equal(to_host(sums), oracle.nuhc_aggregate(ref_packed, N, b, T))
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= 1e-6 * max(abs(m), abs(M))
    favg = torch.empty(N, device="cuda")
    fpk = _words(gar, N, b, P, torch)
    gar.gar_nuhc_allreduce_fused(xd, b, g, T, seed, mM, favg, fpk)
    for w in range(P):
        np.testing.assert_array_equal(to_host(fpk[w])[:ref_packed[w].size], ref_packed[w])
    np.testing.assert_array_equal(to_host(favg).view(np.uint32), to_host(avg).view(np.uint32))


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_identity_table_equals_uniform_kernels(env, b):
    torch, gar = env
    L = (1 << b) - 1
    T = np.arange(L + 1, dtype=np.uint16)
    P, N, seed = 5, 10007, 99
    xd = [to_dev(x, torch) for x in _xs(P, N, 122)]
    mM = torch.empty(2, device="cuda")
    gar.gar_thc_range(xd, mM)
    u_avg, n_avg = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    u_pk, n_pk = _words(gar, N, b, P, torch), _words(gar, N, b, P, torch)
    gar.gar_thc_allreduce_fused(xd, b, seed, mM, u_avg, u_pk)
    gar.gar_nuhc_allreduce_fused(xd, b, L, T, seed, mM, n_avg, n_pk)
    assert torch.equal(u_avg.view(torch.int32), n_avg.view(torch.int32))
    for a, c in zip(u_pk, n_pk):
        assert torch.equal(a, c)


def test_t2_example(env, golden_dir):
    torch, gar = env
    d = json.load(open(os.path.join(golden_dir, "nuhc_t2_example.json")))
    b, g, T = d["b"], d["g"], np.array(d["table"], np.uint16)
    mM = torch.tensor([d["m"], d["M"]], device="cuda")
    for case in d["cases"]:
        xd = [torch.tensor([float(Fraction(q))], device="cuda") for q in case["quantized"]]
        pk = _words(gar, 1, b, len(xd), torch)
        avg = torch.empty(1, device="cuda")
        gar.gar_nuhc_allreduce_fused(xd, b, g, T, 7, mM, avg, pk)
        assert [int(to_host(p)[0]) for p in pk] == case["indices"]
        sums = torch.empty(2, dtype=torch.int16, device="cuda")[:1]
        gar.gar_nuhc_aggregate(pk, 1, b, T, sums)
        assert int(to_host(sums)[0]) == case["table_sum"]
        assert abs(to_host(avg)[0] - float(Fraction(d["average_for_table_sum_3"]))) <= 1e-6


def test_degenerate_and_errors(env):
    torch, gar = env
    T = s_curve_table(4, 36)
    x = np.full(50, 0.25, np.float32)
    xd = [to_dev(x, torch) for _ in range(3)]
    mM = torch.empty(2, device="cuda")
    gar.gar_thc_range(xd, mM)
    avg = torch.empty(50, device="cuda")
    pk = _words(gar, 50, 4, 3, torch)
    gar.gar_nuhc_allreduce_fused(xd, 4, 36, T, 1, mM, avg, pk)
    assert np.all(to_host(avg) == 0.25) and all(np.all(to_host(p) == 0) for p in pk)
    bad = T.copy()
    bad[3] = bad[2]
    with pytest.raises(gar.GarError):
        gar.gar_nuhc_allreduce_fused(xd, 4, 36, bad, 1, mM, avg, pk)
    with pytest.raises(gar.GarError):
        gar.gar_nuhc_allreduce_fused(xd, 4, 40, T, 1, mM, avg, pk)  # T ends at 36, not 40


@pytest.mark.parametrize("P", [4, 16])
def test_sweep_shape_full_size(env, P):
    # N = 2^24 Student-t(3) x 1e-3, b = 4 with granularity 36 (the page's
    # simulation setting): every worker's every index (through its wire
    # words) and every averaged value against the oracle
    torch, gar = env
    b, g, N, seed = 4, 36, 1 << 24, workloads.THC_SEED
    T = s_curve_table(b, g)
    xd = [workloads.device_student_t(N, 3, 1e-3, 50_000 + 100 * P + w, "cuda") for w in range(P)]
    xh = [to_host(x) for x in xd]
    mM = torch.empty(2, device="cuda")
    gar.gar_thc_range(xd, mM)
    m, M = thc_range_parallel(xh)
    assert to_host(mM).tolist() == [m, M]
    avg = torch.empty(N, device="cuda")
    pk = _words(gar, N, b, P, torch)
    gar.gar_nuhc_allreduce_fused(xd, b, g, T, seed, mM, avg, pk)
    got_avg = to_host(avg).astype(np.float64)
    got_pk = [to_host(t) for t in pk]
    tol = 1e-6 * max(abs(float(m)), abs(float(M)))
    per = 32 // b
    chunk = 1 << 20
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        runs_ = [(w, a, z) for w in range(P) for a, z in runs(lo, hi, 4)]
        words = pmap(lambda r: (r, oracle.nuhc_encode_at(xh[r[0]][r[1]:r[2]], r[1], m, M, b, g, T, seed, r[0])),
                     runs_)
        ref_pk = [np.concatenate([wd for (w, a, z), wd in words if w == k]) for k in range(P)]
        for w in range(P):
            np.testing.assert_array_equal(got_pk[w][lo // per:hi // per], ref_pk[w], err_msg=f"worker {w} at {lo}")
        ref_avg = oracle.nuhc_decode(oracle.nuhc_aggregate(ref_pk, hi - lo, b, T), m, M, g, P)
        err = np.max(np.abs(got_avg[lo:hi] - ref_avg))
        assert err <= tol, (lo, err, tol)
    del xd, pk
    torch.cuda.empty_cache()


@pytest.mark.parametrize("P,arrived", [(8, 0b11111111), (8, 0b10110110), (8, 0b00000001), (16, 0xF0F0),
                                       (5, 0b10110), (4, 0b1111)])
@pytest.mark.parametrize("b,g", [(4, 36), (2, 9), (8, 300)])
def test_straggler_masked(env, P, arrived, b, g):
    """Stragglers dropped with non-uniform THC: only the arrived workers
    encode, under their own ids, and their table values are summed; the
    decode divides by their number.  Against the oracle's encode of the arrived
    workers (own ids) -> aggregate -> decode; equal to the separate kernels
    over their vectors; all arrived = the unmasked kernel bit for bit (the
    kernels built for 4, 8 or 16 workers, which key Philox by the slot)."""
    torch, gar = env
    N, seed = 20011, 4343
    T = s_curve_table(b, g)
    xs = _xs(P, N, 131)
    ids = [w for w in range(P) if (arrived >> w) & 1]
    m, M = oracle.thc_range([xs[w] for w in ids])
    mM = torch.tensor([m, M], dtype=torch.float32, device="cuda")
    xd = [to_dev(x, torch) if w in ids else None for w, x in enumerate(xs)]
    pk = [torch.zeros(max(gar.gar_thc_words(N, b), 1), dtype=torch.int32, device="cuda") if w in ids else None
          for w in range(P)]
    avg = torch.empty(N, device="cuda")
    gar.gar_nuhc_allreduce_fused_masked(xd, arrived, b, g, T, seed, mM, avg, pk)
    ref_pk = {w: oracle.nuhc_encode(xs[w], m, M, b, g, T, seed, w) for w in ids}
    for w in ids:
        np.testing.assert_array_equal(to_host(pk[w])[:ref_pk[w].size], ref_pk[w], err_msg=f"worker {w}")
    ref_avg = oracle.nuhc_decode(oracle.nuhc_aggregate([ref_pk[w] for w in ids], N, b, T), m, M, g, len(ids))
    assert np.max(np.abs(to_host(avg).astype(np.float64) - ref_avg)) <= 1e-6 * max(abs(m), abs(M))
    sums = torch.empty(N + 1, dtype=torch.int16, device="cuda")[:N]
    gar.gar_nuhc_aggregate([pk[w] for w in ids], N, b, T, sums)
    avg2 = torch.empty(N, device="cuda")
    gar.gar_nuhc_decode(sums, mM, g, len(ids), avg2)
    assert torch.equal(avg.view(torch.int32), avg2.view(torch.int32))
    if arrived == (1 << P) - 1:
        avg3 = torch.empty(N, device="cuda")
        pk3 = _words(gar, N, b, P, torch)
        gar.gar_nuhc_allreduce_fused(xd, b, g, T, seed, mM, avg3, pk3)
        assert torch.equal(avg.view(torch.int32), avg3.view(torch.int32))
        for w in range(P):
            assert torch.equal(pk[w], pk3[w])


def test_straggler_masked_rejects(env):
    torch, gar = env
    T = s_curve_table(4, 36)
    x = [torch.zeros(64, device="cuda") for _ in range(3)]
    mM = torch.zeros(2, device="cuda")
    with pytest.raises(gar.GarError):  # nobody arrived
        gar.gar_nuhc_allreduce_fused_masked(x, 0, 4, 36, T, 1, mM, torch.empty(64, device="cuda"))
    with pytest.raises(gar.GarError):  # an arrived worker without input
        gar.gar_nuhc_allreduce_fused_masked([x[0], None, x[2]], 0b111, 4, 36, T, 1, mM,
                                            torch.empty(64, device="cuda"))
    big = [torch.zeros(64, device="cuda") for _ in range(64)]
    with pytest.raises(gar.GarError):  # 64 arrived x g = 4000 overflows the 16-bit sums
        gar.gar_nuhc_allreduce_fused_masked(big, ~0 & ((1 << 64) - 1), 4, 4000, s_curve_table(4, 4000), 1, mM,
                                            torch.empty(64, device="cuda"))
