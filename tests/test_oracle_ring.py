"""Pins for the oracle's ring all-reduce (CPU only).

Each test checks the oracle against something other than itself: the worked
demo of the ring-simulator page, the schedule's step and volume invariants
stated on two pages, exact integer arithmetic, a hand-derived fp32 ordering
example, the textbook summation error bound, and torch's bf16 rounding.
"""
import json
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_demo_p4_k8(golden_dir):
    g = _load(golden_dir, "ring_demo_p4_k8.json")
    for op, key in ((oracle.SUM, "sum"), (oracle.AVG, "avg")):
        bufs = [np.array(row, np.float32) for row in g["inputs"]]
        steps, sent = oracle.ring_schedule(bufs, op=op)
        assert steps == g["steps"]
        assert all(int(s) * g["elem_bytes"] == g["bytes_sent_per_worker"] for s in sent)
        for b in bufs:
            np.testing.assert_array_equal(b, np.array(g[key], np.float32))
        fold = oracle.ring_fold([np.array(r, np.float32) for r in g["inputs"]], op=op)
        np.testing.assert_array_equal(fold, np.array(g[key], np.float32))


def test_demo_chunk_ownership_after_scatter_reduce(golden_dir):
    # both pages: after the p-1 scatter-reduce steps worker i holds the full
    # sum of chunk (i + 1) mod p
    g = _load(golden_dir, "ring_demo_p4_k8.json")
    bufs = [np.array(row, np.float32) for row in g["inputs"]]
    steps, _ = oracle.ring_schedule(bufs, op=oracle.SUM, phases=1)
    assert steps == g["P"] - 1
    full = np.array(g["sum"], np.float32)
    clen = g["K"] // g["P"]
    for i, c in enumerate(g["chunk_owned_after_scatter_reduce"]):
        assert c == (i + 1) % g["P"]
        np.testing.assert_array_equal(bufs[i][c * clen:(c + 1) * clen], full[c * clen:(c + 1) * clen])


def test_fp32_order_example(golden_dir):
    g = _load(golden_dir, "ring_order_p3.json")
    P = g["P"]
    xs = [np.full(3, v, np.float32) for v in g["worker_values"]]
    np.testing.assert_array_equal(oracle.ring_fold(xs, op=oracle.SUM), np.array(g["sum"], np.float32))
    bufs = [x.copy() for x in xs]
    oracle.ring_schedule(bufs, op=oracle.SUM)
    for b in bufs:
        np.testing.assert_array_equal(b, np.array(g["sum"], np.float32))
    assert g["sum"] != g["sum_reversed_ring"] and g["sum"] != g["sum_fixed_start"]
    avg = oracle.ring_fold(xs, op=oracle.AVG)
    np.testing.assert_array_equal(avg, np.array(g["sum"], np.float32) / np.float32(P))


@pytest.mark.parametrize("P", [2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("mult", [1, 3, 1000])
def test_step_and_volume_invariants(P, mult):
    N = P * mult
    bufs = [np.random.default_rng([7, w]).standard_normal(N, dtype=np.float32) for w in range(P)]
    steps, sent = oracle.ring_schedule(bufs, op=oracle.AVG)
    assert steps == 2 * (P - 1)
    # 2 (P - 1) / P * N elements per worker when P divides N
    assert all(int(s) * P == 2 * (P - 1) * N for s in sent)


def test_volume_ragged():
    # P does not divide N: trailing chunks are short or empty; each worker still
    # sends one chunk per step, 2(P-1) steps
    P, N = 4, 10  # chunks of ceil(10/4)=3: [0,3) [3,6) [6,9) [9,10)
    bufs = [np.arange(N, dtype=np.float32) + w for w in range(P)]
    steps, sent = oracle.ring_schedule(bufs, op=oracle.SUM)
    assert steps == 6
    assert int(sent.sum()) == 2 * (P - 1) * N


@pytest.mark.parametrize("P", [1, 2, 3, 4, 7, 16, 64])
def test_integer_inputs_sum_exactly(P):
    # integer-valued fp32 inputs with small magnitudes add exactly in any order
    N = 257
    g = np.random.default_rng([11, P])
    ints = g.integers(-1000, 1000, size=(P, N))
    xs = [row.astype(np.float32) for row in ints]
    np.testing.assert_array_equal(oracle.ring_fold(xs, op=oracle.SUM), ints.sum(0).astype(np.float32))
    bufs = [x.copy() for x in xs]
    oracle.ring_schedule(bufs, op=oracle.SUM)
    for b in bufs:
        np.testing.assert_array_equal(b, ints.sum(0).astype(np.float32))


def test_p1_is_identity():
    x = np.random.default_rng(3).standard_normal(33, dtype=np.float32)
    np.testing.assert_array_equal(oracle.ring_fold([x], op=oracle.AVG), x)
    b = [x.copy()]
    steps, sent = oracle.ring_schedule(b, op=oracle.AVG)
    assert steps == 0 and int(sent[0]) == 0
    np.testing.assert_array_equal(b[0], x)


def test_p2_is_plain_add():
    g = np.random.default_rng(5)
    x0, x1 = g.standard_normal(101, dtype=np.float32), g.standard_normal(101, dtype=np.float32)
    np.testing.assert_array_equal(oracle.ring_fold([x0, x1], op=oracle.SUM), x0 + x1)


def test_brute_force_schedule_equals_fold():
    # every P <= 4 and N <= 64 (N < P, P not dividing N included), random floats
    for P in range(1, 5):
        for N in range(0, 65):
            xs = [np.random.default_rng([P, N, w]).standard_normal(N, dtype=np.float32) * 10 ** w
                  for w in range(P)]
            for op in (oracle.SUM, oracle.AVG):
                bufs = [x.copy() for x in xs]
                steps, sent = oracle.ring_schedule(bufs, op=op)
                assert steps == 2 * (P - 1)
                fold = oracle.ring_fold(xs, op=op)
                for b in bufs:
                    np.testing.assert_array_equal(b.view(np.uint32), fold.view(np.uint32))


def test_fold_within_recursive_summation_bound():
    # |fl(sum) - sum| <= (P - 1) u sum|x_i| (+ O(u^2)), u = 2^-24, for any order
    P, N = 16, 4096
    xs = [np.random.default_rng([13, w]).standard_normal(N, dtype=np.float32) for w in range(P)]
    s = oracle.ring_fold(xs, op=oracle.SUM).astype(np.float64)
    exact = np.sum(np.stack(xs).astype(np.float64), axis=0)
    bound = (P - 1) * 2.0 ** -24 * np.sum(np.abs(np.stack(xs).astype(np.float64)), axis=0) * 1.0001
    assert np.all(np.abs(s - exact) <= bound)
    # the fold is not just any order: the per-element start rotates with the chunk
    fixed = xs[0].copy()
    for w in range(1, P):
        fixed = fixed + xs[w]
    assert not np.array_equal(fixed, oracle.ring_fold(xs, op=oracle.SUM))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(17)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(2000) * 1e30).astype(np.float32),
        (g.standard_normal(2000) * 1e-38).astype(np.float32),
        # exact ties: low 16 bits 0x8000 with even and odd upper halves
        (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38], np.float32),
    ])
    vals = vals[np.isfinite(vals) | np.isinf(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.f32_to_bf16(v) for v in vals], np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(oracle.f32_to_bf16_array(vals), ref)
    assert np.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16(np.float32("nan"))))


@pytest.mark.parametrize("P,N", [(3, 50), (4, 64), (16, 1000)])
def test_bf16_fold_and_schedule(P, N):
    torch = pytest.importorskip("torch")
    xs32 = [np.random.default_rng([19, w]).standard_normal(N, dtype=np.float32) * 0.1 for w in range(P)]
    xs = [torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for x in xs32]
    out, f32 = oracle.ring_fold(xs, op=oracle.AVG, return_f32=True)
    bufs = [x.copy() for x in xs]
    steps, _ = oracle.ring_schedule(bufs, op=oracle.AVG)
    assert steps == 2 * (P - 1)
    for b in bufs:
        np.testing.assert_array_equal(b, out)
    # widened inputs, exact fp64 average, fp32 partials within the summation
    # bound and the bf16 output within half a bf16 ulp of the fp32 value
    wide = np.stack([torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy() for x in xs])
    exact = wide.astype(np.float64).mean(0)
    bound = (P + 1) * 2.0 ** -24 * np.abs(wide.astype(np.float64)).sum(0) / P * 1.001
    assert np.all(np.abs(f32.astype(np.float64) - exact) <= bound)
    back = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.all(np.abs(back - f32) <= np.abs(f32) * 2.0 ** -8 + 1e-38)


def test_fold_at_matches_full():
    P, N = 5, 1001
    xs = [np.random.default_rng([23, w]).standard_normal(N, dtype=np.float32) for w in range(P)]
    full = oracle.ring_fold(xs, op=oracle.AVG)
    idx = np.array([0, 1, 200, 201, 999, 1000, 600], np.int64)
    np.testing.assert_array_equal(oracle.ring_fold_at(xs, N, idx, op=oracle.AVG), full[idx])


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.ring_schedule([np.zeros(4, np.float32)], op=7)


def test_all_chunk_rotations_seen():
    # P=4, N=8 (chunks of 2).  Worker w_big holds 2^24, the others 1.0.  In
    # fp32 (ulp 2 above 2^24, ties to even): with 0 or 1 ones added before the
    # big value the result is 2^24; with 2 or 3 ones first it is 2^24 + 4.
    # Chunk c adds (w_big - c) mod 4 ones before the big value.
    P, N = 4, 8
    for w_big in range(P):
        xs = [np.ones(N, np.float32) for _ in range(P)]
        xs[w_big][:] = 2.0 ** 24
        s = oracle.ring_fold(xs, op=oracle.SUM)
        for c in range(P):
            before = (w_big - c) % P
            expect = 2.0 ** 24 if before <= 1 else 2.0 ** 24 + 4
            np.testing.assert_array_equal(s[2 * c:2 * c + 2], np.full(2, expect, np.float32))


def test_samples_match_full_fold():
    torch = pytest.importorskip("torch")
    P, N = 6, 5003
    xs = [np.random.default_rng([71, w]).standard_normal(N, dtype=np.float32) for w in range(P)]
    idx = np.array([0, 1, 833, 834, 835, 4000, 5002], np.int64)
    full = oracle.ring_fold(xs, op=oracle.AVG)
    vals = np.stack([x[idx] for x in xs])
    np.testing.assert_array_equal(oracle.ring_fold_samples(vals, N, idx), full[idx])
    hb = [torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for x in xs]
    fullb = oracle.ring_fold(hb, op=oracle.AVG)
    valsb = np.stack([h[idx] for h in hb])
    np.testing.assert_array_equal(oracle.ring_fold_samples(valsb, N, idx), fullb[idx])
