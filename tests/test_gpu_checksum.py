"""GPU checksum of wire vectors (silent-data-corruption check) against the
oracle, bit-exact: random words at ragged and unaligned sizes, THC's packed
indices as the fused kernel writes them, and single-bit corruptions."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import need_cuda, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return need_cuda()


def _sum(torch, g, t):
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    g.gar_checksum(t, out)
    return int(to_host(out).view(np.uint64)[0])


@pytest.mark.parametrize("n", [0, 1, 3, 4095, 4096, 4097, 100003, 1 << 22, (1 << 26) + 16385])
def test_random_words(env, n):
    torch, g = env
    w = np.random.default_rng([7, n]).integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    t = to_dev(w.view(np.int32), torch) if n else torch.zeros(0, dtype=torch.int32, device="cuda")
    assert _sum(torch, g, t) == oracle.checksum(w)


def test_unaligned_words(env):
    torch, g = env
    w = np.random.default_rng(8).integers(0, 2**32, size=10001, dtype=np.uint64).astype(np.uint32)
    base = to_dev(w.view(np.int32), torch)
    for off in (1, 2, 3):
        assert _sum(torch, g, base[off:]) == oracle.checksum(w[off:])


def test_wire_vectors_and_corruption(env):
    torch, g = env
    P, N, b = 4, 1 << 20, 4
    xs = workloads.workers_normal(P, N, 1.0, 93)
    xd = [to_dev(x, torch) for x in xs]
    mM = torch.empty(2, device="cuda")
    avg = torch.empty(N, device="cuda")
    pk = [torch.empty(g.gar_thc_words(N, b), dtype=torch.int32, device="cuda") for _ in range(P)]
    g.gar_thc_range(xd, mM)
    g.gar_thc_allreduce_fused(xd, b, 5, mM, avg, pk)
    for w in range(P):
        host = to_host(pk[w])
        c = _sum(torch, g, pk[w])
        assert c == oracle.checksum(host)
        bad = pk[w].clone()
        bad[12345] ^= 1 << 9  # one flipped bit on the wire
        assert _sum(torch, g, bad) != c
