"""Pins of the oracle's wire-vector checksum: values worked by hand, the
mod-2^32 wrap, and the corruptions it must reveal (a flipped bit, two
swapped words)."""
import numpy as np

import oracle


def test_hand_values():
    assert oracle.checksum([]) == 0
    assert oracle.checksum([1, 2, 3]) == (14 << 32) | 6  # s1 = 6, s2 = 1*1 + 2*2 + 3*3
    assert oracle.checksum([0xFFFFFFFF, 1]) == (((0xFFFFFFFF + 2) % 2**32) << 32) | 0  # both sums wrap


def test_against_python_integers():
    w = np.random.default_rng(5).integers(0, 2**32, size=10007, dtype=np.uint64).astype(np.uint32)
    s1 = int(sum(int(v) for v in w)) % 2**32
    s2 = int(sum((i + 1) * int(v) for i, v in enumerate(w))) % 2**32
    assert oracle.checksum(w) == (s2 << 32) | s1


def test_reveals_flips_and_swaps():
    rng = np.random.default_rng(6)
    w = rng.integers(0, 2**32, size=4096, dtype=np.uint64).astype(np.uint32)
    c = oracle.checksum(w)
    for i in rng.integers(0, w.size, 50):
        for bit in (0, 7, 31):
            v = w.copy()
            v[i] ^= np.uint32(1 << bit)
            assert oracle.checksum(v) != c
    for i, j in rng.integers(0, w.size, (50, 2)):
        v = w.copy()
        v[i], v[j] = w[j], w[i]
        seen = ((int(j) - int(i)) * (int(w[i]) - int(w[j]))) % 2**32 != 0  # the change of s2
        assert (oracle.checksum(v) != c) == seen


def test_swap_blind_spot():
    """A swap changes s2 by (j - i)(w_i - w_j) mod 2^32: words 2^16 apart whose
    values differ by 2^16 swap unseen, as the definition says they must."""
    w = np.zeros(1 << 17, np.uint32)
    w[5], w[5 + (1 << 16)] = 7, 7 + (1 << 16)
    v = w.copy()
    v[5], v[5 + (1 << 16)] = w[5 + (1 << 16)], w[5]
    assert oracle.checksum(v) == oracle.checksum(w)
    v[5] += 1  # any other change to either word is seen
    assert oracle.checksum(v) != oracle.checksum(w)
