"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* libgar.so loads and exports every function include/gar.h declares;
* gar_fusion_plan (host only) equals the oracle's plan exactly;
* argument checks return the documented status before any device work;
* the product package never imports the oracle.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gar():
    from gradient_allreduce_homomorphic_gb300 import build

    build.build()
    import gradient_allreduce_homomorphic_gb300 as g

    g.load()
    return g


def header_functions():
    text = open(os.path.join(ROOT, "include", "gar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gar_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(gar):
    names = header_functions()
    assert len(names) >= 17
    lib = C.CDLL(gar.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gar.h but not exported"
    # and the binding wraps every one of them under the same name
    for n in names:
        assert hasattr(gar, n), f"binding lacks {n}"


def _plan_both(gar, sizes, dtype, cap, align):
    p = gar.gar_fusion_plan(sizes, dtype, cap, align)
    sb, so, bn = oracle.fusion_plan(sizes, dtype, cap, align)
    np.testing.assert_array_equal(p.buffers(), sb)
    np.testing.assert_array_equal(p.offsets(), so)
    np.testing.assert_array_equal(p.buf_numel, bn)
    np.testing.assert_array_equal([s.numel for s in p.segs][:len(sizes)], sizes)


def test_plan_matches_oracle_workloads(gar):
    for sizes in (workloads.resnet_fusion_sizes(), workloads.vgg_fusion_sizes()):
        _plan_both(gar, sizes, np.zeros(sizes.size, np.int32), 64 << 20, 16)
        _plan_both(gar, sizes, np.zeros(sizes.size, np.int32), 64 << 20, 4)
        _plan_both(gar, sizes, np.zeros(sizes.size, np.int32), 25 << 20, 256)


@pytest.mark.parametrize("trial", range(30))
def test_plan_matches_oracle_random(gar, trial):
    g = np.random.default_rng([81, trial])
    count = int(g.integers(1, 60))
    sizes = g.integers(0, 5000, size=count).astype(np.int64)
    dtype = g.integers(0, 2, size=count).astype(np.int32) if trial % 3 else np.zeros(count, np.int32)
    _plan_both(gar, sizes, dtype, int(g.choice([100, 4096, 30000])), int(g.choice([4, 16, 128])))


def test_status_codes_without_launch(gar):
    lib = gar.load()
    null = C.c_void_p(0)
    ptrs = (C.c_void_p * 2)(C.c_void_p(0x1000), C.c_void_p(0x2000))
    assert lib.gar_ring_allreduce_sim(ptrs, 0, 10, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_ring_allreduce_sim(ptrs, 65, 10, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_ring_allreduce_sim(ptrs, 2, -1, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_ring_allreduce_sim(ptrs, 2, 10, 7, 1, null) == gar.GAR_EDTYPE
    assert lib.gar_ring_allreduce_sim(ptrs, 2, 10, 0, 9, null) == gar.GAR_EINVAL
    same = (C.c_void_p * 2)(C.c_void_p(0x1000), C.c_void_p(0x1000))
    assert lib.gar_ring_allreduce_sim(same, 2, 10, 0, 1, null) == gar.GAR_EINVAL
    odd = (C.c_void_p * 2)(C.c_void_p(0x1001), C.c_void_p(0x2000))
    assert lib.gar_ring_allreduce_sim(odd, 2, 10, 0, 1, null) == gar.GAR_EALIGN
    assert "aligned" in gar.gar_last_error()
    assert lib.gar_ring_allreduce_steps(ptrs, 2, 10, 3, None, None, null) == gar.GAR_EINVAL
    assert lib.gar_thc_encode(C.c_void_p(0x1000), 10, C.c_void_p(0x2000), 3, 0, 0, C.c_void_p(0x3000), null) == gar.GAR_EINVAL
    assert lib.gar_thc_aggregate(ptrs, 2, 10, 5, C.c_void_p(0x3000), null) == gar.GAR_EINVAL
    assert lib.gar_thc_decode(C.c_void_p(0x1000), 10, C.c_void_p(0x2000), 4, 0, C.c_void_p(0x3000), null) == gar.GAR_EINVAL
    assert lib.gar_nmse(C.c_void_p(0x1000), C.c_void_p(0x2000), 1000, C.c_void_p(0x3000), C.c_void_p(0x4000), 8,
                        null) == gar.GAR_EINVAL
    assert lib.gar_fusion_plan(None, None, -1, 100, 16, None, None, None) == gar.GAR_EINVAL
    assert lib.gar_dbtree_allreduce(ptrs, 0, 10, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_dbtree_allreduce(ptrs, 65, 10, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_dbtree_allreduce(ptrs, 2, 10, 7, 1, null) == gar.GAR_EDTYPE
    assert lib.gar_dbtree_allreduce(ptrs, 2, 10, 0, 9, null) == gar.GAR_EINVAL
    assert lib.gar_dbtree_allreduce(same, 2, 10, 0, 1, null) == gar.GAR_EINVAL
    assert lib.gar_dbtree_allreduce(odd, 2, 10, 0, 1, null) == gar.GAR_EALIGN
    assert lib.gar_dbtree_allreduce(None, 2, 0, 0, 1, null) == gar.GAR_OK  # N = 0: nothing touched
    assert lib.gar_dbtree_parents(0, 0, C.c_void_p(0x1000)) == gar.GAR_EINVAL
    assert lib.gar_sync_status(null, None, 1) == gar.GAR_EINVAL
    assert lib.gar_checksum(C.c_void_p(0x1000), -1, C.c_void_p(0x2000), null) == gar.GAR_EINVAL
    assert lib.gar_checksum(None, 10, C.c_void_p(0x2000), null) == gar.GAR_EINVAL
    assert lib.gar_checksum(C.c_void_p(0x1000), 10, None, null) == gar.GAR_EINVAL
    assert lib.gar_checksum(C.c_void_p(0x1002), 10, C.c_void_p(0x2000), null) == gar.GAR_EALIGN
    assert lib.gar_checksum(C.c_void_p(0x1000), 10, C.c_void_p(0x2004), null) == gar.GAR_EALIGN
    assert lib.gar_dbtree_parents(4, 2, C.c_void_p(0x1000)) == gar.GAR_EINVAL


@pytest.mark.parametrize("tree", [0, 1])
def test_dbtree_parents_match_oracle(gar, tree):
    """The library's trees (parent links from bit arithmetic on the labels)
    against the oracle's (recursive split of the label run)."""
    for P in range(1, 65):
        _, par, _, _ = oracle.dbtree_build(P, tree)
        np.testing.assert_array_equal(gar.gar_dbtree_parents(P, tree), par, err_msg=f"P={P} tree={tree}")


def test_thc_words(gar):
    for n, b, w in [(0, 4, 0), (1, 4, 1), (8, 4, 1), (9, 4, 2), (33, 1, 2), (4, 8, 1), (5, 8, 2), (16, 2, 1), (10, 3, 0)]:
        assert gar.gar_thc_words(n, b) == w
    assert gar.gar_nmse_workspace_bytes(1) >= 16
    assert gar.gar_nmse_workspace_bytes(1 << 30) <= 1 << 20


def test_binding_rejects_host_tensors(gar):
    torch = pytest.importorskip("torch")
    with pytest.raises(gar.GarError):
        gar.gar_ring_allreduce_sim([torch.zeros(8), torch.zeros(8)])


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "gradient_allreduce_homomorphic_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle.h" not in text and "liboracle" not in text, f
    text = open(os.path.join(ROOT, "oracle", "oracle.c")).read() + open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "gradient_allreduce_homomorphic_gb300" not in text and "gar.h" not in text
