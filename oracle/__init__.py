"""CPU oracle for the gradient-averaging hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, one IEEE rounding per written
operation); this module only marshals numpy arrays into it.  Every function
cites the page and section it follows (see ``oracle.h``).

Pins (what checks this oracle against something other than itself) live in
``tests/test_oracle_*.py`` and ``tests/golden/``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
SUM, AVG = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math, no FMA contraction)."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_LIB)
            i32, i64, u32, u64 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64
            vp, pp = C.c_void_p, C.POINTER(C.c_void_p)
            sig = {
                "oracle_philox4x32": (None, [vp, vp, C.c_int, vp]),
                "oracle_ring_chunk_len": (i64, [i64, C.c_int]),
                "oracle_ring_schedule_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, C.c_int, vp, vp]),
                "oracle_ring_fold_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, vp]),
                "oracle_ring_fold_f32_at": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_bf16_to_f32": (C.c_float, [C.c_uint16]),
                "oracle_f32_to_bf16": (C.c_uint16, [C.c_float]),
                "oracle_f32_to_bf16_n": (None, [vp, i64, vp]),
                "oracle_ring_fold_bf16": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, vp]),
                "oracle_ring_fold_bf16_at": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_ring_schedule_bf16": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, vp]),
                "oracle_bidir_subchunk_len": (i64, [i64, C.c_int]),
                "oracle_bidir_schedule_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, vp]),
                "oracle_bidir_fold_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, vp]),
                "oracle_bidir_fold_f32_samples": (C.c_int, [vp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_dbtree_build": (C.c_int, [C.c_int, C.c_int, vp, vp, vp]),
                "oracle_dbtree_half": (i64, [i64]),
                "oracle_dbtree_schedule_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, vp]),
                "oracle_dbtree_fold_f32": (C.c_int, [pp, C.c_int, i64, C.c_int, vp]),
                "oracle_dbtree_fold_bf16": (C.c_int, [pp, C.c_int, i64, C.c_int, vp]),
                "oracle_dbtree_fold_f32_samples": (C.c_int, [vp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_dbtree_fold_bf16_samples": (C.c_int, [vp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_ring_fold_f32_samples": (C.c_int, [vp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_ring_fold_bf16_samples": (C.c_int, [vp, C.c_int, i64, C.c_int, vp, i64, vp]),
                "oracle_thc_allreduce_samples": (C.c_int, [vp, C.c_int, vp, i64, C.c_int, u64, C.c_float,
                                                           C.c_float, vp, vp]),
                "oracle_fusion_plan": (C.c_int, [vp, vp, C.c_int, i64, C.c_int, vp, vp, vp]),
                "oracle_fusion_pack": (C.c_int, [pp, vp, vp, vp, C.c_int, C.c_int, vp, i64, C.c_int]),
                "oracle_fusion_unpack": (C.c_int, [vp, vp, vp, vp, C.c_int, C.c_int, pp, C.c_int]),
                "oracle_thc_range": (None, [pp, C.c_int, i64, vp, vp]),
                "oracle_thc_position": (C.c_float, [C.c_float, C.c_float, C.c_float, C.c_int]),
                "oracle_thc_index": (u32, [C.c_float, C.c_float, C.c_float, C.c_int, u64, C.c_int, i64]),
                "oracle_thc_encode": (C.c_int, [vp, i64, C.c_float, C.c_float, C.c_int, u64, C.c_int, vp]),
                "oracle_thc_unpack": (C.c_int, [vp, i64, C.c_int, vp]),
                "oracle_thc_aggregate": (C.c_int, [pp, C.c_int, i64, C.c_int, vp]),
                "oracle_thc_decode": (C.c_int, [vp, i64, C.c_float, C.c_float, C.c_int, C.c_int, vp]),
                "oracle_thc_allreduce": (C.c_int, [pp, C.c_int, i64, C.c_int, u64, C.c_float, C.c_float, vp, pp]),
                "oracle_thc_allreduce_masked": (C.c_int, [pp, C.c_int, u64, i64, C.c_int, u64, C.c_float,
                                                          C.c_float, vp, pp]),
                "oracle_nuhc_check_table": (C.c_int, [vp, C.c_int, C.c_int]),
                "oracle_nuhc_position": (C.c_float, [C.c_float, C.c_float, C.c_float, C.c_int]),
                "oracle_nuhc_index": (u32, [C.c_float, C.c_float, C.c_float, C.c_int, C.c_int, vp, u64, C.c_int,
                                            i64]),
                "oracle_nuhc_encode": (C.c_int, [vp, i64, C.c_float, C.c_float, C.c_int, C.c_int, vp, u64,
                                                 C.c_int, vp]),
                "oracle_nuhc_encode_at": (C.c_int, [vp, i64, i64, C.c_float, C.c_float, C.c_int, C.c_int, vp, u64,
                                                    C.c_int, vp]),
                "oracle_nuhc_aggregate": (C.c_int, [pp, C.c_int, i64, C.c_int, vp, vp]),
                "oracle_nuhc_decode": (C.c_int, [vp, i64, C.c_float, C.c_float, C.c_int, C.c_int, vp]),
                "oracle_rht_signs": (C.c_int, [i64, u64, vp]),
                "oracle_rht": (C.c_int, [vp, i64, u64, C.c_int, vp]),
                "oracle_rht_norm_range": (None, [pp, C.c_int, i64, C.c_double, vp, vp]),
                "oracle_ef_apply": (None, [vp, vp, vp, i64]),
                "oracle_ef_update": (None, [vp, vp, vp, i64]),
                "oracle_nmse": (C.c_double, [vp, vp, i64]),
                "oracle_checksum": (C.c_uint64, [vp, i64]),
                "oracle_nmse_f64": (C.c_double, [vp, vp, i64]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _ptrs(arrs):
    return (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# ----------------------------------------------------------------- Philox
def philox4x32(ctr, key, rounds: int = 10) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32(_ptr(c), _ptr(k), rounds, _ptr(out))
    return out


# ------------------------------------------------------------------- ring
def ring_chunk_len(n: int, p: int) -> int:
    return int(_load().oracle_ring_chunk_len(n, p))


def ring_schedule(bufs, op: int = AVG, phases: int = 2):
    """Run the literal schedule in place on fp32 (or bf16 as uint16) arrays.

    Returns (steps, sent_elems[p])."""
    p = len(bufs)
    n = bufs[0].size
    sent = np.zeros(p, np.int64)
    steps = C.c_int(0)
    lib = _load()
    if bufs[0].dtype == np.float32:
        rc = lib.oracle_ring_schedule_f32(_ptrs(bufs), p, n, op, phases, _ptr(sent), C.byref(steps))
    elif bufs[0].dtype == np.uint16:
        if phases != 2:
            raise ValueError("bf16 schedule runs both phases")
        rc = lib.oracle_ring_schedule_bf16(_ptrs(bufs), p, n, op, _ptr(sent), C.byref(steps))
    else:
        raise TypeError(bufs[0].dtype)
    _check(rc, "ring_schedule")
    return steps.value, sent


def ring_fold(xs, op: int = AVG, return_f32: bool = False):
    """Closed-form ring-order fold; fp32 arrays -> fp32, uint16 (bf16 bits) -> uint16."""
    p = len(xs)
    n = xs[0].size
    lib = _load()
    if xs[0].dtype == np.float32:
        out = np.empty(n, np.float32)
        _check(lib.oracle_ring_fold_f32(_ptrs(xs), p, n, op, _ptr(out)), "ring_fold")
        return out
    out = np.empty(n, np.uint16)
    f32 = np.empty(n, np.float32)
    _check(lib.oracle_ring_fold_bf16(_ptrs(xs), p, n, op, _ptr(out), _ptr(f32)), "ring_fold")
    return (out, f32) if return_f32 else out


def ring_fold_at(xs, n: int, idx, op: int = AVG):
    """Ring fold for chosen element indices only. xs[w] may be any array
    indexable at idx (e.g. host copies of the sampled positions are not
    enough: the fold needs x_w[idx] for every w, so xs are full arrays)."""
    p = len(xs)
    idx = np.ascontiguousarray(idx, np.int64)
    lib = _load()
    if xs[0].dtype == np.float32:
        out = np.empty(idx.size, np.float32)
        _check(lib.oracle_ring_fold_f32_at(_ptrs(xs), p, n, op, _ptr(idx), idx.size, _ptr(out)), "fold_at")
    else:
        out = np.empty(idx.size, np.uint16)
        _check(lib.oracle_ring_fold_bf16_at(_ptrs(xs), p, n, op, _ptr(idx), idx.size, _ptr(out)), "fold_at")
    return out


def bidir_schedule(bufs, op: int = AVG):
    """Literal bidirectional dual-ring schedule in place (fp32); returns (steps, sent_elems[p])."""
    p, n = len(bufs), bufs[0].size
    sent = np.zeros(p, np.int64)
    steps = C.c_int(0)
    _check(_load().oracle_bidir_schedule_f32(_ptrs(bufs), p, n, op, _ptr(sent), C.byref(steps)), "bidir_schedule")
    return steps.value, sent


def bidir_fold(xs, op: int = AVG):
    out = np.empty(xs[0].size, np.float32)
    _check(_load().oracle_bidir_fold_f32(_ptrs(xs), len(xs), xs[0].size, op, _ptr(out)), "bidir_fold")
    return out


def bidir_fold_samples(vals, n: int, idx, op: int = AVG):
    """vals[w, k] = worker w's fp32 value at element idx[k]; the two-ring fold there."""
    vals = np.ascontiguousarray(vals, np.float32)
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    _check(_load().oracle_bidir_fold_f32_samples(_ptr(vals), vals.shape[0], n, op, _ptr(idx), idx.size, _ptr(out)),
           "bidir_samples")
    return out


def ring_fold_samples(vals, n: int, idx, op: int = AVG):
    """vals[w, k] = worker w's value at element idx[k] of its n-element buffer
    (fp32, or uint16 bf16 bits); returns the ring fold at those elements."""
    vals = np.ascontiguousarray(vals)
    idx = np.ascontiguousarray(idx, np.int64)
    p = vals.shape[0]
    lib = _load()
    if vals.dtype == np.float32:
        out = np.empty(idx.size, np.float32)
        _check(lib.oracle_ring_fold_f32_samples(_ptr(vals), p, n, op, _ptr(idx), idx.size, _ptr(out)), "samples")
    else:
        out = np.empty(idx.size, np.uint16)
        _check(lib.oracle_ring_fold_bf16_samples(_ptr(vals), p, n, op, _ptr(idx), idx.size, _ptr(out)), "samples")
    return out


def bf16_to_f32(h: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(h)))


def f32_to_bf16(f: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(np.float32(f))))


def f32_to_bf16_array(a) -> np.ndarray:
    """f32_to_bf16 of every value of an fp32 array (bf16 bits as uint16)."""
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.size, np.uint16)
    _load().oracle_f32_to_bf16_n(_ptr(a), a.size, _ptr(out))
    return out


# ------------------------------------------------------ double binary tree
def dbtree_build(p: int, tree: int):
    """(root, parent[p], left[p], right[p]) of tree 0 or 1 (-1: none)."""
    par, lc, rc = (np.zeros(p, np.int32) for _ in range(3))
    root = _load().oracle_dbtree_build(p, tree, _ptr(par), _ptr(lc), _ptr(rc))
    _check(0 if root >= 0 else -1, "dbtree_build")
    return root, par, lc, rc


def dbtree_half(n: int) -> int:
    return int(_load().oracle_dbtree_half(n))


def dbtree_schedule(bufs, op: int = AVG):
    """Literal two-tree reduce + broadcast in place (fp32); returns (steps, sent_elems[p])."""
    p, n = len(bufs), bufs[0].size
    sent = np.zeros(p, np.int64)
    steps = C.c_int(0)
    _check(_load().oracle_dbtree_schedule_f32(_ptrs(bufs), p, n, op, _ptr(sent), C.byref(steps)),
           "dbtree_schedule")
    return steps.value, sent


def dbtree_fold(xs, op: int = AVG):
    """Closed-form two-tree fold; fp32 arrays -> fp32, uint16 (bf16 bits) -> uint16."""
    p, n = len(xs), xs[0].size
    lib = _load()
    if xs[0].dtype == np.float32:
        out = np.empty(n, np.float32)
        _check(lib.oracle_dbtree_fold_f32(_ptrs(xs), p, n, op, _ptr(out)), "dbtree_fold")
    else:
        out = np.empty(n, np.uint16)
        _check(lib.oracle_dbtree_fold_bf16(_ptrs(xs), p, n, op, _ptr(out)), "dbtree_fold")
    return out


def dbtree_fold_samples(vals, n: int, idx, op: int = AVG):
    """vals[w, k] = worker w's value (fp32, or bf16 bits as uint16) at element idx[k]."""
    idx = np.ascontiguousarray(idx, np.int64)
    lib = _load()
    if vals.dtype == np.float32:
        vals = np.ascontiguousarray(vals)
        out = np.empty(idx.size, np.float32)
        rc = lib.oracle_dbtree_fold_f32_samples(_ptr(vals), vals.shape[0], n, op, _ptr(idx), idx.size, _ptr(out))
    else:
        vals = np.ascontiguousarray(vals, np.uint16)
        out = np.empty(idx.size, np.uint16)
        rc = lib.oracle_dbtree_fold_bf16_samples(_ptr(vals), vals.shape[0], n, op, _ptr(idx), idx.size, _ptr(out))
    _check(rc, "dbtree_samples")
    return out


# ----------------------------------------------------------------- fusion
def fusion_plan(numel, dtype, capacity_bytes: int = 64 << 20, align_bytes: int = 16):
    """Returns (seg_buffer[count], seg_offset[count], buf_numel[n_buffers])."""
    numel = np.ascontiguousarray(numel, np.int64)
    dtype = np.ascontiguousarray(dtype, np.int32)
    count = numel.size
    sb = np.zeros(max(count, 1), np.int32)
    so = np.zeros(max(count, 1), np.int64)
    bn = np.zeros(max(count, 1), np.int64)
    nb = _load().oracle_fusion_plan(_ptr(numel), _ptr(dtype), count, capacity_bytes, align_bytes,
                                    _ptr(sb), _ptr(so), _ptr(bn))
    if nb < 0:
        raise ValueError("oracle fusion_plan rejected its arguments")
    return sb[:count].copy(), so[:count].copy(), bn[:nb].copy()


def fusion_pack(srcs, seg_buffer, seg_offset, buffer: int, buf_numel: int):
    members = [i for i, b in enumerate(seg_buffer) if b == buffer]
    dt = srcs[members[0]].dtype if members else np.dtype(np.float32)
    es = dt.itemsize
    numel = np.array([s.size for s in srcs], np.int64)
    srcs = [s if s.dtype == dt else np.zeros(0, dt) for s in srcs]  # other buffers' tensors are not read
    sb = np.ascontiguousarray(seg_buffer, np.int32)
    so = np.ascontiguousarray(seg_offset, np.int64)
    out = np.empty(int(buf_numel), dt)
    _check(_load().oracle_fusion_pack(_ptrs(srcs), _ptr(sb), _ptr(so), _ptr(numel), len(srcs), buffer,
                                      _ptr(out), int(buf_numel), es), "fusion_pack")
    return out


def fusion_unpack(fusion_buf, seg_buffer, seg_offset, numel, buffer: int):
    """Returns a list with one array per tensor (None for tensors of other buffers)."""
    numel = np.ascontiguousarray(numel, np.int64)
    sb = np.ascontiguousarray(seg_buffer, np.int32)
    so = np.ascontiguousarray(seg_offset, np.int64)
    outs = [np.zeros(int(k), fusion_buf.dtype) for k in numel]
    _check(_load().oracle_fusion_unpack(_ptr(fusion_buf), _ptr(sb), _ptr(so), _ptr(numel), numel.size,
                                        buffer, _ptrs(outs), fusion_buf.dtype.itemsize), "fusion_unpack")
    return [o if b == buffer else None for o, b in zip(outs, sb)]


# -------------------------------------------------------------------- THC
def thc_range(xs):
    m = C.c_float(0)
    M = C.c_float(0)
    _load().oracle_thc_range(_ptrs(xs), len(xs), xs[0].size, C.byref(m), C.byref(M))
    return np.float32(m.value), np.float32(M.value)


def thc_position(x: float, m: float, M: float, b: int) -> np.float32:
    return np.float32(_load().oracle_thc_position(float(x), float(m), float(M), b))


def thc_index(x, m, M, b, seed, worker, e) -> int:
    return int(_load().oracle_thc_index(float(np.float32(x)), float(m), float(M), b, seed, worker, e))


def thc_words(n: int, b: int) -> int:
    per = 32 // b
    return (n + per - 1) // per


def thc_encode(x, m, M, b: int, seed: int, worker: int) -> np.ndarray:
    out = np.empty(max(thc_words(x.size, b), 1), np.uint32)
    _check(_load().oracle_thc_encode(_ptr(x), x.size, float(m), float(M), b, seed, worker, _ptr(out)),
           "thc_encode")
    return out[:thc_words(x.size, b)]


def thc_unpack(packed, n: int, b: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint32)
    out = np.empty(n, np.uint8)
    _check(_load().oracle_thc_unpack(_ptr(packed), n, b, _ptr(out)), "thc_unpack")
    return out


def thc_aggregate(packed_list, n: int, b: int) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _check(_load().oracle_thc_aggregate(_ptrs(packed_list), len(packed_list), n, b, _ptr(out)),
           "thc_aggregate")
    return out


def thc_decode(sums, m, M, b: int, p: int) -> np.ndarray:
    sums = np.ascontiguousarray(sums, np.uint16)
    out = np.empty(sums.size, np.float64)
    _check(_load().oracle_thc_decode(_ptr(sums), sums.size, float(m), float(M), b, p, _ptr(out)),
           "thc_decode")
    return out


def thc_allreduce_samples(vals, idx, b: int, seed: int, m, M):
    """vals[w, k] = worker w's value at element idx[k]; returns (indices[w, k], avg[k])."""
    vals = np.ascontiguousarray(vals, np.float32)
    idx = np.ascontiguousarray(idx, np.int64)
    p, k = vals.shape
    ind = np.empty((p, k), np.uint8)
    avg = np.empty(k, np.float64)
    _check(_load().oracle_thc_allreduce_samples(_ptr(vals), p, _ptr(idx), k, b, seed, float(m), float(M),
                                                _ptr(ind), _ptr(avg)), "thc_samples")
    return ind, avg


def thc_allreduce(xs, b: int, seed: int, m=None, M=None, want_packed: bool = False):
    """Uniform THC round on p workers; returns avg (fp64) [, packed list]."""
    if m is None or M is None:
        m, M = thc_range(xs)
    p, n = len(xs), xs[0].size
    avg = np.empty(n, np.float64)
    packed = [np.empty(max(thc_words(n, b), 1), np.uint32) for _ in range(p)]
    _check(_load().oracle_thc_allreduce(_ptrs(xs), p, n, b, seed, float(m), float(M), _ptr(avg),
                                        _ptrs(packed)), "thc_allreduce")
    if want_packed:
        return avg, [pk[:thc_words(n, b)] for pk in packed]
    return avg


def thc_allreduce_masked(xs, arrived: int, b: int, seed: int, m, M, want_packed: bool = False):
    """THC round over the workers whose bit is set in `arrived` (stragglers dropped)."""
    p, n = len(xs), xs[0].size
    avg = np.empty(n, np.float64)
    packed = [np.zeros(max(thc_words(n, b), 1), np.uint32) for _ in range(p)]
    _check(_load().oracle_thc_allreduce_masked(_ptrs(xs), p, arrived, n, b, seed, float(m), float(M), _ptr(avg),
                                               _ptrs(packed)), "thc_allreduce_masked")
    if want_packed:
        return avg, [pk[:thc_words(n, b)] for pk in packed]
    return avg


# ----------------------------------------------------- non-uniform THC
def _table(table):
    return np.ascontiguousarray(table, np.uint16)


def nuhc_table_ok(table, b: int, g: int) -> bool:
    return _load().oracle_nuhc_check_table(_ptr(_table(table)), b, g) == 0


def nuhc_position(x, m, M, g: int) -> np.float32:
    return np.float32(_load().oracle_nuhc_position(float(x), float(m), float(M), g))


def nuhc_index(x, m, M, b, g, table, seed, worker, e) -> int:
    return int(_load().oracle_nuhc_index(float(np.float32(x)), float(m), float(M), b, g, _ptr(_table(table)), seed,
                                         worker, e))


def nuhc_encode(x, m, M, b: int, g: int, table, seed: int, worker: int) -> np.ndarray:
    out = np.empty(max(thc_words(x.size, b), 1), np.uint32)
    _check(_load().oracle_nuhc_encode(_ptr(x), x.size, float(m), float(M), b, g, _ptr(_table(table)), seed, worker,
                                      _ptr(out)), "nuhc_encode")
    return out[:thc_words(x.size, b)]


def nuhc_encode_at(x, e0: int, m, M, b: int, g: int, table, seed: int, worker: int) -> np.ndarray:
    """nuhc_encode of elements e0 .. e0 + x.size - 1 of a longer vector (e0 a
    multiple of 32 / b): that vector's packed words from word e0 / (32 / b) on."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(max(thc_words(x.size, b), 1), np.uint32)
    _check(_load().oracle_nuhc_encode_at(_ptr(x), x.size, int(e0), float(m), float(M), b, g, _ptr(_table(table)),
                                         seed, worker, _ptr(out)), "nuhc_encode_at")
    return out[:thc_words(x.size, b)]


def nuhc_aggregate(packed_list, n: int, b: int, table) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _check(_load().oracle_nuhc_aggregate(_ptrs(packed_list), len(packed_list), n, b, _ptr(_table(table)),
                                         _ptr(out)), "nuhc_aggregate")
    return out


def nuhc_decode(sums, m, M, g: int, p: int) -> np.ndarray:
    sums = np.ascontiguousarray(sums, np.uint16)
    out = np.empty(sums.size, np.float64)
    _check(_load().oracle_nuhc_decode(_ptr(sums), sums.size, float(m), float(M), g, p, _ptr(out)), "nuhc_decode")
    return out


def nuhc_allreduce(xs, b: int, g: int, table, seed: int, m=None, M=None, want_packed: bool = False):
    """Non-uniform THC round: encode every worker, look up and sum, decode."""
    if m is None or M is None:
        m, M = thc_range(xs)
    packed = [nuhc_encode(x, m, M, b, g, table, seed, w) for w, x in enumerate(xs)]
    avg = nuhc_decode(nuhc_aggregate(packed, xs[0].size, b, table), m, M, g, len(xs))
    return (avg, packed) if want_packed else avg


# ----------------------------------------------------------------- RHT
def rht_signs(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, np.int8)
    _check(_load().oracle_rht_signs(n, seed, _ptr(out)), "rht_signs")
    return out


def rht(x, seed: int, inverse: bool = False) -> np.ndarray:
    """(1/sqrt(n)) H D x, or its inverse (1/sqrt(n)) D H y, in fp64."""
    v = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(v)
    _check(_load().oracle_rht(_ptr(v), v.size, seed, 1 if inverse else 0, _ptr(out)), "rht")
    return out


def rht_norm_range(xs, t_p: float):
    """m = -M, M = (t_p / sqrt(n)) max_w ||x_w||_2 (fp64)."""
    vs = [np.ascontiguousarray(x, np.float64) for x in xs]
    m, M = C.c_double(0), C.c_double(0)
    _load().oracle_rht_norm_range(_ptrs(vs), len(vs), vs[0].size, float(t_p), C.byref(m), C.byref(M))
    return m.value, M.value


def ef_apply(grad, e) -> np.ndarray:
    """Error feedback before compression: x = grad + e (fp32)."""
    g = np.ascontiguousarray(grad, np.float32)
    ev = np.ascontiguousarray(e, np.float32)
    x = np.empty_like(g)
    _load().oracle_ef_apply(_ptr(g), _ptr(ev), _ptr(x), g.size)
    return x


def ef_update(x, x_hat) -> np.ndarray:
    """Error feedback after decompression: e = x - x_hat (fp32)."""
    xv = np.ascontiguousarray(x, np.float32)
    hv = np.ascontiguousarray(x_hat, np.float32)
    e = np.empty_like(xv)
    _load().oracle_ef_update(_ptr(e), _ptr(xv), _ptr(hv), xv.size)
    return e


def nmse(x, x_hat) -> float:
    if x.dtype == np.float64:
        return float(_load().oracle_nmse_f64(_ptr(x), _ptr(x_hat), x.size))
    return float(_load().oracle_nmse(_ptr(np.ascontiguousarray(x, np.float32)),
                                     _ptr(np.ascontiguousarray(x_hat, np.float32)), x.size))


# --------------------------------------------------------------- checksum
def checksum(words) -> int:
    """(s2 << 32) | s1 with s1 = sum w_i, s2 = sum (i + 1) w_i (mod 2^32) over uint32 words."""
    w = np.ascontiguousarray(words, np.uint32)
    return int(_load().oracle_checksum(_ptr(w), w.size))
