"""The oracle on every host core, for full-size parity checks.

The oracle's functions are plain C called through ctypes, which releases
the GIL for the length of each call, so threads run them in parallel.  The
helpers cut work into independent pieces (fusion buffers, or runs of
elements handed to the oracle's per-element entry points with their global
element indices) and never change what the oracle computes for an element.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def pmap(fn, items, threads=None):
    """[fn(x) for x in items], the calls spread over host threads."""
    items = list(items)
    if not items:
        return []
    with ThreadPoolExecutor(max_workers=min(threads or host_threads(), len(items))) as ex:
        return list(ex.map(fn, items))


def runs(lo: int, hi: int, k: int):
    """[lo, hi) cut into at most k contiguous runs of about equal length."""
    n = hi - lo
    k = max(1, min(k, n))
    cuts = [lo + (n * j) // k for j in range(k + 1)]
    return [(cuts[j], cuts[j + 1]) for j in range(k) if cuts[j] < cuts[j + 1]]


def fold_range(samples, vals, n: int, lo: int, op=oracle.AVG, threads=None, out_dtype=None):
    """samples(vals, n, idx, op) -- one of the oracle's per-element folds --
    at elements lo .. lo + len - 1 of n-element buffers; vals[w] = worker w's
    values there."""
    vals = np.ascontiguousarray(vals)
    k = vals.shape[1]
    out = np.empty(k, out_dtype or vals.dtype)

    def one(r):
        a, b = r
        out[a:b] = samples(vals[:, a:b], n, np.arange(lo + a, lo + b, dtype=np.int64), op=op)

    pmap(one, runs(0, k, 4 * (threads or host_threads())), threads)
    return out


def ring_fold_range(vals, n: int, lo: int, op=oracle.AVG, threads=None):
    """The oracle's ring fold of elements lo .. lo + len - 1 of n-element
    buffers; vals[w] = worker w's values there (fp32, or bf16 bits as uint16)."""
    return fold_range(oracle.ring_fold_samples, vals, n, lo, op, threads)


def dbtree_fold_range(vals, n: int, lo: int, op=oracle.AVG, threads=None):
    """The oracle's double-binary-tree fold, as ring_fold_range."""
    return fold_range(oracle.dbtree_fold_samples, vals, n, lo, op, threads)


def bidir_fold_range_bf16(vals, n: int, lo: int, op=oracle.AVG, threads=None):
    """The oracle's bidirectional-ring fold of bf16 inputs (uint16 bits):
    the inputs widened exactly, the fp32 fold, one rounding to bf16."""
    wide = (np.ascontiguousarray(vals, np.uint16).astype(np.uint32) << 16).view(np.float32)
    f32 = fold_range(oracle.bidir_fold_samples, wide, n, lo, op, threads)
    return oracle.f32_to_bf16_array(f32)


def thc_range_parallel(xs, threads=None):
    """The oracle's (m, M) over all workers' vectors: the range of each run
    of elements, then the range of those (min and max are exact, so the
    order of the two levels does not matter)."""
    n = xs[0].size
    parts = pmap(lambda r: oracle.thc_range([x[r[0]:r[1]] for x in xs]), runs(0, n, threads or host_threads()),
                 threads)
    return np.float32(min(p[0] for p in parts)), np.float32(max(p[1] for p in parts))


def thc_range_samples(vals, lo: int, b: int, seed: int, m, M, threads=None):
    """The oracle's THC round at elements lo .. lo + len - 1: (indices[w, k]
    as uint8, the average as fp64); vals[w] = worker w's fp32 values there."""
    vals = np.ascontiguousarray(vals, np.float32)
    p, k = vals.shape
    ind = np.empty((p, k), np.uint8)
    avg = np.empty(k, np.float64)

    def one(r):
        a, b_ = r
        i, v = oracle.thc_allreduce_samples(vals[:, a:b_], np.arange(lo + a, lo + b_, dtype=np.int64), b, seed, m, M)
        ind[:, a:b_] = i
        avg[a:b_] = v

    pmap(one, runs(0, k, 4 * (threads or host_threads())), threads)
    return ind, avg


def fusion_step(host, sizes, capacity: int, align: int, b: int, seed: int):
    """The oracle's averaging step over one plan, one fusion buffer per
    thread: pack every worker's tensors, ring fold (average), range, THC
    round with the wire vectors.  host[w][i] = worker w's tensor i.  Returns
    (seg_buffer, seg_offset, buf_numel, per-buffer dicts with 'ring' (fp32),
    'mM' (two fp32), 'thc' (fp64 average), 'packed' (one uint32 vector per
    worker))."""
    P = len(host)
    dt = np.zeros(len(sizes), np.int32)
    sb, so, bn = oracle.fusion_plan(sizes, dt, capacity, align)

    def one(k):
        bufs = [oracle.fusion_pack(host[w], sb, so, k, bn[k]) for w in range(P)]
        ring = oracle.ring_fold(bufs, op=oracle.AVG)
        m, M = oracle.thc_range(bufs)
        avg, packed = oracle.thc_allreduce(bufs, b, seed, m, M, want_packed=True)
        return {"ring": ring, "mM": (m, M), "thc": avg, "packed": packed}

    return sb, so, bn, pmap(one, range(len(bn)))
