"""Python binding of libgar.so, the GB300 gradient-averaging library.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The functions carry
the names of the C entry points declared in ``include/gar.h``; they take
torch tensors (and lists of them) in place of raw pointers, enqueue on the
current CUDA stream unless ``stream`` is given, and raise ``GarError`` on a
non-zero status.  There is no fallback: if the library is not built, or the
tensors are not on a CUDA device, the call fails.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgar.so")

GAR_OK, GAR_EINVAL, GAR_EDTYPE, GAR_EALIGN, GAR_EOVERFLOW, GAR_ECUDA = 0, -1, -2, -3, -4, -5
GAR_F32, GAR_BF16 = 0, 1
GAR_SUM, GAR_AVG = 0, 1
GAR_MAX_WORKERS = 64


class GarError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gar status {status}: {message}")
        self.status = status


class gar_seg(C.Structure):
    _fields_ = [("buffer", C.c_int32), ("reserved", C.c_int32), ("offset", C.c_int64), ("numel", C.c_int64)]


_lock = threading.Lock()
_lib = None

_vp, _pp = C.c_void_p, C.POINTER(C.c_void_p)
_i32, _i64, _u64 = C.c_int32, C.c_int64, C.c_uint64
_SIGNATURES = {
    "gar_version": (C.c_int, []),
    "gar_last_error": (C.c_char_p, []),
    "gar_launch_count": (C.c_uint64, []),
    "gar_sync_status": (C.c_int, [_vp, _vp, _i32]),
    "gar_checksum": (C.c_int, [_vp, _i64, _vp, _vp]),
    "gar_fusion_plan": (C.c_int, [_vp, _vp, _i32, _i64, _i32, _vp, C.POINTER(_i32), _vp]),
    "gar_fusion_pack": (C.c_int, [_pp, _vp, _vp, _i32, _i32, _vp, _i64, _vp]),
    "gar_fusion_unpack": (C.c_int, [_vp, _vp, _vp, _i32, _i32, _pp, _vp]),
    "gar_fused_allreduce": (C.c_int, [_pp, _pp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _vp]),
    "gar_fusion_pack_all": (C.c_int, [_pp, _i32, _vp, _vp, _i32, _pp, _vp, _i32, _vp, _vp]),
    "gar_fused_allreduce_range": (C.c_int, [_pp, _pp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _vp]),
    "gar_ring_allreduce_sim": (C.c_int, [_pp, _i32, _i64, _i32, _i32, _vp]),
    "gar_ring_allreduce_sim_out": (C.c_int, [_pp, _i32, _i64, _i32, _i32, _pp, _i32, _vp]),
    "gar_ring_allreduce_bidir": (C.c_int, [_pp, _i32, _i64, _i32, _i32, _vp]),
    "gar_ring_allreduce_steps": (C.c_int, [_pp, _i32, _i64, _i32, C.POINTER(_i32), _vp, _vp]),
    "gar_dbtree_allreduce": (C.c_int, [_pp, _i32, _i64, _i32, _i32, _vp]),
    "gar_dbtree_parents": (C.c_int, [_i32, _i32, _vp]),
    "gar_thc_words": (_i64, [_i64, _i32]),
    "gar_thc_range": (C.c_int, [_pp, _i32, _i64, _vp, _vp]),
    "gar_thc_encode": (C.c_int, [_vp, _i64, _vp, _i32, _u64, _i32, _vp, _vp]),
    "gar_thc_aggregate": (C.c_int, [_pp, _i32, _i64, _i32, _vp, _vp]),
    "gar_thc_decode": (C.c_int, [_vp, _i64, _vp, _i32, _i32, _vp, _vp]),
    "gar_thc_allreduce_fused": (C.c_int, [_pp, _i32, _i64, _i32, _u64, _vp, _vp, _pp, _vp]),
    "gar_thc_allreduce_fused_masked": (C.c_int, [_pp, _i32, _u64, _i64, _i32, _u64, _vp, _vp, _pp, _vp]),
    "gar_thc_allreduce_fused_plan": (C.c_int, [_pp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _u64, _vp, _pp, _pp,
                                               _vp]),
    "gar_thc_plan_nmse_workspace_bytes": (C.c_size_t, [_vp, _i32, _i32, _i32]),
    "gar_thc_allreduce_fused_plan_nmse": (C.c_int, [_pp, _i32, _vp, _vp, _i32, _vp, _i32, _i32, _u64, _vp, _pp,
                                                    _pp, _pp, _vp, _vp, C.c_size_t, _vp]),
    "gar_nuhc_encode": (C.c_int, [_vp, _i64, _vp, _i32, _i32, _vp, _u64, _i32, _vp, _vp]),
    "gar_nuhc_aggregate": (C.c_int, [_pp, _i32, _i64, _i32, _vp, _vp, _vp]),
    "gar_nuhc_decode": (C.c_int, [_vp, _i64, _vp, _i32, _i32, _vp, _vp]),
    "gar_nuhc_allreduce_fused": (C.c_int, [_pp, _i32, _i64, _i32, _i32, _vp, _u64, _vp, _vp, _pp, _vp]),
    "gar_nuhc_allreduce_fused_masked": (C.c_int, [_pp, _i32, _u64, _i64, _i32, _i32, _vp, _u64, _vp, _vp, _pp,
                                                  _vp]),
    "gar_rht": (C.c_int, [_vp, _vp, _i64, _u64, _i32, _vp]),
    "gar_rht_norm_range_workspace_bytes": (C.c_size_t, [_i32, _i64]),
    "gar_rht_norm_range": (C.c_int, [_pp, _i32, _i64, C.c_double, _vp, _vp, C.c_size_t, _vp]),
    "gar_rht_tiles": (_i64, [_i64]),
    "gar_rht_ef_forward": (C.c_int, [_vp, _vp, _vp, _i64, _u64, _vp, _vp]),
    "gar_rht_norm_range_from_sums": (C.c_int, [_pp, _i32, _i64, C.c_double, _vp, _vp]),
    "gar_rht_ef_update": (C.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _u64, _vp]),
    "gar_ef_apply": (C.c_int, [_vp, _vp, _vp, _i64, _vp]),
    "gar_ef_update": (C.c_int, [_vp, _vp, _vp, _i64, _vp]),
    "gar_nmse_workspace_bytes": (C.c_size_t, [_i64]),
    "gar_nmse": (C.c_int, [_vp, _vp, _i64, _vp, _vp, C.c_size_t, _vp]),
    "gar_nmse_noalloc": (C.c_int, [_vp, _vp, _i64, _vp, _vp]),
    "gar_nmse_sums": (C.c_int, [_vp, _vp, _i64, _vp, _vp, C.c_size_t, _vp]),
    "gar_nmse_combine": (C.c_int, [_vp, _i32, _vp, _vp]),
}


def load(path: str = LIB_PATH):
    """Load libgar.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with gradient_allreduce_homomorphic_gb300.build.build() "
                    "(there is no CPU fallback)")
            lib = C.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class _StreamArg(C.c_void_p):
    """The cudaStream_t argument of a device call (marks the call for the timeline)."""


class Timeline:
    """Horovod-Timeline-like trace of the library's device calls ([H]
    "Horovod Timeline"): with the environment variable GAR_TIMELINE set to a
    path, every call that enqueues device work is bracketed by a pair of CUDA
    events on its own stream, and at exit (or on ``dump()``) the calls are
    written as Chrome Trace Event JSON (chrome://tracing): one complete event
    per call, named after the entry point, timestamps in microseconds from
    the first call, one track per stream.  Events cost a few microseconds of
    host time per call, so the timeline is off unless asked for."""

    def __init__(self, path: str):
        import atexit

        self.path = path
        self.records = []  # (name, stream handle, start event, end event)
        self._lock = threading.Lock()
        atexit.register(self.dump)

    def begin(self, name, stream_handle):
        import torch

        ext = torch.cuda.ExternalStream(stream_handle) if stream_handle else torch.cuda.default_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(ext)
        return (name, stream_handle or 0, start, end, ext)

    def end(self, token):
        name, handle, start, end, ext = token
        end.record(ext)
        with self._lock:
            self.records.append((name, handle, start, end))

    def events(self):
        """The recorded calls as Chrome trace events (synchronises the device)."""
        import torch

        with self._lock:
            recs = list(self.records)
        if not recs:
            return []
        torch.cuda.synchronize()
        t0 = recs[0][2]
        tracks = {}
        out = []
        for name, handle, start, end in recs:
            tid = tracks.setdefault(handle, len(tracks))
            out.append({"name": name, "cat": "gar", "ph": "X", "pid": 0, "tid": tid,
                        "ts": round(t0.elapsed_time(start) * 1e3, 3), "dur": round(start.elapsed_time(end) * 1e3, 3),
                        "args": {"stream": hex(handle)}})
        return out

    def dump(self):
        import json

        try:
            ev = self.events()
        except Exception:  # the CUDA context may be gone at interpreter exit
            return
        with open(self.path, "w") as f:
            json.dump({"traceEvents": ev, "displayTimeUnit": "ms"}, f)


_timeline = Timeline(os.environ["GAR_TIMELINE"]) if os.environ.get("GAR_TIMELINE") else None


def timeline():
    """The active Timeline, or None when GAR_TIMELINE is not set."""
    return _timeline


def _call(name, *args):
    token = None
    if _timeline is not None and args and isinstance(args[-1], _StreamArg):
        token = _timeline.begin(name, args[-1].value)
    rc = getattr(load(), name)(*args)
    if token is not None:
        _timeline.end(token)
    if rc != GAR_OK:
        raise GarError(rc, load().gar_last_error().decode(errors="replace"))


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return _StreamArg(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t):
    if not t.is_cuda:
        raise GarError(GAR_EINVAL, "tensor is not on a CUDA device (the library has no CPU path)")
    return t.data_ptr()


class PtrTable:
    """A host array of device pointers built once from a list of tensors, so
    that repeated calls skip the per-call marshalling.  Keeps the tensors
    alive; numel and dtype describe the first tensor."""

    def __init__(self, tensors, allow_none: bool = False):
        self.tensors = list(tensors)
        ptrs = [(_dev(t) if t is not None else None) if allow_none else _dev(t) for t in self.tensors]
        self.array = (C.c_void_p * len(ptrs))(*ptrs)
        first = next((t for t in self.tensors if t is not None), None)
        self.numel = first.numel() if first is not None else 0
        self.first = first

    def __len__(self):
        return len(self.tensors)


def pointer_table(tensors, allow_none: bool = False) -> PtrTable:
    return tensors if isinstance(tensors, PtrTable) else PtrTable(tensors, allow_none)


def _ptr_array(tensors):
    return pointer_table(tensors).array


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return GAR_F32
    if t.dtype == torch.bfloat16:
        return GAR_BF16
    raise GarError(GAR_EDTYPE, f"unsupported dtype {t.dtype}")


def gar_version() -> int:
    return int(load().gar_version())


def gar_last_error() -> str:
    return load().gar_last_error().decode(errors="replace")


def gar_launch_count() -> int:
    return int(load().gar_launch_count())


# ------------------------------------------------------------ Tensor Fusion
@dataclass
class FusionPlan:
    segs: C.Array           # gar_seg[count]
    dtype: np.ndarray       # int32[count]
    buf_numel: np.ndarray   # int64[n_buffers]

    @property
    def count(self) -> int:
        return len(self.dtype)

    @property
    def n_buffers(self) -> int:
        return len(self.buf_numel)

    def buffers(self) -> np.ndarray:
        return np.array([s.buffer for s in self.segs], np.int32)

    def offsets(self) -> np.ndarray:
        return np.array([s.offset for s in self.segs], np.int64)

    def subplan(self, first: int, count: int) -> "FusionPlan":
        """The plan restricted to tensors first .. first+count-1 (a view of the
        same segments; buffer ids and buffer lengths unchanged)."""
        segs = (gar_seg * max(count, 1)).from_address(C.addressof(self.segs) + first * C.sizeof(gar_seg))
        sub = FusionPlan(segs, self.dtype[first:first + count].copy(), self.buf_numel)
        sub._parent = self  # keep the segment storage alive
        return sub

    def buffer_tensors(self, buffer: int):
        """(first, count) of the tensors of one buffer (contiguous in plan order)."""
        ids = np.nonzero(self.buffers() == buffer)[0]
        return (int(ids[0]), int(ids.size)) if ids.size else (0, 0)


def gar_fusion_plan(numel, dtype, capacity_bytes: int = 64 << 20, align_bytes: int = 16) -> FusionPlan:
    numel = np.ascontiguousarray(numel, np.int64)
    dtype = np.ascontiguousarray(dtype, np.int32)
    count = int(numel.size)
    segs = (gar_seg * max(count, 1))()
    bn = np.zeros(max(count, 1), np.int64)
    nb = _i32(0)
    _call("gar_fusion_plan", numel.ctypes.data, dtype.ctypes.data, count, capacity_bytes, align_bytes,
          C.addressof(segs), C.byref(nb), bn.ctypes.data)
    return FusionPlan(segs, dtype, bn[:nb.value].copy())


def gar_fusion_pack(src, plan: FusionPlan, buffer: int, fusion_buf, stream=None):
    """src: one worker's tensors (list or PtrTable; entries of other buffers may be None)."""
    ptrs = pointer_table(src, allow_none=True).array
    _call("gar_fusion_pack", ptrs, C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count, buffer,
          _dev(fusion_buf), int(plan.buf_numel[buffer]), _stream(stream))


def gar_fusion_unpack(fusion_buf, plan: FusionPlan, buffer: int, dst, stream=None):
    ptrs = pointer_table(dst, allow_none=True).array
    _call("gar_fusion_unpack", _dev(fusion_buf), C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count,
          buffer, ptrs, _stream(stream))


def gar_fusion_pack_all(src, plan: FusionPlan, fusion_bufs, d_mM=None, stream=None, tables=None):
    """Pack every worker's tensors into its fusion buffers in one pass.

    src[w][i]: worker w's tensor i; fusion_bufs[w][b]: worker w's buffer b;
    d_mM (optional, fp32 plans): [n_buffers, 2] per-buffer min/max output."""
    if tables is None:
        tables = pack_all_tables(src, fusion_bufs)
    s, f = tables
    P = len(s) // max(plan.count, 1)
    _call("gar_fusion_pack_all", s.array, P, C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count, f.array,
          plan.buf_numel.ctypes.data, plan.n_buffers, _dev(d_mM) if d_mM is not None else None, _stream(stream))


def pack_all_tables(src, fusion_bufs):
    """Host pointer tables for gar_fusion_pack_all (reuse them across steps)."""
    return (PtrTable([t for row in src for t in row]), PtrTable([t for row in fusion_bufs for t in row]))


def fused_pointer_tables(src, dst):
    """Host pointer tables for gar_fused_allreduce (reuse them across steps)."""
    return (PtrTable([t for row in src for t in row]), PtrTable([t for row in dst for t in row]))


def gar_fused_allreduce(src, dst, plan: FusionPlan, op: int = GAR_AVG, stream=None, tables=None):
    """src[w][i], dst[w][i]: worker w's tensor i (dst may be src)."""
    P = len(src)
    s, d = tables if tables is not None else fused_pointer_tables(src, dst)
    _call("gar_fused_allreduce", s.array, d.array, P, C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count,
          plan.buf_numel.ctypes.data, plan.n_buffers, op, _stream(stream))


def gar_fused_allreduce_range(src, dst, plan: FusionPlan, d_mM, op: int = GAR_AVG, stream=None, tables=None):
    """gar_fused_allreduce that also writes each buffer's THC range [m, M]
    (d_mM: [n_buffers, 2] fp32 device tensor) from the same reads."""
    P = len(src)
    s, d = tables if tables is not None else fused_pointer_tables(src, dst)
    _call("gar_fused_allreduce_range", s.array, d.array, P, C.addressof(plan.segs), plan.dtype.ctypes.data,
          plan.count, plan.buf_numel.ctypes.data, plan.n_buffers, op, _dev(d_mM), _stream(stream))


GAR_STATUS_NONFINITE = 1


def gar_checksum(words, d_out, stream=None):
    """(s2 << 32) | s1 of the 32-bit words (a CUDA tensor of 4-byte elements)
    into d_out (one int64/uint64 element on the device)."""
    n = words.numel() * words.element_size() // 4
    _call("gar_checksum", _dev(words), n, _dev(d_out), _stream(stream))


def gar_sync_status(stream=None, clear: bool = True) -> int:
    """Wait for `stream`, then return the device status word (GAR_STATUS_*
    bits: conditions the kernels found on the device), clearing it if asked."""
    out = C.c_uint32(0)
    _call("gar_sync_status", _stream(stream), C.byref(out), 1 if clear else 0)
    return int(out.value)


# ----------------------------------------------------------- ring all-reduce
def gar_ring_allreduce_sim(bufs, op: int = GAR_AVG, stream=None):
    t = pointer_table(bufs)
    _call("gar_ring_allreduce_sim", t.array, len(t), t.numel, _dtype_code(t.first), op, _stream(stream))


def gar_ring_allreduce_bidir(bufs, op: int = GAR_AVG, stream=None):
    """Bidirectional dual ring (in place): first half clockwise, second half counter-clockwise."""
    t = pointer_table(bufs)
    _call("gar_ring_allreduce_bidir", t.array, len(t), t.numel, _dtype_code(t.first), op, _stream(stream))


def gar_dbtree_allreduce(bufs, op: int = GAR_AVG, stream=None):
    """Double-binary-tree all-reduce (in place): first half over tree 1, the rest over tree 2."""
    t = pointer_table(bufs)
    _call("gar_dbtree_allreduce", t.array, len(t), t.numel, _dtype_code(t.first), op, _stream(stream))


def gar_dbtree_parents(P: int, tree: int):
    """Host only: parent rank of every rank in tree 0 or 1 (-1: the root)."""
    out = np.zeros(P, np.int32)
    _call("gar_dbtree_parents", P, tree, out.ctypes.data)
    return out


def gar_ring_allreduce_sim_out(bufs, out, op: int = GAR_AVG, stream=None):
    t, o = pointer_table(bufs), pointer_table(out)
    _call("gar_ring_allreduce_sim_out", t.array, len(t), t.numel, _dtype_code(t.first), op,
          o.array, len(o), _stream(stream))


def gar_ring_allreduce_steps(bufs, op: int = GAR_AVG, stream=None):
    """Literal schedule (fp32, in place); returns (steps, sent_elems[P])."""
    P = len(bufs)
    steps = _i32(0)
    sent = np.zeros(P, np.int64)
    _call("gar_ring_allreduce_steps", _ptr_array(bufs), P, bufs[0].numel(), op, C.byref(steps),
          sent.ctypes.data, _stream(stream))
    return steps.value, sent


# --------------------------------------------------------------------- THC
def gar_thc_words(N: int, b: int) -> int:
    return int(load().gar_thc_words(N, b))


def gar_thc_range(x, d_mM, stream=None):
    t = pointer_table(x)
    _call("gar_thc_range", t.array, len(t), t.numel, _dev(d_mM), _stream(stream))


def gar_thc_encode(x, d_mM, b: int, seed: int, worker: int, packed, stream=None):
    _call("gar_thc_encode", _dev(x), x.numel(), _dev(d_mM), b, seed, worker, _dev(packed), _stream(stream))


def gar_thc_aggregate(packed, N: int, b: int, sums, stream=None):
    t = pointer_table(packed)
    _call("gar_thc_aggregate", t.array, len(t), N, b, _dev(sums), _stream(stream))


def gar_thc_decode(sums, d_mM, b: int, P: int, avg, stream=None):
    _call("gar_thc_decode", _dev(sums), sums.numel(), _dev(d_mM), b, P, _dev(avg), _stream(stream))


def gar_thc_allreduce_fused(x, b: int, seed: int, d_mM, avg, packed=None, stream=None):
    t = pointer_table(x)
    pk = pointer_table(packed).array if packed is not None else None
    _call("gar_thc_allreduce_fused", t.array, len(t), t.numel, b, seed, _dev(d_mM), _dev(avg), pk,
          _stream(stream))


def gar_thc_allreduce_fused_masked(x, arrived: int, b: int, seed: int, d_mM, avg, packed=None, stream=None):
    """THC round over the workers whose bit is set in `arrived` (stragglers
    dropped); x[w] / packed[w] of the others may be None."""
    xt = pointer_table(x, allow_none=True)
    pk = pointer_table(packed, allow_none=True).array if packed is not None else None
    _call("gar_thc_allreduce_fused_masked", xt.array, len(xt), arrived, xt.numel, b, seed, _dev(d_mM), _dev(avg),
          pk, _stream(stream))


def thc_plan_tables(src, out, packed=None):
    """Host pointer tables for gar_thc_allreduce_fused_plan (reuse them across steps):
    src[w][i] worker w's tensor i, out[i] output tensor i, packed[w][b] or None."""
    return (PtrTable([t for row in src for t in row]), PtrTable(out),
            PtrTable([t for row in packed for t in row]) if packed is not None else None)


def gar_thc_allreduce_fused_plan(src, plan: FusionPlan, b: int, seed: int, d_mM, out, packed=None, stream=None,
                                 tables=None):
    """Uniform THC of every fusion buffer of `plan`, reading the workers'
    tensors src[w][i] directly and writing the average to out[i]; d_mM is the
    [n_buffers, 2] per-buffer range; packed[w][b] optionally receives worker
    w's indices of buffer b."""
    s, o, pk = tables if tables is not None else thc_plan_tables(src, out, packed)
    P = len(s) // max(plan.count, 1)
    _call("gar_thc_allreduce_fused_plan", s.array, P, C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count,
          plan.buf_numel.ctypes.data, plan.n_buffers, b, seed, _dev(d_mM), o.array,
          pk.array if pk is not None else None, _stream(stream))


def gar_thc_plan_nmse_workspace_bytes(plan: FusionPlan, b: int) -> int:
    return int(load().gar_thc_plan_nmse_workspace_bytes(plan.buf_numel.ctypes.data, plan.n_buffers, plan.count, b))


def gar_thc_allreduce_fused_plan_nmse(src, plan: FusionPlan, b: int, seed: int, d_mM, out, ref, d_pair, workspace,
                                      packed=None, stream=None, tables=None, ref_table=None):
    """gar_thc_allreduce_fused_plan that also writes d_pair (2 fp64, device) =
    (sum (ref - avg)^2, sum ref^2) over the call's tensors; ref[i] is the
    reference tensor of tensor i (e.g. the ring average)."""
    s, o, pk = tables if tables is not None else thc_plan_tables(src, out, packed)
    r = ref_table if ref_table is not None else PtrTable(ref)
    P = len(s) // max(plan.count, 1)
    nbytes = workspace.numel() * workspace.element_size()
    _call("gar_thc_allreduce_fused_plan_nmse", s.array, P, C.addressof(plan.segs), plan.dtype.ctypes.data, plan.count,
          plan.buf_numel.ctypes.data, plan.n_buffers, b, seed, _dev(d_mM), o.array,
          pk.array if pk is not None else None, r.array, _dev(d_pair), _dev(workspace), nbytes, _stream(stream))


# --------------------------------------------------------- non-uniform THC
def _table(table):
    t = np.ascontiguousarray(table, np.uint16)
    return t, t.ctypes.data


def gar_nuhc_encode(x, d_mM, b: int, g: int, table, seed: int, worker: int, packed, stream=None):
    t, tp = _table(table)
    _call("gar_nuhc_encode", _dev(x), x.numel(), _dev(d_mM), b, g, tp, seed, worker, _dev(packed), _stream(stream))


def gar_nuhc_aggregate(packed, N: int, b: int, table, sums, stream=None):
    t, tp = _table(table)
    pt = pointer_table(packed)
    _call("gar_nuhc_aggregate", pt.array, len(pt), N, b, tp, _dev(sums), _stream(stream))


def gar_nuhc_decode(sums, d_mM, g: int, P: int, avg, stream=None):
    _call("gar_nuhc_decode", _dev(sums), sums.numel(), _dev(d_mM), g, P, _dev(avg), _stream(stream))


def gar_nuhc_allreduce_fused(x, b: int, g: int, table, seed: int, d_mM, avg, packed=None, stream=None):
    t, tp = _table(table)
    xt = pointer_table(x)
    pk = pointer_table(packed).array if packed is not None else None
    _call("gar_nuhc_allreduce_fused", xt.array, len(xt), xt.numel, b, g, tp, seed, _dev(d_mM), _dev(avg), pk,
          _stream(stream))


def gar_nuhc_allreduce_fused_masked(x, arrived: int, b: int, g: int, table, seed: int, d_mM, avg, packed=None,
                                    stream=None):
    """Non-uniform THC round over the workers whose bit is set in `arrived`
    (stragglers dropped); x[w] / packed[w] of the others may be None."""
    t, tp = _table(table)
    xt = pointer_table(x, allow_none=True)
    pk = pointer_table(packed, allow_none=True).array if packed is not None else None
    _call("gar_nuhc_allreduce_fused_masked", xt.array, len(xt), arrived, xt.numel, b, g, tp, seed, _dev(d_mM),
          _dev(avg), pk, _stream(stream))


# ------------------------------------------- RHT, range and error feedback
def gar_rht(x, out, seed: int, inverse: bool = False, stream=None):
    """out = (1/sqrt n) H D x, or (1/sqrt n) D H x with inverse=True; out may be x."""
    _call("gar_rht", _dev(x), _dev(out), x.numel(), seed, int(bool(inverse)), _stream(stream))


def gar_rht_norm_range_workspace_bytes(P: int, n: int) -> int:
    return int(load().gar_rht_norm_range_workspace_bytes(P, n))


def gar_rht_norm_range(x, t_p: float, d_mM, workspace, stream=None):
    t = pointer_table(x)
    nbytes = workspace.numel() * workspace.element_size()
    _call("gar_rht_norm_range", t.array, len(t), t.numel, float(t_p), _dev(d_mM), _dev(workspace), nbytes,
          _stream(stream))


def gar_rht_tiles(n: int) -> int:
    return int(load().gar_rht_tiles(n))


def gar_rht_ef_forward(grad, e, y, seed: int, sumsq=None, stream=None):
    """y = (1/sqrt n) H D (grad + e); sumsq (fp64, gar_rht_tiles(n)) receives
    the per-tile sums of squares of grad + e if given."""
    _call("gar_rht_ef_forward", _dev(grad), _dev(e), _dev(y), grad.numel(), seed,
          _dev(sumsq) if sumsq is not None else None, _stream(stream))


def gar_rht_norm_range_from_sums(sumsq, n: int, t_p: float, d_mM, stream=None):
    """The norm-based range from the workers' per-tile sums (a list of fp64 tensors)."""
    t = pointer_table(sumsq)
    _call("gar_rht_norm_range_from_sums", t.array, len(t), n, float(t_p), _dev(d_mM), _stream(stream))


def gar_rht_ef_update(packed, b: int, steps: int, table, d_mM, grad, e, tmp, seed: int, stream=None):
    """e = (grad + e) - (1/sqrt n) D H decode(packed); table None for uniform THC (steps = 2^b - 1)."""
    tp = None
    if table is not None:
        t, tp = _table(table)
    _call("gar_rht_ef_update", _dev(packed), b, steps, tp, _dev(d_mM), _dev(grad), _dev(e), _dev(tmp), e.numel(),
          seed, _stream(stream))


def gar_ef_apply(grad, e, x, stream=None):
    _call("gar_ef_apply", _dev(grad), _dev(e), _dev(x), grad.numel(), _stream(stream))


def gar_ef_update(e, x, x_hat, stream=None):
    _call("gar_ef_update", _dev(e), _dev(x), _dev(x_hat), e.numel(), _stream(stream))


# -------------------------------------------------------------------- NMSE
def gar_nmse_workspace_bytes(N: int) -> int:
    return int(load().gar_nmse_workspace_bytes(N))


def gar_nmse(x, x_hat, d_out, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _call("gar_nmse", _dev(x), _dev(x_hat), x.numel(), _dev(d_out), _dev(workspace), nbytes, _stream(stream))


def gar_nmse_sums(x, x_hat, d_pair, workspace, stream=None):
    """(sum (x - x_hat)^2, sum x^2) of one range into d_pair (2 fp64, device)."""
    nbytes = workspace.numel() * workspace.element_size()
    _call("gar_nmse_sums", _dev(x), _dev(x_hat), x.numel(), _dev(d_pair), _dev(workspace), nbytes, _stream(stream))


def gar_nmse_combine(d_pairs, d_out, stream=None):
    """NMSE from the pairs of gar_nmse_sums (d_pairs: [n, 2] fp64, device)."""
    _call("gar_nmse_combine", _dev(d_pairs), d_pairs.numel() // 2, _dev(d_out), _stream(stream))


def gar_nmse_noalloc(x, x_hat, d_out, stream=None):
    """NMSE without a workspace, for callers that may not allocate device
    memory: partial sums go to a fixed array inside the library (see gar.h)."""
    _call("gar_nmse_noalloc", _dev(x), _dev(x_hat), x.numel(), _dev(d_out), _stream(stream))


__all__ = [n for n in dir() if n.startswith(("gar_", "GAR_"))] + ["GarError", "FusionPlan", "PtrTable", "load",
                                                                    "pointer_table", "fused_pointer_tables", "thc_plan_tables",
                                                                    "Timeline", "timeline"]
