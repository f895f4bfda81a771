"""One gradient-averaging step over P workers' flat gradient buffers, bucketed
by fusion buffer and pipelined on CUDA streams.

The step runs every row of the path through the library's entry points:

  1. the Tensor Fusion plan of the tensor list (host)          gar_fusion_plan
  2. per fusion buffer, the exact average: Tensor Fusion +      gar_fused_allreduce_range
     ring all-reduce in one pass (pack, ring, unpack), the
     buffer's THC range [m, M] from the same reads
  3. per fusion buffer, the compressed average: every worker's  gar_thc_allreduce_fused_plan
     THC indices (the wire vectors), their integer sum and the
     decode, read straight from the tensors and written straight
     to the output tensors
  4. the NMSE of the compressed average against the exact one:  gar_thc_allreduce_fused_plan_nmse,
     its sums taken inside step 3 (one more read of the exact   gar_nmse_combine
     average), then combined (nmse="separate": one pass over    (gar_nmse)
     both averages at the end)

Overlap ([R] "8. Compute-Communication Overlapping & Gradient Bucketing"):
fusion buffers are the buckets.  The ring runs on one stream, bucket after
bucket, and records an event behind each bucket; THC of bucket b runs on a
second stream once that event has fired (it needs the range the ring wrote),
so it overlaps the ring of bucket b + 1.  The NMSE waits for both streams.
Both streams wait for the caller's stream at the start of a step and the
caller's stream waits for both at its end, so consecutive steps (and whatever
the caller queues around them) stay ordered.

Everything here is host-side orchestration of streams and events; each step
of the arithmetic runs in the library's CUDA kernels.  Buffers are allocated
once, at construction; a step allocates nothing on the device.
"""
from __future__ import annotations

import numpy as np

from . import (GAR_AVG, gar_fused_allreduce_range, gar_fusion_plan, gar_nmse, gar_nmse_combine,
               gar_nmse_workspace_bytes, gar_thc_allreduce_fused_plan, gar_thc_allreduce_fused_plan_nmse,
               gar_thc_plan_nmse_workspace_bytes, gar_thc_words, fused_pointer_tables, pointer_table,
               thc_plan_tables)

STAGES = ("ring", "thc", "nmse")


def flat_offsets(sizes, align_elems: int = 4) -> np.ndarray:
    """Start of each tensor in a flat buffer that places every tensor on an
    `align_elems`-element boundary (4 fp32 = one 16-byte line), plus the
    buffer's length as the last entry."""
    sizes = np.asarray(sizes, np.int64)
    padded = (sizes + align_elems - 1) // align_elems * align_elems
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


class AveragingStep:
    """Device-resident state of the bucketed averaging step.

    grads: P flat fp32 CUDA tensors, worker w's gradient tensors being the
    views grads[w][offsets[i] : offsets[i] + sizes[i]].  The outputs are flat
    buffers of the same layout: ``ring_flat[w]`` (the exact average, every
    worker's copy) and ``thc_flat`` (the compressed average); their padding
    stays zero, so an NMSE over the flat buffers equals the NMSE over the
    tensors.  ``packed[w][b]`` holds worker w's wire vector of fusion buffer
    b, ``mM[b]`` that buffer's range, ``nmse`` the step's NMSE."""

    def __init__(self, grads, sizes, offsets=None, *, b: int = 4, capacity_bytes: int = 64 << 20,
                 align_bytes: int = 16, nmse: str = "fused"):
        import torch

        if nmse not in ("separate", "fused"):
            raise ValueError(f"nmse must be 'separate' or 'fused', not {nmse!r}")
        self.torch = torch
        self.P = len(grads)
        self.b = int(b)
        self.capacity, self.align = int(capacity_bytes), int(align_bytes)
        self.nmse_mode = nmse
        self.sizes = np.ascontiguousarray(sizes, np.int64)
        self.offs = flat_offsets(self.sizes) if offsets is None else np.asarray(offsets, np.int64)
        self.dtype = np.zeros(self.sizes.size, np.int32)
        self.flat = list(grads)
        self.flat_len = int(self.flat[0].numel())
        if int(self.offs[self.sizes.size - 1] + self.sizes[-1]) > self.flat_len:
            raise ValueError("the tensors overrun the flat gradient buffers")
        dev = self.flat[0].device
        self.device = dev
        self.src = [self._views(f) for f in self.flat]
        self.ring_flat = [torch.zeros(self.flat_len, dtype=torch.float32, device=dev) for _ in range(self.P)]
        self.ring = [self._views(f) for f in self.ring_flat]
        self.thc_flat = torch.zeros(self.flat_len, dtype=torch.float32, device=dev)
        self.thc = self._views(self.thc_flat)
        self.plan = gar_fusion_plan(self.sizes, self.dtype, self.capacity, self.align)
        self.nb = self.plan.n_buffers
        bn = self.plan.buf_numel
        self.words = [gar_thc_words(int(bn[k]), self.b) for k in range(self.nb)]
        self.packed = [[torch.zeros(max(self.words[k], 1), dtype=torch.int32, device=dev) for k in range(self.nb)]
                       for _ in range(self.P)]
        self.mM = torch.zeros((self.nb, 2), dtype=torch.float32, device=dev)
        self.nmse = torch.zeros(1, dtype=torch.float64, device=dev)
        self.pairs = torch.zeros((self.nb, 2), dtype=torch.float64, device=dev)
        self.ws = torch.empty(gar_thc_plan_nmse_workspace_bytes(self.plan, self.b) // 8 + 1, dtype=torch.float64,
                              device=dev)
        self.ws_nmse = torch.empty(gar_nmse_workspace_bytes(self.flat_len) // 8 + 1, dtype=torch.float64,
                                   device=dev)
        # host pointer tables per fusion buffer, built once (the buffers do not move)
        self.parts = []
        for k in range(self.nb):
            first, cnt = self.plan.buffer_tensors(k)
            rows = slice(first, first + cnt)
            src_k = [self.src[w][rows] for w in range(self.P)]
            self.parts.append({
                "first": first, "count": cnt,
                "lo": int(self.offs[first]), "hi": int(self.offs[first + cnt - 1] + self.sizes[first + cnt - 1]),
                "ring": fused_pointer_tables(src_k, [self.ring[w][rows] for w in range(self.P)]),
                "thc": thc_plan_tables(src_k, self.thc[rows], self.packed),
                "ref": pointer_table(self.ring[0][rows]),  # NMSE reference: the exact (ring) average
                "ev": torch.cuda.Event(),
            })
        self.stream_ring = torch.cuda.Stream(device=dev)
        self.stream_thc = torch.cuda.Stream(device=dev)
        self._host = None

    def _views(self, flat):
        return [flat[int(self.offs[i]):int(self.offs[i]) + int(s)] for i, s in enumerate(self.sizes)]

    # ------------------------------------------------------------ stages
    def _ring(self, plan, k, stream):
        part = self.parts[k]
        sub = plan.subplan(part["first"], part["count"])
        gar_fused_allreduce_range([None] * self.P, None, sub, self.mM, op=GAR_AVG, stream=stream,
                                  tables=part["ring"])

    def _thc(self, plan, k, seed, stream):
        part = self.parts[k]
        sub = plan.subplan(part["first"], part["count"])
        if self.nmse_mode == "fused":
            gar_thc_allreduce_fused_plan_nmse(None, sub, self.b, seed, self.mM, None, None, self.pairs[k], self.ws,
                                              stream=stream, tables=part["thc"], ref_table=part["ref"])
        else:
            gar_thc_allreduce_fused_plan(None, sub, self.b, seed, self.mM, None, stream=stream, tables=part["thc"])

    def _nmse(self, stream):
        if self.nmse_mode == "fused":
            gar_nmse_combine(self.pairs, self.nmse, stream=stream)
        else:
            gar_nmse(self.ring_flat[0], self.thc_flat, self.nmse, self.ws_nmse, stream=stream)

    def algorithmic_bytes(self):
        """HBM bytes each stage must move per step (the roofline's numerator)."""
        n = int(self.sizes.sum()) * 4
        words = 4 * sum(self.words)
        return {
            "ring": 2 * self.P * n,  # read P x n, write P x n (the range from the same reads)
            # read P x n (and the reference, fused NMSE); write the average and the wire vectors
            "thc": self.P * n + (2 if self.nmse_mode == "fused" else 1) * n + self.P * words,
            # the per-buffer pairs of sums, combined; or one pass over both flat averages
            "nmse": 16 * self.nb if self.nmse_mode == "fused" else 2 * self.flat_len * 4,
        }

    # -------------------------------------------------------------- step
    def run(self, seed: int, schedule: str = "overlap", events=None):
        """One step on the current stream's timeline.  schedule="overlap":
        the ring and THC on their own streams, THC of bucket b behind the
        ring of bucket b; "serial": every launch on the current stream.
        events: optional dict stage -> (start, end) CUDA events to record."""
        torch = self.torch
        main = torch.cuda.current_stream(self.device)
        overlap = schedule == "overlap"
        s_ring = self.stream_ring if overlap else main
        s_thc = self.stream_thc if overlap else main

        def mark(stage, i, stream):
            if events is not None:
                events[stage][i].record(stream)

        plan = gar_fusion_plan(self.sizes, self.dtype, self.capacity, self.align)
        if overlap:
            s_ring.wait_stream(main)
            s_thc.wait_stream(main)
        mark("ring", 0, s_ring)
        for k in range(self.nb):
            self._ring(plan, k, s_ring)
            if overlap:
                self.parts[k]["ev"].record(s_ring)
        mark("ring", 1, s_ring)
        for k in range(self.nb):
            if overlap:
                s_thc.wait_event(self.parts[k]["ev"])
            if k == 0:
                mark("thc", 0, s_thc)
            self._thc(plan, k, seed, s_thc)
        mark("thc", 1, s_thc)
        if overlap:
            main.wait_stream(s_thc)
            main.wait_stream(s_ring)
        mark("nmse", 0, main)
        self._nmse(main)
        mark("nmse", 1, main)

    # ------------------------------------------------------ from the host
    def setup_host(self, n_h2d: int = 2):
        """Streams and events of the host-to-host step (call once)."""
        torch = self.torch
        dev = self.device
        self._host = {
            "h2d": [torch.cuda.Stream(device=dev) for _ in range(n_h2d)],
            "d2h": torch.cuda.Stream(device=dev),
            "ev_in": [[torch.cuda.Event() for _ in range(n_h2d)] for _ in range(self.nb)],
            "ev_out": [torch.cuda.Event() for _ in range(self.nb)],
            "ev_read": [torch.cuda.Event() for _ in range(self.nb)],  # bucket k's inputs consumed
            "ev_sent": [torch.cuda.Event() for _ in range(self.nb)],  # bucket k's outputs copied out
            "ev_nmse": torch.cuda.Event(),
            "ev_nmse_sent": torch.cuda.Event(),
        }

    def host_begin(self):
        """Order the copy streams after everything queued so far."""
        h = self._host
        main = self.torch.cuda.current_stream(self.device)
        for s in h["h2d"] + [h["d2h"]]:
            s.wait_stream(main)

    def host_end(self):
        """Join the copy streams into the current stream: once it reaches
        this point the last step's results are on the host."""
        h = self._host
        main = self.torch.cuda.current_stream(self.device)
        for s in h["h2d"] + [h["d2h"]]:
            main.wait_stream(s)

    def run_from_host(self, seed: int, host_in, host_ring=None, host_thc=None, host_nmse=None):
        """One step from pinned host gradients (host_in[w], flat, this
        layout) to host results: the exact and the compressed averages
        (host_ring, host_thc: pinned flat fp32; None skips that copy) and the
        NMSE (host_nmse: one pinned fp64).  Pipelined by bucket: bucket k+1's
        inputs cross the link (the workers spread over the copy streams)
        while bucket k is averaged, and bucket k's averages travel back
        meanwhile.  Consecutive steps overlap too: a bucket's inputs are
        overwritten only once the previous step has read them, its averages
        only once the previous step's have been copied out.  Bracket a run
        of steps with host_begin() / host_end()."""
        torch = self.torch
        h = self._host
        if h is None:
            raise RuntimeError("call setup_host() first")
        main = torch.cuda.current_stream(self.device)
        plan = gar_fusion_plan(self.sizes, self.dtype, self.capacity, self.align)
        n_in = len(h["h2d"])
        out = host_ring is not None or host_thc is not None
        for k, part in enumerate(self.parts):
            lo, hi = part["lo"], part["hi"]
            for j, s in enumerate(h["h2d"]):
                s.wait_event(h["ev_read"][k])
                with torch.cuda.stream(s):
                    for w in range(j, self.P, n_in):
                        self.flat[w][lo:hi].copy_(host_in[w][lo:hi], non_blocking=True)
                    h["ev_in"][k][j].record(s)
                main.wait_event(h["ev_in"][k][j])
            if out:
                main.wait_event(h["ev_sent"][k])
            self._ring(plan, k, main)
            self._thc(plan, k, seed, main)
            h["ev_read"][k].record(main)
            if out:
                h["ev_out"][k].record(main)
                h["d2h"].wait_event(h["ev_out"][k])
                with torch.cuda.stream(h["d2h"]):
                    if host_ring is not None:
                        host_ring[lo:hi].copy_(self.ring_flat[0][lo:hi], non_blocking=True)
                    if host_thc is not None:
                        host_thc[lo:hi].copy_(self.thc_flat[lo:hi], non_blocking=True)
                    h["ev_sent"][k].record(h["d2h"])
        main.wait_event(h["ev_nmse_sent"])  # the previous step's NMSE is on the host
        self._nmse(main)
        h["ev_nmse"].record(main)
        if host_nmse is not None:
            h["d2h"].wait_event(h["ev_nmse"])
            with torch.cuda.stream(h["d2h"]):
                host_nmse.copy_(self.nmse, non_blocking=True)
                h["ev_nmse_sent"].record(h["d2h"])

    def bytes_from_host(self, host_ring=True, host_thc=True, host_nmse=True):
        """(host-to-device, device-to-host) bytes of one run_from_host step."""
        h2d = sum((p["hi"] - p["lo"]) * 4 for p in self.parts) * self.P
        d2h = (int(host_ring) + int(host_thc)) * sum((p["hi"] - p["lo"]) * 4 for p in self.parts) + 8 * int(host_nmse)
        return h2d, d2h
