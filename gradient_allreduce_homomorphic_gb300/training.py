"""One step of THC's training process ([T] section 5) for P workers'
gradient vectors of n values, through the library's fused entry points, the
workers' chains spread over CUDA streams.

Per step ([T] section 5, error feedback around the rotation and the
quantization):

  1. per worker: x = grad + e, rotated, y = (1/sqrt n) H D x, with     gar_rht_ef_forward
     the sums of squares of x per 4096-element tile
  2. the norm-based range [-M, M], M = (t_p / sqrt n) max ||x_w||     gar_rht_norm_range_from_sums
     (the rotation keeps norms, so the sums of x serve)
  3. THC of the rotated vectors: every worker's wire vector, their     gar_nuhc_allreduce_fused
     sum and the decoded average (non-uniform with a table T on a      (gar_thc_allreduce_fused)
     granularity-g grid, or uniform)
  4. the average rotated back: the gradient estimate                   gar_rht (inverse)
  5. per worker: e = x - (1/sqrt n) D H decode(own wire vector)       gar_rht_ef_update

Steps 1 and 5 are P independent chains (each touches only its own worker's
buffers, and each stream has its own scratch vector for step 5), so they go
round-robin over `streams` side streams: one worker's cluster pass of the
transform (bound by its cluster barriers, not by HBM) runs beside another's
tile pass (bound by HBM).  Steps 2-4 run on the caller's stream, which waits
for every side stream before step 2, and the side streams wait for it before
step 5; the caller's stream waits for them at the end of the step.  With one
stream the step is the plain sequence of calls; every stream count gives the
same results bit for bit (the calls and their inputs do not change, only
their order across independent workers).

Everything here is host-side orchestration of streams and events; each step
of the arithmetic runs in the library's CUDA kernels.  Buffers are allocated
once, at construction; a step allocates nothing on the device.
"""
from __future__ import annotations

import numpy as np

from . import (gar_nuhc_allreduce_fused, gar_rht, gar_rht_ef_forward, gar_rht_ef_update,
               gar_rht_norm_range_from_sums, gar_rht_tiles, gar_thc_allreduce_fused, gar_thc_words,
               pointer_table)


class TrainingStep:
    """Device-resident state of THC's training step for P workers.

    grads, errs: P fp32 CUDA tensors of n elements each (n a power of two),
    the workers' gradients and error-feedback vectors; ``errs`` are updated in
    place by every step.  b: bits per index; table: the non-uniform table T
    (2^b increasing integers from 0 to g, numpy uint16), or None for uniform
    THC (g = 2^b - 1); t_p: the truncation point of the norm-based range;
    rht_seed keys the rotation's signs.  After ``run(seed)``: ``ys[w]`` the
    rotated vectors, ``packed[w]`` the wire vectors, ``mM`` the range,
    ``avg`` the decoded average in the rotated domain and ``est`` the
    gradient estimate (the average rotated back).
    """

    def __init__(self, grads, errs, *, b: int = 4, table=None, t_p: float = 2.15, rht_seed: int = 11,
                 streams: int = 2):
        import torch

        if len(grads) != len(errs) or not grads:
            raise ValueError("grads and errs must be two non-empty lists of the same length")
        self.P, self.n = len(grads), int(grads[0].numel())
        if self.n < 1 or self.n & (self.n - 1):
            raise ValueError(f"n={self.n} is not a power of two")
        if streams < 1:
            raise ValueError("streams must be at least 1")
        self.grads, self.errs = list(grads), list(errs)
        self.b, self.t_p, self.rht_seed = b, float(t_p), rht_seed
        self.table = None if table is None else np.asarray(table, np.uint16)
        self.g = (1 << b) - 1 if self.table is None else int(self.table[-1])
        dev = self.device = grads[0].device
        self.ys = [torch.empty(self.n, device=dev) for _ in range(self.P)]
        self.packed = [torch.empty(max(gar_thc_words(self.n, b), 1), dtype=torch.int32, device=dev)
                       for _ in range(self.P)]
        self.sums = [torch.empty(gar_rht_tiles(self.n), dtype=torch.float64, device=dev) for _ in range(self.P)]
        self.mM = torch.empty(2, device=dev)
        self.avg = torch.empty(self.n, device=dev)
        self.est = torch.empty(self.n, device=dev)
        self.streams = [torch.cuda.Stream(device=dev) for _ in range(streams)] if streams > 1 else []
        nscratch = max(1, len(self.streams))
        self.tmp = [torch.empty(self.n, device=dev) for _ in range(nscratch)]
        self._ys_t, self._pk_t, self._sums_t = (pointer_table(self.ys), pointer_table(self.packed),
                                                pointer_table(self.sums))

    def _stream_of(self, w):
        return self.streams[w % len(self.streams)] if self.streams else None

    def _fork(self, main):
        for s in self.streams:
            s.wait_stream(main)

    def _join(self, main):
        for s in self.streams:
            main.wait_stream(s)

    def run(self, seed: int):
        """One step on the caller's current stream (the side streams fork
        from it and join it); THC's draws are keyed by `seed`."""
        import torch

        main = torch.cuda.current_stream(self.device)
        self._fork(main)
        for w in range(self.P):
            gar_rht_ef_forward(self.grads[w], self.errs[w], self.ys[w], self.rht_seed, self.sums[w],
                               stream=self._stream_of(w))
        self._join(main)
        gar_rht_norm_range_from_sums(self._sums_t, self.n, self.t_p, self.mM)
        if self.table is None:
            gar_thc_allreduce_fused(self._ys_t, self.b, seed, self.mM, self.avg, self._pk_t)
        else:
            gar_nuhc_allreduce_fused(self._ys_t, self.b, self.g, self.table, seed, self.mM, self.avg, self._pk_t)
        self._fork(main)
        gar_rht(self.avg, self.est, self.rht_seed, inverse=True)
        for w in range(self.P):
            k = w % len(self.streams) if self.streams else 0
            gar_rht_ef_update(self.packed[w], self.b, self.g, self.table, self.mM, self.grads[w], self.errs[w],
                              self.tmp[k], self.rht_seed, stream=self._stream_of(w))
        self._join(main)

    def algorithmic_bytes(self) -> int:
        """HBM bytes one step must move: per worker grad and e read, y
        written, y read by THC, the wire vector written and read, grad and e
        read and e written again; once the average written, read and its
        rotation written."""
        words = gar_thc_words(self.n, self.b)
        return self.P * self.n * 4 * 7 + self.P * 2 * words * 4 + 3 * self.n * 4
