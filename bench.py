"""Benchmark of the gradient-averaging hot path on GB300.

One step = one pass of the whole path over the ResNet-101-like Tensor
Fusion workload: P = 8 workers, 300 fp32 gradient tensors (~45M parameters,
log-uniform sizes 256..2.4M, N(0, 0.01)), 64 MB fusion buffers:

  1. fusion plan (host)                                    gar_fusion_plan
  2. per fusion buffer: Tensor Fusion + ring all-reduce     gar_fused_allreduce_range
     average in one pass (pack, ring, unpack), the buffer's
     THC range [min, max] taken from the same reads
  3. per fusion buffer: THC encode (every worker) +         gar_thc_allreduce_fused_plan
     integer aggregate + decode, read straight from the
     tensors, average written straight to the output
     tensors, wire vectors written (b = 4, fresh seed each step)
  4. NMSE of the THC average against the ring average:      gar_thc_allreduce_fused_plan_nmse,
     its sums taken inside step 3 (one more read of the     gar_nmse_combine
     ring average), then combined (--nmse separate: one     (gar_nmse)
     pass over both averages at the end)

The fused calls give bit for bit what pack -> ring / THC -> unpack gives
(the tests hold them to that); the fusion buffers are never materialised.
In the default two-stream schedule THC of buffer b runs while the ring
averages buffer b + 1.

Metric: gradient bytes reduced per second = P x 45M x 4 B per step / step
time (each step averages those bytes twice: exactly by the ring and
compressed by THC).  ``value`` is device-timed with inputs resident in HBM
(1.44 GB of inputs per step, larger than L2, so no L2 flush is needed).  The
same steps then run once more on one stream so each kernel is timed alone
for the roofline entry.  ``e2e`` runs the step from pinned host memory to
host memory: every step copies the workers' gradients in and both averages
and the NMSE out, pipelined by fusion buffer on separate copy streams.

``--impl reference`` times the CPU oracle (plain C) on a bounded sample of
the same workload, one process per host core over runs of the tensor list;
``cpu_baseline`` reports the same all-cores rate and the single-core one.  Under torchrun with N > 1 GPUs every rank runs
an independent replica (the path does not shard across GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "gradient GB/s reduced (P-worker ring + THC) and % of GB300 HBM peak"
UNIT = "GB/s"
P = 8
B_THC = 4
CAPACITY = 64 << 20
ALIGN = 16
WORKLOAD = "resnet_fusion"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _config(n_params, n_buffers, **extra):
    c = {"workload": "ResNet-101-like Tensor Fusion: P=8 workers x 300 fp32 tensors "
                     f"({n_params} params, log-uniform 256..2.4M, N(0,0.01)), 64 MB fusion buffers "
                     f"({n_buffers} buffers), ring average + uniform THC b=4 + NMSE",
         "P": P, "tensors": 300, "params_per_worker": int(n_params), "fusion_buffer_bytes": CAPACITY,
         "thc_bits": B_THC, "l2": "inputs larger than L2 (P x params x 4 B per step); no flush"}
    c.update(extra)
    return c


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest `value` over all ranks (every rank gets it); `value` itself
    when running alone.  `device`: where the reduction tensor lives (a CUDA
    device for NCCL, None for CPU backends such as gloo)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, f in zip(names, flags) if f.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ GPU (ours)
def make_step(dev, nmse="fused"):
    """The benchmark's workload on the device: every worker's 300 gradient
    tensors as 16-byte-aligned views of one flat buffer (as a framework's
    flat gradient buffer), seeded N(0, 0.01), and the bucketed averaging step
    over them (gradient_allreduce_homomorphic_gb300.pipeline)."""
    import torch

    from gradient_allreduce_homomorphic_gb300 import pipeline

    sizes = workloads.resnet_fusion_sizes()
    offs = pipeline.flat_offsets(sizes)
    cfg = workloads.CONFIG_IDS[WORKLOAD]
    flat = [workloads.device_normal(int(offs[-1]), 0.01, 1000 * cfg + w, torch.float32, dev) for w in range(P)]
    return pipeline.AveragingStep(flat, sizes, offs, b=B_THC, capacity_bytes=CAPACITY, align_bytes=ALIGN, nmse=nmse)


def step_seed(step_idx):
    return workloads.THC_SEED + step_idx


KERNEL_OF_STAGE = {
    "separate": {"ring": "ring_fold_kernel", "thc": "thc_fused_plan_kernel",
                 "nmse": "nmse_partial_kernel + nmse_final_kernel"},
    "fused": {"ring": "ring_fold_kernel", "thc": "thc_fused_plan_kernel (NMSE sums in the pass) + thc_nmse_pair_kernel",
              "nmse": "nmse_combine_kernel"},
}
PER_OF_STAGE = {
    "separate": {
        "ring": "all launches of one step's 3 gar_fused_allreduce_range calls (one per fusion buffer; "
                "300 tensors x 8 workers in all)",
        "thc": "all launches of one step's 3 gar_thc_allreduce_fused_plan calls (one per fusion buffer)",
        "nmse": "one step's gar_nmse over the flat averages"},
    "fused": {
        "ring": "all launches of one step's 3 gar_fused_allreduce_range calls (one per fusion buffer; "
                "300 tensors x 8 workers in all)",
        "thc": "all launches of one step's 3 gar_thc_allreduce_fused_plan_nmse calls (one per fusion buffer; "
               "NMSE sums against the ring average taken in the same pass)",
        "nmse": "one step's gar_nmse_combine of the 3 buffers' NMSE sums"},
}
# stage -> committed ncu summary holding its per-step DRAM traffic (the default, separate-NMSE step)
PROFILE_OF_STAGE = {"ring": ("ring_fold_kernel_range_resnet_fusion", ["ring.cu", "ring.cuh", "common.cuh"]),
                    "thc": ("thc_fused_plan_kernel_resnet_fusion", ["thc.cu", "thc_fused.cuh", "thc_p8.cu", "common.cuh"])}


def kernel_source_hash(files):
    """sha256 over the kernel's source files (the hash an ncu summary records)."""
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "gradient_allreduce_homomorphic_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def _profile_traffic(stage):
    """Per-step DRAM traffic of a stage from its committed ncu summary, only if
    the summary was taken on the current kernel source (else None)."""
    if stage not in PROFILE_OF_STAGE:
        return None
    tag, files = PROFILE_OF_STAGE[stage]
    path = os.path.join(ROOT, "profiles", f"{tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_step:\s*([0-9]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    return int(m.group(1)) if kernel_source_hash(files) == h.group(1) else None


def run_ours(args, rank, world, dist):
    import torch

    import gradient_allreduce_homomorphic_gb300 as g
    from gradient_allreduce_homomorphic_gb300.pipeline import STAGES

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g.load()
    st = make_step(dev, nmse=args.nmse)
    n_params = int(st.sizes.sum())
    nbytes = P * n_params * 4

    def barrier():
        if dist is not None:
            dist.barrier()

    def stage_events(n):
        return [{s: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for s in STAGES}
                for _ in range(n)]

    def mean_stage_ms(evs):
        return {s: float(np.mean([e[s][0].elapsed_time(e[s][1]) for e in evs])) for s in STAGES}

    for i in range(args.warmup):
        st.run(step_seed(i), args.schedule)
    torch.cuda.synchronize()

    # ---- device-timed region: inputs resident in HBM; no instrumentation
    # inside it (the stage breakdown below takes its own pass).  A spin
    # before the start event holds the stream while the host queues the K
    # steps, so that the events time the GPU's work and not the host's
    # queueing: the clock sampler's nvidia-smi queries can stall the host's
    # launches for tens of milliseconds (once seen: 2.45 ms a step against
    # 0.80), and a GPU that has run out of queued work would count that.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    launches0 = g.gar_launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(min(0.5e-3 * args.steps, 0.25) * 2.07e9))  # ~0.5 ms of SM cycles per step queued
    start.record()
    for i in range(args.steps):
        st.run(step_seed(args.warmup + i), args.schedule)
    stop.record()
    torch.cuda.synchronize()
    launches = g.gar_launch_count() - launches0
    barrier()
    clk = clocks.stop()
    ms = start.elapsed_time(stop) / args.steps
    ms = max_over_ranks(ms, dist, dev)

    # ---- the stages of the same steps, with a pair of events around each
    # stage (recording them costs a little, so not in the timed region)
    evs = stage_events(args.steps)
    for i in range(args.steps):
        st.run(step_seed(args.warmup + i), args.schedule, evs[i])
    torch.cuda.synchronize()
    stage_ms = mean_stage_ms(evs)
    overlap_evs = evs if args.schedule == "overlap" else None

    # ---- the same steps with every kernel alone on one stream: per-kernel
    # times for the roofline (in the two-stream schedule the ring and THC
    # kernels share HBM, so their individual durations stretch)
    serial_stage_ms = stage_ms
    if args.schedule == "overlap":
        for i in range(3):
            st.run(step_seed(20_000 + i), "serial")
        sevs = stage_events(args.steps)
        torch.cuda.synchronize()
        # the stage events time the GPU only if the launches are already
        # queued when it gets there: hold the stream with a spin (outside
        # every stage's events) while the host queues the next steps
        hold = int(0.015 * 2.07e9)  # about 15 ms of SM cycles
        for i in range(args.steps):
            if i % 10 == 0:
                torch.cuda._sleep(hold)
            st.run(step_seed(20_003 + i), "serial", sevs[i])
        torch.cuda.synchronize()
        serial_stage_ms = mean_stage_ms(sevs)

    # ---- the same step captured once in a CUDA graph and replayed K times
    # (the graph holds the two streams' fork, events and join; its THC seed
    # is the one it was captured with, so it is reported beside the eager
    # steps, each with its own seed, not instead of them)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            st.run(step_seed(30_000), args.schedule)
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(args.steps):
        graph.replay()
    g1.record()
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / args.steps
    del graph

    # ---- end to end: pinned host gradients in; both averages and the NMSE
    # out (and, beside it, the NMSE alone out)
    host_in = [torch.empty(st.flat_len, dtype=torch.float32, pin_memory=True) for _ in range(P)]
    for w in range(P):
        host_in[w].copy_(st.flat[w])
    host_ring = torch.empty(st.flat_len, dtype=torch.float32, pin_memory=True)
    host_thc = torch.empty(st.flat_len, dtype=torch.float32, pin_memory=True)
    host_nmse = torch.empty(1, dtype=torch.float64, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 20))
    st.setup_host(args.h2d_streams)

    def e2e_ms_per_step(averages):
        outs = (host_ring, host_thc) if averages else (None, None)
        st.host_begin()
        for i in range(3):
            st.run_from_host(step_seed(10_000 + i), host_in, *outs, host_nmse)
        st.host_end()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        st.host_begin()
        for i in range(e2e_steps):
            st.run_from_host(step_seed(10_003 + i), host_in, *outs, host_nmse)
        st.host_end()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)

    e2e_ms = e2e_ms_per_step(True)
    e2e_bytes = st.bytes_from_host(True, True, True)
    # the averages that came back are the step's: the THC average decodes to
    # within the range of its buffer, the ring average is finite
    assert np.isfinite(host_ring.numpy()).all() and np.isfinite(host_thc.numpy()).all()
    e2e_metric_ms = e2e_ms_per_step(False)
    metric_bytes = st.bytes_from_host(False, False, True)
    nmse_vals = host_nmse.numpy().tolist()
    assert all(np.isfinite(nmse_vals)), nmse_vals

    if rank != 0:
        return None
    peak, peak_kind = _peaks()
    algo = st.algorithmic_bytes()
    dom = max(serial_stage_ms, key=lambda s: serial_stage_ms[s])
    achieved = algo[dom] / (serial_stage_ms[dom] * 1e-3) / 1e9
    traffic = _profile_traffic(dom) if args.nmse == "separate" or dom == "ring" else None
    value = world * nbytes / (ms * 1e-3) / 1e9
    overlap_region = None
    if overlap_evs is not None:
        # ring and THC quantization share HBM: their combined bytes over the
        # span from the ring's start to the later of the two ends
        evs = overlap_evs
        span = float(np.mean([max(evs[i]["ring"][0].elapsed_time(evs[i]["ring"][1]),
                                  evs[i]["ring"][0].elapsed_time(evs[i]["thc"][1]))
                              for i in range(args.steps)]))
        both = algo["ring"] + algo["thc"]
        overlap_region = {"stages": ["ring", "thc"], "ms": round(span, 4),
                          "gbs": round(both / (span * 1e-3) / 1e9, 1),
                          "frac": round(both / (span * 1e-3) / 1e9 / peak, 4)}
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,0.01) gradients drawn on the device)",
        "config": _config(n_params, st.nb),
        "run": {"parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
                "schedule": ("two streams: THC of fusion buffer b overlapped with the ring of buffer b+1"
                             if args.schedule == "overlap" else "one stream, stages in sequence"),
                "path": "fused: pack + ring + unpack and pack + THC + unpack in one pass each, per fusion buffer",
                "nmse": "sums inside the THC pass" if args.nmse == "fused" else "one pass over both averages"},
        "elements_per_s": round(world * P * n_params / (ms * 1e-3), 1),
        "hbm_fraction_of_step": round(sum(algo.values()) / (ms * 1e-3) / 1e9 / peak, 4),
        "graph": {"ms_per_step": round(graph_ms, 4),
                  "value": round(world * P * n_params * 4 / (graph_ms * 1e-3) / 1e9, 2),
                  "what": "the step captured once in a CUDA graph, replayed K times (one THC seed)"},
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stage_ms_alone": {k: round(v, 4) for k, v in serial_stage_ms.items()},
        "stage_gbs_alone": {k: round(algo[k] / (serial_stage_ms[k] * 1e-3) / 1e9, 1) for k in serial_stage_ms},
        "overlap_region": overlap_region,
        "roofline": {"kernel": KERNEL_OF_STAGE[args.nmse][dom],
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "per": PER_OF_STAGE[args.nmse][dom], "stage": dom,
                     "timed": ("alone: the same steps run once more on one stream in this run, so the kernel "
                               "does not share HBM with a concurrent one" if args.schedule == "overlap"
                               else "in the timed steps")},
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": e2e_bytes[0],
                "d2h_bytes_per_step": e2e_bytes[1], "h2d_streams": args.h2d_streams,
                "readback": "both averages (exact and THC) and the NMSE, every step"},
        "e2e_metric_only": {"value": round(world * nbytes / (e2e_metric_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                            "ms_per_step": round(e2e_metric_ms, 4), "h2d_bytes_per_step": metric_bytes[0],
                            "d2h_bytes_per_step": metric_bytes[1],
                            "readback": "the NMSE only; the averages stay on the device"},
        "gpu_launches": int(launches),
        "nmse_thc_b4": round(nmse_vals[0], 6),
        "clocks": clk,
    }
    return out


# --------------------------------------------------------- CPU (oracle)
def oracle_step(sample_sizes, host, seed):
    """The same pass with the CPU oracle on a sample of the workload."""
    import oracle

    dt = np.zeros(sample_sizes.size, np.int32)
    sb, so, bn = oracle.fusion_plan(sample_sizes, dt, CAPACITY, ALIGN)
    nmses = []
    for b in range(len(bn)):
        fbs = [oracle.fusion_pack(host[w], sb, so, b, bn[b]) for w in range(P)]
        ring = oracle.ring_fold(fbs, op=oracle.AVG)
        oracle.fusion_unpack(ring, sb, so, sample_sizes, b)
        m, M = oracle.thc_range(fbs)
        avg = oracle.thc_allreduce(fbs, B_THC, seed, m, M)
        nmses.append(oracle.nmse(ring, avg.astype(np.float32)))
    return nmses


def sample_workload(target_params):
    sizes = workloads.resnet_fusion_sizes()
    take = []
    total = 0
    for s in sizes:  # a prefix of the tensor list, in ready order
        if total >= target_params and take:
            break
        take.append(int(s))
        total += int(s)
    ss = np.array(take, np.int64)
    cfg = workloads.CONFIG_IDS[WORKLOAD]
    host = [workloads.tensors_normal(ss, 0.01, cfg, w) for w in range(P)]
    return ss, host


def time_oracle(budget_s: float, reps: int):
    """Calibrate a sample so `reps` oracle steps take about budget_s seconds."""
    ss, host = sample_workload(600_000)  # larger than the host caches, so the rate holds
    t0 = time.perf_counter()
    oracle_step(ss, host, 1)
    rate = ss.sum() / max(time.perf_counter() - t0, 1e-6)  # params per second per step
    target = int(np.clip(0.8 * rate * budget_s / reps, 50_000, 45_000_000))
    ss, host = sample_workload(target)
    return ss, host


# All host cores: the oracle as it stands, one process per core, each running
# the same pass over its own run of the tensor list (its own fusion plan),
# started together at a barrier; the rate counts every process's parameters
# over the wall time from the first start to the last end.
def _slice_bounds(sizes, k):
    """k contiguous runs of the tensor list with about equal parameter counts."""
    cum = np.cumsum(sizes)
    cuts = [0]
    for j in range(1, k):
        cuts.append(min(max(int(np.searchsorted(cum, cum[-1] * j / k)), cuts[-1] + 1), len(sizes)))
    cuts.append(len(sizes))
    return [(cuts[j], cuts[j + 1]) for j in range(k) if cuts[j] < cuts[j + 1]]


def _slice_worker(conn, barrier, sizes, slot):
    """Child process: hold one slice's inputs, run steps on command."""
    import oracle

    oracle.build()
    cfg = workloads.CONFIG_IDS[WORKLOAD]
    host = [workloads.tensors_normal(sizes, 0.01, cfg, 1000 * (slot + 1) + w) for w in range(P)]
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            return
        try:
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            oracle_step(sizes, host, msg)
            conn.send((t0, time.perf_counter()))
        except Exception as e:  # reported to the parent, which stops the run
            conn.send(repr(e))


class ParallelOracle:
    """The oracle step over `sizes` (a prefix of the tensor list) cut into one
    run per process; `step(seed)` returns the wall time of one parallel step."""

    def __init__(self, sizes, procs):
        import multiprocessing as mp

        ctx = mp.get_context("spawn")
        runs = _slice_bounds(np.asarray(sizes, np.int64), procs)
        self.barrier = ctx.Barrier(len(runs))
        self.params = int(np.sum(sizes))
        self.procs, self.conns = [], []
        for slot, (i0, i1) in enumerate(runs):
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_slice_worker, args=(b, self.barrier, np.asarray(sizes[i0:i1], np.int64), slot),
                             daemon=True)
            pr.start()
            self.procs.append(pr)
            self.conns.append(a)
        for c in self.conns:
            if self._recv(c, 600) != "ready":
                self.close()
                raise RuntimeError("oracle slice process did not start")

    def step(self, seed):
        for c in self.conns:
            c.send(seed)
        spans = []
        for c in self.conns:
            r = self._recv(c, 3600)
            if not isinstance(r, tuple):
                self.close()
                raise RuntimeError(f"oracle slice process failed: {r}")
            spans.append(r)
        return max(t1 for _, t1 in spans) - min(t0 for t0, _ in spans)

    @staticmethod
    def _recv(conn, timeout):
        """The child's next message, or None if it died or stayed silent."""
        try:
            return conn.recv() if conn.poll(timeout) else None
        except (EOFError, OSError):
            return None

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for pr in self.procs:
            pr.join(timeout=10)
            if pr.is_alive():
                pr.terminate()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_all_cores(budget_s=15.0):
    """One parallel oracle step over a prefix of the workload sized so that
    it takes about budget_s seconds on all host cores."""
    procs = host_cores()
    ss, _ = time_oracle(budget_s * procs, 1)
    po = ParallelOracle(ss, procs)
    try:
        dt = po.step(workloads.THC_SEED)
    finally:
        po.close()
    n = int(ss.sum())
    return {"value": round(P * n * 4 / dt / 1e9, 4), "cores": len(po.procs), "seconds": round(dt, 2),
            "sample": f"first {ss.size} of the 300 tensors ({n} params per worker, P=8), cut into "
                      f"{len(po.procs)} runs of tensors, one oracle process each, started together"}


def cpu_baseline(budget_s=15.0):
    ss, host = time_oracle(budget_s, 1)
    t0 = time.perf_counter()
    oracle_step(ss, host, workloads.THC_SEED)
    dt = time.perf_counter() - t0
    n = int(ss.sum())
    one = {"value": round(P * n * 4 / dt / 1e9, 4), "cores": 1,
           "sample": f"first {ss.size} of the 300 tensors ({n} params per worker, P=8), one full step "
                     f"(plan, pack, ring fold, unpack, THC range + encode/aggregate/decode, NMSE), {dt:.1f} s"}
    try:
        allc = cpu_baseline_all_cores(budget_s)
    except Exception as e:  # the single-core figure still stands
        allc = None
        one["all_cores_error"] = repr(e)[:200]
    if allc is None or allc["cores"] < 2:
        return {"value": one["value"], "unit": UNIT, "cores": 1, "kind": "oracle", "sample": one["sample"],
                **({"all_cores_error": one["all_cores_error"]} if "all_cores_error" in one else {})}
    return {"value": allc["value"], "unit": UNIT, "cores": allc["cores"], "kind": "oracle",
            "sample": allc["sample"] + f", {allc['seconds']} s", "single_core": one}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle

    oracle.build()
    budget = float(args.reference_budget_s)  # seconds of oracle work for the whole --steps/--warmup run
    reps = args.steps + args.warmup
    procs = host_cores()
    ss, _ = time_oracle(budget * procs, reps)
    po = ParallelOracle(ss, procs)
    try:
        for i in range(args.warmup):
            po.step(workloads.THC_SEED + i)
        times = [po.step(workloads.THC_SEED + args.warmup + i) for i in range(args.steps)]
    finally:
        po.close()
    ms = float(np.mean(times)) * 1e3
    n = int(ss.sum())
    full = workloads.resnet_fusion_sizes()
    value = P * n * 4 / (ms * 1e-3) / 1e9
    cores = len(po.procs)
    sample = (f"first {ss.size} of the 300 tensors ({n} params per worker, P=8) per step, cut into {cores} runs "
              f"of tensors (one oracle process per host core, started together), sized so {reps} steps fit in "
              f"~{budget:.0f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy N(0,0.01))",
            "config": _config(int(full.sum()), int(len(oracle.fusion_plan(full, np.zeros(full.size, np.int32),
                                                                          CAPACITY, ALIGN)[2]))),
            "run": {"reference": f"CPU oracle (plain C), {cores} processes"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------- all five workloads
def _median_ms(torch, fn, iters, flush=None):
    """Median device time of fn() over `iters` calls (CUDA events on the
    current stream, 3 warm-up calls); `flush` runs untimed before each call."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(iters):
        if flush is not None:
            flush()
        torch.cuda._sleep(100_000)  # the call is queued before the start event: the events time the GPU
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return float(np.median(times))


def _gpu_line(name, ms, nbytes, inbytes, elems, peak):
    return {"ms": round(ms, 4), "gbs_reduced": round(inbytes / (ms * 1e-3) / 1e9, 1),
            "elements_per_s": round(elems / (ms * 1e-3), 1),
            "algorithmic_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "what": name}


def _cpu_time(fn, reps=3):
    """Median wall time of fn() (the oracle, one core) over `reps` calls."""
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    return float(np.median(ts))


def run_configs(args):
    """Every workload of the pages' configurations on this GPU through the
    library (one JSON line each), with the oracle timed on one host core on a
    bounded sample of the same workload."""
    import torch

    import gradient_allreduce_homomorphic_gb300 as g

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g.load()
    peak, _ = _peaks()
    it = args.config_iters
    l2 = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)  # 256 MB > the 129 MB L2
    l2_clean = torch.ones_like(l2)

    def flush():
        # 256 MB written (the inputs leave L2), then 256 MB read, so that the
        # dirty lines are written back before the timed call starts
        l2.zero_()
        l2_clean.sum()
    oracle = None
    if not args.no_cpu_baseline:
        import oracle

        oracle.build()
    out = []
    seed = workloads.THC_SEED
    cores = 1

    # C1: four workers, one 4 MB partition (fits in L2: flushed before each call)
    P, N = 4, 1 << 20
    cfg = workloads.CONFIG_IDS["partition_4mb"]
    x = [workloads.device_normal(N, 1.0, 1000 * cfg + w, torch.float32, dev) for w in range(P)]
    buf = [t.clone() for t in x]
    tb, tx = g.pointer_table(buf), g.pointer_table(x)
    mM = torch.empty(2, device=dev)
    avg = torch.empty(N, device=dev)
    words = g.gar_thc_words(N, 4)
    packed = [torch.empty(words, dtype=torch.int32, device=dev) for _ in range(P)]
    tp = g.pointer_table(packed)
    ring_ms = _median_ms(torch, lambda: g.gar_ring_allreduce_sim(tb), it, flush)

    def thc():
        g.gar_thc_range(tx, mM)
        g.gar_thc_allreduce_fused(tx, 4, seed, mM, avg, tp)

    thc_ms = _median_ms(torch, thc, it, flush)
    line = {"config": "partition_4mb: P=4, N=2^20 fp32 N(0,1); ring average + THC b=4 (range, fused)",
            "l2": "flushed before each call (256 MB written, then 256 MB read)",
            "gpu": {"ring": _gpu_line("gar_ring_allreduce_sim, in place", ring_ms, 2 * P * N * 4, P * N * 4,
                                      P * N, peak),
                    "thc": _gpu_line("gar_thc_range + gar_thc_allreduce_fused (wire vectors written)", thc_ms,
                                     P * N * 4 + P * N * 4 + N * 4 + P * words * 4, P * N * 4, P * N, peak)}}
    if oracle is not None:
        n = 1 << 18
        hx = workloads.workers_normal(P, n, 1.0, cfg)
        t_ring = _cpu_time(lambda: oracle.ring_fold(hx))
        t_thc = _cpu_time(lambda: oracle.thc_allreduce(hx, 4, seed))
        line["oracle"] = {"sample": f"P=4 x 2^18", "cores": cores,
                          "ring_gbs": round(P * n * 4 / t_ring / 1e9, 4),
                          "thc_gbs": round(P * n * 4 / t_thc / 1e9, 4)}
    out.append(line)
    del x, buf, packed, avg
    torch.cuda.empty_cache()

    # C1 as THC runs it on a model: a stream of 64 partitions of 4 MB per
    # worker, each its own fusion buffer with its own range, one call each for
    # the ring (with the ranges) and for THC over the stream (1 GB of inputs)
    k = 64
    sizes = np.full(k, N, np.int64)
    plan = g.gar_fusion_plan(sizes, np.zeros(k, np.int32), N * 4, ALIGN)
    src = [[workloads.device_normal(N, 1.0, 100_000 * (w + 1) + i, torch.float32, dev) for i in range(k)]
           for w in range(P)]
    dst = [[torch.empty_like(t) for t in row] for row in src]
    smM = torch.empty((k, 2), device=dev)
    tabs = g.fused_pointer_tables(src, dst)
    spk = [[torch.empty(words, dtype=torch.int32, device=dev) for _ in range(k)] for _ in range(P)]
    stt = g.thc_plan_tables(src, dst[0], spk)
    sring_ms = _median_ms(torch, lambda: g.gar_fused_allreduce_range(src, dst, plan, smM, tables=tabs), it)
    sthc_ms = _median_ms(torch, lambda: g.gar_thc_allreduce_fused_plan(src, plan, 4, seed, smM, dst[0], tables=stt),
                         it)
    out.append({"config": "partition_4mb as a stream: P=4, 64 partitions of 2^20 fp32 N(0,1) per worker, each its "
                          "own fusion buffer and range; ring average with the ranges, then THC b=4 over the stream",
                "l2": "inputs (1 GB) larger than L2",
                "gpu": {"ring": _gpu_line("gar_fused_allreduce_range over the 64 partitions", sring_ms,
                                          2 * P * N * 4 * k, P * N * 4 * k, P * N * k, peak),
                        "thc": _gpu_line("gar_thc_allreduce_fused_plan over the 64 partitions (wire vectors written)",
                                         sthc_ms, (P * N * 4 + N * 4 + P * words * 4) * k, P * N * 4 * k, P * N * k,
                                         peak)}})
    del src, dst, spk, stt, tabs
    torch.cuda.empty_cache()

    # C2: the main benchmark's workload and step (two streams)
    st = make_step(dev)
    for i in range(3):
        st.run(step_seed(i))
    step_ms = _median_ms(torch, lambda: st.run(step_seed(7)), it)
    algo = st.algorithmic_bytes()
    line = {"config": "resnet_fusion: P=8, 300 fp32 tensors (45M params), 64 MB fusion buffers; ring average "
                      "with range + THC b=4 over the plan + NMSE (the main benchmark step)",
            "l2": "inputs (1.44 GB) larger than L2",
            "gpu": {"step": _gpu_line("one bench step", step_ms, sum(algo.values()), 8 * int(st.sizes.sum()) * 4,
                                      8 * int(st.sizes.sum()), peak)}}
    if oracle is not None:
        ss, host = sample_workload(300_000)
        t = _cpu_time(lambda: oracle_step(ss, host, seed), reps=1)
        line["oracle"] = {"sample": f"first {ss.size} tensors ({int(ss.sum())} params) x 8 workers, one step",
                          "cores": cores, "step_gbs": round(8 * int(ss.sum()) * 4 / t / 1e9, 4)}
    out.append(line)
    del st
    torch.cuda.empty_cache()

    # C3: VGG-16-like, communication bound: fused pack + ring + unpack, in place
    P = 8
    cfg = workloads.CONFIG_IDS["vgg_fusion"]
    sizes = workloads.vgg_fusion_sizes()
    n = int(sizes.sum())
    dt = np.zeros(sizes.size, np.int32)
    plan = g.gar_fusion_plan(sizes, dt, CAPACITY, ALIGN)
    flat = [workloads.device_normal(n, 1e-3, 1000 * cfg + w, torch.float32, dev) for w in range(P)]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    src = [[f[int(offs[i]):int(offs[i + 1])] for i in range(sizes.size)] for f in flat]
    tables = g.fused_pointer_tables(src, src)
    ms = _median_ms(torch, lambda: g.gar_fused_allreduce(src, src, plan, tables=tables), it)
    line = {"config": "vgg_fusion: P=8, 16 fp32 tensors (138M params, largest 102.8M), 64 MB fusion buffers; "
                      "fused pack + ring average + unpack, in place",
            "l2": "inputs (4.4 GB) larger than L2",
            "gpu": {"fused_ring": _gpu_line("gar_fused_allreduce", ms, 2 * P * n * 4, P * n * 4, P * n, peak)}}
    if oracle is not None:
        ss = sizes[:6]
        hs = [workloads.tensors_normal(ss, 1e-3, cfg, w) for w in range(P)]

        def vgg_oracle():
            sb, so, bn = oracle.fusion_plan(ss, np.zeros(ss.size, np.int32), CAPACITY, ALIGN)
            for b in range(len(bn)):
                fbs = [oracle.fusion_pack(hs[w], sb, so, b, bn[b]) for w in range(P)]
                oracle.fusion_unpack(oracle.ring_fold(fbs), sb, so, ss, b)

        t = _cpu_time(vgg_oracle, reps=1)
        line["oracle"] = {"sample": f"first 6 tensors ({int(ss.sum())} params) x 8 workers", "cores": cores,
                          "fused_ring_gbs": round(P * int(ss.sum()) * 4 / t / 1e9, 4)}
    out.append(line)
    del flat, src, tables
    torch.cuda.empty_cache()

    # C4: THC sweep on heavy-tailed gradients, P in {4, 16, 64}, b in {2, 4, 8}
    N = 1 << 24
    cfg = workloads.CONFIG_IDS["thc_sweep"]
    sweep = []
    for P in (4, 16, 64):
        x = [workloads.device_student_t(N, 3, 1e-3, 1000 * cfg + w, dev) for w in range(P)]
        tx = g.pointer_table(x)
        exact = torch.empty(N, device=dev)
        g.gar_ring_allreduce_sim_out(tx, g.pointer_table([exact]))
        mM = torch.empty(2, device=dev)
        avg = torch.empty(N, device=dev)
        nm = torch.empty(1, dtype=torch.float64, device=dev)
        ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8 + 1, dtype=torch.float64, device=dev)
        range_ms = _median_ms(torch, lambda: g.gar_thc_range(tx, mM), it)
        nmse_ms = _median_ms(torch, lambda: g.gar_nmse(exact, avg, nm, ws), it)
        for b in (2, 4, 8):
            words = g.gar_thc_words(N, b)
            packed = [torch.empty(words, dtype=torch.int32, device=dev) for _ in range(P)]
            tp = g.pointer_table(packed)
            fused_ms = _median_ms(torch, lambda: g.gar_thc_allreduce_fused(tx, b, seed, mM, avg, tp), it)
            g.gar_nmse(exact, avg, nm, ws)
            torch.cuda.synchronize()
            fb = P * N * 4 + N * 4 + P * words * 4
            sweep.append({"P": P, "b": b, "nmse": round(float(nm.item()), 6),
                          "range": _gpu_line("gar_thc_range", range_ms, P * N * 4, P * N * 4, P * N, peak),
                          "fused": _gpu_line("gar_thc_allreduce_fused (wire vectors written)", fused_ms, fb,
                                             P * N * 4, P * N, peak),
                          "nmse_kernel": _gpu_line("gar_nmse", nmse_ms, 2 * N * 4, 2 * N * 4, N, peak),
                          "round_gbs_reduced": round(P * N * 4 / ((range_ms + fused_ms) * 1e-3) / 1e9, 1)})
            del packed
        del x, exact
        torch.cuda.empty_cache()
    line = {"config": "thc_sweep: N=2^24 fp32 Student-t(3) x 1e-3 per worker, P in {4,16,64}, b in {2,4,8}; "
                      "range, fused encode/aggregate/decode, NMSE against the exact (ring) average",
            "l2": "inputs (256 MB to 4 GB) larger than L2", "gpu": sweep}
    if oracle is not None:
        n = 1 << 16
        o = []
        for P in (4, 16, 64):
            hx = [workloads.student_t_f32(n, 3, 1e-3, cfg, w) for w in range(P)]
            t = _cpu_time(lambda: oracle.thc_allreduce(hx, 4, seed), reps=1)
            o.append({"P": P, "b": 4, "thc_gbs": round(P * n * 4 / t / 1e9, 4)})
        line["oracle"] = {"sample": "N=2^16 per worker", "cores": cores, "thc": o}
    out.append(line)

    # C5: large bf16 bucket: P=16 x 2^28 bf16, fp32 accumulation in ring order
    P, N = 16, 1 << 28
    cfg = workloads.CONFIG_IDS["large_bf16"]
    x = [workloads.device_normal(N, 1e-2, 1000 * cfg + w, torch.bfloat16, dev) for w in range(P)]
    tx = g.pointer_table(x)
    reps = max(3, it // 4)
    ms = _median_ms(torch, lambda: g.gar_ring_allreduce_sim(tx), reps)
    bidir_ms = _median_ms(torch, lambda: g.gar_ring_allreduce_bidir(tx), reps)
    tree_ms = _median_ms(torch, lambda: g.gar_dbtree_allreduce(tx), reps)
    ab = 2 * P * N * 2  # every input read, every buffer written
    line = {"config": "large_bf16: P=16, N=2^28 bf16 N(0, 1e-2) per worker (8 GiB); ring average in place, "
                      "fp32 accumulation in ring order, bf16 out; the bidirectional ring and the double binary "
                      "tree (other fold orders) on the same buffers",
            "l2": "inputs (8 GiB) larger than L2",
            "gpu": {"ring": _gpu_line("gar_ring_allreduce_sim (bf16)", ms, ab, P * N * 2, P * N, peak),
                    "bidir": _gpu_line("gar_ring_allreduce_bidir (bf16)", bidir_ms, ab, P * N * 2, P * N, peak),
                    "dbtree": _gpu_line("gar_dbtree_allreduce (bf16)", tree_ms, ab, P * N * 2, P * N, peak)}}
    if oracle is not None:
        n = 1 << 18
        hx = [workloads.normal_f32(n, 1e-2, cfg, w) for w in range(P)]
        hb = [(a.view(np.uint32) >> 16).astype(np.uint16) for a in hx]  # bf16 bits (truncated): timing input only
        t = _cpu_time(lambda: oracle.ring_fold(hb))
        t_tree = _cpu_time(lambda: oracle.dbtree_fold(hb))
        line["oracle"] = {"sample": "P=16 x 2^18", "cores": cores, "ring_gbs": round(P * n * 2 / t / 1e9, 4),
                          "dbtree_gbs": round(P * n * 2 / t_tree / 1e9, 4)}
    out.append(line)
    del x
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", choices=["overlap", "serial"], default="overlap")
    ap.add_argument("--h2d-streams", type=int, default=2, help="copy streams for the end-to-end inputs")
    ap.add_argument("--nmse", choices=["fused", "separate"], default="fused",
                    help="NMSE sums inside the THC pass, or one NMSE pass over both averages at the end")
    ap.add_argument("--reference-budget-s", type=float, default=100.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--configs", action="store_true",
                    help="time every workload configuration (one JSON line each) instead of the benchmark step")
    ap.add_argument("--config-iters", type=int, default=20)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.configs:
        for line in run_configs(args):
            print(json.dumps(line))
        return
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist

            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
        out = run_ours(args, rank, world, dist)
        if out is not None and world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline()
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
