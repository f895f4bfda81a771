"""Per-kernel microbenchmark of libgar.so on one GPU.

    python -m gradient_allreduce_homomorphic_gb300.microbench <case> [--P 8] [--N 16777216]
           [--b 4] [--iters 20] [--warmup 3] [--dtype f32|bf16]

Cases: ring (in-place ring all-reduce of P buffers), ring_out (reduce to one
output), stream_ring, stream_thc (a stream of --k partitions of N values per
worker, each its own fusion buffer and range: the ring with the ranges, or
THC with wire vectors, one call over the stream), bidir (bidirectional dual ring), dbtree (double-binary-tree all-reduce), fused (plan-driven all-reduce of the 300-tensor ResNet-like model),
fused_range (the same into separate outputs, each buffer's THC range from the same reads), thc_plan
(THC b-bit of every fusion buffer of that model read straight from the tensors, wire vectors written),
thc_plan_nmse (the same with the NMSE sums against a reference taken in the pass),
pack, unpack (per worker and buffer), pack_all, pack_all_range (every worker
in one call, with THC's range fused in), thc_range, thc_encode, thc_aggregate, thc_decode, thc_fused,
thc_fused_packed, nuhc_fused, nuhc_fused_packed (non-uniform THC with a
table on a granularity-g grid), nmse, train_step, train_step_fused (one step
of THC's training process over P workers: error feedback, rotation, range,
non-uniform THC, inverse rotation, error-feedback update; separate calls, or
the fused ones as training.TrainingStep runs them, the workers' chains over
--streams side streams).  Inputs are seeded N(0, 1) draws made on the device;
every size is chosen by the caller, so a case can be kept small enough for a
profiler capture.  Prints one JSON line: time per call (CUDA events on the
launching stream, after warm-up) and algorithmic GB/s.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)


def main(argv=None):
    import torch

    import gradient_allreduce_homomorphic_gb300 as g
    import workloads

    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--N", type=int, default=1 << 24)
    ap.add_argument("--b", type=int, default=4)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--dtype", default="f32")
    ap.add_argument("--g", type=int, default=0, help="granularity for the nuhc cases")
    ap.add_argument("--k", type=int, default=64, help="partitions of the stream cases")
    ap.add_argument("--streams", type=int, default=2,
                    help="train_step_fused: side streams the workers' chains go round-robin over")
    ap.add_argument("--flush", action="store_true",
                    help="write then read 256 MB (more than L2) before every timed call")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g.load()
    P, N, b = a.P, a.N, a.b
    tdt = torch.float32 if a.dtype == "f32" else torch.bfloat16
    es = 4 if a.dtype == "f32" else 2

    def bufs(n, k, dt=tdt, seed=0):
        return [workloads.device_normal(n, 1.0, 77_000 + seed + i, dt, dev) for i in range(k)]

    if a.case in ("ring", "ring_out", "bidir", "dbtree"):
        x = bufs(N, P)
        if a.case == "ring":
            t = g.pointer_table(x)
            fn = lambda: g.gar_ring_allreduce_sim(t)  # noqa: E731
            nbytes = 2 * P * N * es
        elif a.case == "bidir":
            t = g.pointer_table(x)
            fn = lambda: g.gar_ring_allreduce_bidir(t)  # noqa: E731
            nbytes = 2 * P * N * es
        elif a.case == "dbtree":
            t = g.pointer_table(x)
            fn = lambda: g.gar_dbtree_allreduce(t)  # noqa: E731
            nbytes = 2 * P * N * es
        else:
            out = [torch.empty(N, dtype=tdt, device=dev)]
            t, o = g.pointer_table(x), g.pointer_table(out)
            fn = lambda: g.gar_ring_allreduce_sim_out(t, o)  # noqa: E731
            nbytes = P * N * es + N * es
    elif a.case in ("stream_ring", "stream_thc"):
        # a stream of k partitions of N fp32 per worker, each its own fusion
        # buffer with its own range: the ring with the ranges (stream_ring),
        # or THC b-bit of every partition with wire vectors (stream_thc), one
        # call over the whole stream
        sizes = np.full(a.k, N, np.int64)
        plan = g.gar_fusion_plan(sizes, np.zeros(a.k, np.int32), N * 4, 16)
        src = [[workloads.device_normal(N, 1.0, 3000 * w + i, torch.float32, dev) for i in range(a.k)]
               for w in range(P)]
        dst = [[torch.empty_like(t) for t in row] for row in src]
        mM = torch.empty((a.k, 2), device=dev)
        tables = g.fused_pointer_tables(src, dst)
        g.gar_fused_allreduce_range(src, dst, plan, mM, tables=tables)
        if a.case == "stream_ring":
            fn = lambda: g.gar_fused_allreduce_range(src, dst, plan, mM, tables=tables)  # noqa: E731
            nbytes = 2 * P * N * 4 * a.k
        else:
            words = g.gar_thc_words(N, b)
            packed = [[torch.empty(words, dtype=torch.int32, device=dev) for _ in range(a.k)] for _ in range(P)]
            tt = g.thc_plan_tables(src, dst[0], packed)
            fn = lambda: g.gar_thc_allreduce_fused_plan(src, plan, b, 5, mM, dst[0], tables=tt)  # noqa: E731
            nbytes = (P * N * 4 + N * 4 + P * words * 4) * a.k
    elif a.case in ("fused", "fused_range", "thc_plan", "thc_plan_nmse", "pack", "unpack", "pack_all",
                    "pack_all_range"):
        sizes = workloads.resnet_fusion_sizes()
        dt = np.zeros(sizes.size, np.int32)
        plan = g.gar_fusion_plan(sizes, dt, 64 << 20, 16)
        n = int(sizes.sum())
        src = [[workloads.device_normal(int(s), 1.0, 1000 * w + i, torch.float32, dev) for i, s in enumerate(sizes)]
               for w in range(P)]
        if a.case == "fused":
            tables = g.fused_pointer_tables(src, src)
            fn = lambda: g.gar_fused_allreduce(src, src, plan, tables=tables)  # noqa: E731
            nbytes = 2 * P * n * 4
        elif a.case in ("fused_range", "thc_plan", "thc_plan_nmse"):
            dst = [[torch.empty_like(t) for t in row] for row in src]
            mM = torch.empty((plan.n_buffers, 2), device=dev)
            tables = g.fused_pointer_tables(src, dst)
            g.gar_fused_allreduce_range(src, dst, plan, mM, tables=tables)
            if a.case == "fused_range":
                fn = lambda: g.gar_fused_allreduce_range(src, dst, plan, mM, tables=tables)  # noqa: E731
                nbytes = 2 * P * n * 4
            else:
                out = dst[0]
                words = [g.gar_thc_words(int(k), b) for k in plan.buf_numel]
                packed = [[torch.empty(k, dtype=torch.int32, device=dev) for k in words] for _ in range(P)]
                tt = g.thc_plan_tables(src, out, packed)
                if a.case == "thc_plan":
                    fn = lambda: g.gar_thc_allreduce_fused_plan(src, plan, b, 5, mM, out, tables=tt)  # noqa: E731
                    nbytes = P * n * 4 + n * 4 + P * sum(words) * 4
                else:  # with the NMSE sums against worker 1's ring output as reference
                    ws = torch.empty(g.gar_thc_plan_nmse_workspace_bytes(plan, b) // 8 + 1, dtype=torch.float64,
                                     device=dev)
                    pair = torch.empty(2, dtype=torch.float64, device=dev)
                    rt = g.pointer_table(dst[1])
                    fn = lambda: g.gar_thc_allreduce_fused_plan_nmse(  # noqa: E731
                        src, plan, b, 5, mM, out, None, pair, ws, tables=tt, ref_table=rt)
                    nbytes = P * n * 4 + 2 * n * 4 + P * sum(words) * 4
        elif a.case.startswith("pack_all"):
            fbs = [[torch.empty(int(k), device=dev) for k in plan.buf_numel] for _ in range(P)]
            mM = torch.empty((plan.n_buffers, 2), device=dev) if a.case == "pack_all_range" else None
            tables = g.pack_all_tables(src, fbs)
            fn = lambda: g.gar_fusion_pack_all(src, plan, fbs, mM, tables=tables)  # noqa: E731
            nbytes = P * (n + int(plan.buf_numel.sum())) * 4
        else:
            fbs = [[torch.empty(int(k), device=dev) for k in plan.buf_numel] for _ in range(P)]
            tabs = [g.pointer_table(src[w]) for w in range(P)]

            def fn():
                for w in range(P):
                    for bb in range(plan.n_buffers):
                        if a.case == "pack":
                            g.gar_fusion_pack(tabs[w], plan, bb, fbs[w][bb])
                        else:
                            g.gar_fusion_unpack(fbs[w][bb], plan, bb, tabs[w])

            nbytes = P * (n + int(plan.buf_numel.sum())) * 4 if a.case == "pack" else 2 * P * n * 4
    elif a.case.startswith(("thc", "nuhc")) or a.case == "nmse":
        x = bufs(N, P, torch.float32)
        mM = torch.empty(2, device=dev)
        g.gar_thc_range(x, mM)
        words = g.gar_thc_words(N, b)
        packed = [torch.zeros(words, dtype=torch.int32, device=dev) for _ in range(P)]
        sums = torch.zeros(N, dtype=torch.int16, device=dev)
        avg = torch.empty(N, device=dev)
        xt, pt = g.pointer_table(x), g.pointer_table(packed)
        if a.case == "thc_range":
            fn = lambda: g.gar_thc_range(xt, mM)  # noqa: E731
            nbytes = P * N * 4
        elif a.case == "thc_encode":
            fn = lambda: g.gar_thc_encode(x[0], mM, b, 5, 0, packed[0])  # noqa: E731
            nbytes = N * 4 + words * 4
        elif a.case == "thc_aggregate":
            fn = lambda: g.gar_thc_aggregate(pt, N, b, sums)  # noqa: E731
            nbytes = P * words * 4 + 2 * N
        elif a.case == "thc_decode":
            fn = lambda: g.gar_thc_decode(sums, mM, b, P, avg)  # noqa: E731
            nbytes = 2 * N + 4 * N
        elif a.case == "thc_fused":
            fn = lambda: g.gar_thc_allreduce_fused(xt, b, 5, mM, avg)  # noqa: E731
            nbytes = P * N * 4 + N * 4
        elif a.case == "thc_fused_packed":
            fn = lambda: g.gar_thc_allreduce_fused(xt, b, 5, mM, avg, pt)  # noqa: E731
            nbytes = P * N * 4 + N * 4 + P * words * 4
        elif a.case in ("nuhc_fused", "nuhc_fused_packed"):
            # granularity 36 for b = 4, 2(2^b - 1) + 1 otherwise; a table denser near the middle
            L = (1 << b) - 1
            gr = a.g if a.g else (36 if b == 4 else 2 * L + 1)
            zz = np.arange(L + 1) / L * 2 - 1
            tab = np.rint(gr / 2 + gr / 2 * np.sign(zz) * np.abs(zz) ** 1.6).astype(np.int64)
            tab[0], tab[-1] = 0, gr
            for i in range(1, L):
                tab[i] = max(tab[i], tab[i - 1] + 1)
            for i in range(L - 1, -1, -1):
                tab[i] = min(tab[i], tab[i + 1] - 1)
            pk = pt if a.case == "nuhc_fused_packed" else None
            fn = lambda: g.gar_nuhc_allreduce_fused(xt, b, gr, tab, 5, mM, avg, pk)  # noqa: E731
            nbytes = P * N * 4 + N * 4 + (P * words * 4 if pk is not None else 0)
        else:
            ws = torch.empty(g.gar_nmse_workspace_bytes(N) // 8, dtype=torch.float64, device=dev)
            out = torch.empty(1, dtype=torch.float64, device=dev)
            fn = lambda: g.gar_nmse(x[0], x[1], out, ws)  # noqa: E731
            nbytes = 2 * N * 4
    elif a.case in ("rht", "rht_inv", "rht_inplace", "rht_norm", "ef_apply"):
        # algorithmic bytes: one read and one write of the vector (rht), P reads (norm), 2 reads + 1 write (ef)
        x = bufs(N, max(P, 2), torch.float32)
        y = torch.empty(N, device=dev)
        if a.case == "rht_norm":
            ws = torch.empty(g.gar_rht_norm_range_workspace_bytes(P, N) // 8, dtype=torch.float64, device=dev)
            mM = torch.empty(2, device=dev)
            xt = g.pointer_table(x[:P])
            fn = lambda: g.gar_rht_norm_range(xt, 2.15, mM, ws)  # noqa: E731
            nbytes = P * N * 4
        elif a.case == "ef_apply":
            fn = lambda: g.gar_ef_apply(x[0], x[1], y)  # noqa: E731
            nbytes = 3 * N * 4
        else:
            src, dst = (y, y) if a.case == "rht_inplace" else (x[0], y)
            inv = a.case == "rht_inv"
            fn = lambda: g.gar_rht(src, dst, 7, inverse=inv)  # noqa: E731
            nbytes = 2 * N * 4
    elif a.case in ("train_step", "train_step_fused"):
        # one step of THC's training process for P workers of N values (the
        # page's section 5): error feedback, rotation, norm-based range,
        # non-uniform THC b-bit with granularity g (36 for b = 4), inverse
        # rotation of the average, every worker's error-feedback update from
        # its own wire vector -- through the separate calls, or the fused ones.
        # algorithmic bytes: per worker grad and e read, y written, y read, the
        # wire vector written and read, grad and e read and e written again;
        # once the average written, read and its rotation written
        L = (1 << b) - 1
        gr = a.g if a.g else (36 if b == 4 else 2 * L + 1)
        tab = np.rint(np.linspace(0, gr, L + 1)).astype(np.uint16)
        grads = bufs(N, P, torch.float32)
        errs = [t.mul_(1e-3) for t in bufs(N, P, torch.float32, seed=500)]
        e_work = [t.clone() for t in errs]
        ys = [torch.empty(N, device=dev) for _ in range(P)]
        words = g.gar_thc_words(N, b)
        packed = [torch.empty(words, dtype=torch.int32, device=dev) for _ in range(P)]
        pt, yt = g.pointer_table(packed), g.pointer_table(ys)
        mM = torch.empty(2, device=dev)
        avg, est, tmp = (torch.empty(N, device=dev) for _ in range(3))
        t_p = 2.15
        if a.case == "train_step_fused":
            from .training import TrainingStep

            step = TrainingStep(grads, e_work, b=b, table=tab, t_p=t_p, rht_seed=11, streams=a.streams)
            fn = lambda: step.run(5)  # noqa: E731
        else:
            xs = [torch.empty(N, device=dev) for _ in range(P)]
            xt = g.pointer_table(xs)
            ws = torch.empty(g.gar_rht_norm_range_workspace_bytes(P, N) // 8 + 1, dtype=torch.float64, device=dev)
            own = torch.empty(N, dtype=torch.int16, device=dev)
            y_hat, x_hat = torch.empty(N, device=dev), torch.empty(N, device=dev)

            def fn():
                for w in range(P):
                    g.gar_ef_apply(grads[w], e_work[w], xs[w])
                g.gar_rht_norm_range(xt, t_p, mM, ws)
                for w in range(P):
                    g.gar_rht(xs[w], ys[w], 11)
                g.gar_nuhc_allreduce_fused(yt, b, gr, tab, 5, mM, avg, pt)
                g.gar_rht(avg, est, 11, inverse=True)
                for w in range(P):
                    g.gar_nuhc_aggregate([packed[w]], N, b, tab, own)
                    g.gar_nuhc_decode(own, mM, gr, 1, y_hat)
                    g.gar_rht(y_hat, x_hat, 11, inverse=True)
                    g.gar_ef_update(e_work[w], xs[w], x_hat)
        nbytes = P * N * 4 * (2 + 1 + 1 + 2 + 1) + P * 2 * words * 4 + 3 * N * 4
    elif a.case == "checksum":
        # algorithmic bytes: one read of N 32-bit words
        w = bufs(N, 1, torch.float32)[0].view(torch.int32)
        out = torch.empty(1, dtype=torch.int64, device=dev)
        fn = lambda: g.gar_checksum(w, out)  # noqa: E731
        nbytes = N * 4
    else:
        raise SystemExit(f"unknown case {a.case}")

    for _ in range(a.warmup):
        fn()
    torch.cuda.synchronize()
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev) if a.flush else None
    clean = torch.ones((256 << 20) // 4, dtype=torch.float32, device=dev) if a.flush else None
    launches0 = g.gar_launch_count()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(a.iters):
        if flush is not None:
            # 256 MB written (nothing of the inputs left in L2), then 256 MB read:
            # the dirty lines are written back before the timed call, which
            # starts with an L2 of clean lines
            flush.zero_()
            clean.sum()
        # hold the stream briefly so that the call is queued before the start
        # event: the events then time the GPU, not the host's enqueue
        torch.cuda._sleep(100_000)
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    launches = (g.gar_launch_count() - launches0) // max(a.iters, 1)
    ms = float(np.median(times))
    print(json.dumps({"case": a.case, "P": P, "N": N, "b": b, "dtype": a.dtype, "ms": round(ms, 4),
                      "ms_min": round(float(np.min(times)), 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                      "bytes": int(nbytes), "launches_per_call": int(launches),
                      "launches_total": int(g.gar_launch_count())}))


if __name__ == "__main__":
    main()
