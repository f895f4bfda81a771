"""ncu table of every kernel of libgar.so: achieved HBM GB/s and DRAM traffic.

    python -m gradient_allreduce_homomorphic_gb300.kernel_table --out DIR [--cases c1,c2,...]

For each microbench case (default: all of them) the case first runs on its
own (it must exit 0; it reports how many launches the library made in all
and how many one timed call makes).  Then two ncu runs, both restricted to
the library's kernels (``-k regex:``) and with ``--clock-control none``:

1. durations: ``--metrics gpu__time_duration.sum`` (one pass per launch,
   nothing saved or restored), skipping to the timed call (``-s``) and
   capturing its launches (``-c``);
2. DRAM traffic: ``dram__bytes_read.sum,dram__bytes_write.sum`` on at most
   the first three launches of the timed call (``-s``, ``-c`` <= 3), inputs
   of a few GB at most.  Where the call makes more than three launches the
   traffic column covers only those and is left out of the ratio.

The timed call's summed ncu duration gives its algorithmic GB/s (the case's
algorithmic bytes over that time).  ncu runs every launch alone with cold
caches, so the durations are serialised, cold-cache figures.  The peak is
the measured copy rate (MEASURED_PEAKS.json), not a bound: a kernel that
leaves part of its writes in L2 reads a little above 1.0.  Writes
DIR/<case>_time.csv and DIR/<case>_dram.csv (ncu's rows) and prints one
markdown table.
"""
from __future__ import annotations

import argparse
import csv
import json
import os
import re
import subprocess
import sys

CASES = [
    ("ring", []), ("ring", ["--dtype", "bf16", "--P", "16", "--N", "67108864"]), ("ring_out", []),
    ("bidir", []), ("dbtree", []), ("dbtree", ["--dtype", "bf16", "--P", "16", "--N", "67108864"]),
    ("fused", []), ("fused_range", []), ("pack", []), ("unpack", []), ("pack_all", []), ("pack_all_range", []),
    ("thc_range", []), ("thc_encode", []), ("thc_aggregate", []), ("thc_decode", []), ("thc_fused", []),
    ("thc_fused_packed", []), ("thc_plan", []), ("thc_plan_nmse", []), ("nuhc_fused", []),
    ("nuhc_fused_packed", []), ("nmse", []), ("rht", []), ("rht_inv", []), ("rht_norm", []), ("ef_apply", []),
    ("checksum", ["--N", "268435456"]),
    ("stream_ring", ["--P", "4", "--N", "1048576", "--k", "64"]),
    ("stream_thc", ["--P", "4", "--N", "1048576", "--k", "64"]),
    ("train_step", []), ("train_step_fused", []),
]
LIB_KERNEL = re.compile(r"(ring_fold|ring_step|ring_divide|copy_jobs|pack_all|pack_range_init|range_reset|thc_|"
                        r"nuhc_|nmse_|rht_|ef_kernel|dbtree_|checksum_)")
TIME_METRICS = "gpu__time_duration.sum"
DRAM_METRICS = "dram__bytes_read.sum,dram__bytes_write.sum"
KERNEL_FILTER = "regex:" + LIB_KERNEL.pattern
MAX_DRAM_LAUNCHES = 3
UNIT = {"ns": 1e-3, "us": 1.0, "usecond": 1.0, "nsecond": 1e-3, "ms": 1e3, "msecond": 1e3,
        "byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}


def _launches(path):
    """[(kernel name, {metric: value in us or bytes})] in launch order."""
    rows = list(csv.reader(open(path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, ii, mi, ui, vi = (h.index(k) for k in ("Kernel Name", "ID", "Metric Name", "Metric Unit", "Metric Value"))
    out = {}
    for r in rows[hi + 1:]:
        if len(r) <= vi:
            continue
        d = out.setdefault(int(r[ii]), [r[ki], {}])[1]
        d[r[mi]] = float(r[vi].replace(",", "")) * UNIT.get(r[ui], 1.0)
    return [tuple(out[k]) for k in sorted(out)]


def _base(name):
    """The kernel's own identifier (the first one followed by its template
    arguments or its parameter list)."""
    m = re.search(r"([A-Za-z_]\w*)[<(]", name)
    return m.group(1) if m else name


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", required=True)
    ap.add_argument("--cases", default="")
    ap.add_argument("--peak", type=float, default=0.0, help="GB/s for the fraction (default: MEASURED_PEAKS.json)")
    a = ap.parse_args(argv)
    os.makedirs(a.out, exist_ok=True)
    peak = a.peak
    if not peak:
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        try:
            peak = float(json.load(open(os.path.join(root, "MEASURED_PEAKS.json")))["hbm_gbs"])
        except (OSError, KeyError, ValueError):
            peak = 6800.0
    want = set(a.cases.split(",")) if a.cases else None
    rows = []
    for case, extra in CASES:
        if want and case not in want:
            continue
        cmd = [sys.executable, "-m", "gradient_allreduce_homomorphic_gb300.microbench", case, "--iters", "1",
               "--warmup", "1", *extra]
        tag = case + ("_" + "_".join(x.strip("-") for x in extra) if extra else "")
        plain = subprocess.run(cmd, capture_output=True, text=True)
        if plain.returncode != 0:
            rows.append((tag, "plain run failed", plain.stderr.strip().splitlines()[-1:]))
            continue
        info = json.loads(plain.stdout.strip().splitlines()[-1])
        per_call, total = info["launches_per_call"], info["launches_total"]
        if per_call < 1:
            rows.append((tag, "no library launch in the timed call", []))
            continue
        skip = total - per_call  # the timed call's launches are the library's last ones

        def ncu(metrics, count, suffix):
            log = os.path.join(a.out, f"{tag}_{suffix}.csv")
            r = subprocess.run(["ncu", "--metrics", metrics, "--clock-control", "none", "-k", KERNEL_FILTER,
                                "-s", str(skip), "-c", str(count), "--csv", "--log-file", log, *cmd],
                               capture_output=True, text=True)
            return (_launches(log), None) if r.returncode == 0 else (None, r.stderr.strip().splitlines()[-1:])

        timed, err = ncu(TIME_METRICS, per_call, "time")
        if err is not None:
            rows.append((tag, "ncu run failed", err))
            continue
        n_dram = min(per_call, MAX_DRAM_LAUNCHES)
        dram_l, err = ncu(DRAM_METRICS, n_dram, "dram")
        dram = (sum(m.get("dram__bytes_read.sum", 0.0) + m.get("dram__bytes_write.sum", 0.0) for _, m in dram_l)
                if dram_l else float("nan"))
        whole = dram_l is not None and n_dram == per_call
        us = sum(m.get("gpu__time_duration.sum", 0.0) for _, m in timed)
        names = sorted({_base(n) for n, _ in timed})
        gbs = info["bytes"] / (us * 1e-6) / 1e9 if us else 0.0
        rows.append((tag, ", ".join(names), len(timed), us, info["bytes"], gbs, gbs / peak, dram,
                     dram / info["bytes"] if whole and info["bytes"] else float("nan"), info["ms"] * 1e3,
                     "" if whole else f" (first {n_dram} launches)"))
    print(f"| case | kernels | launches | ncu time (us) | algorithmic bytes | GB/s (ncu) | of peak "
          f"| DRAM bytes | DRAM / algorithmic | events (us) |")
    print("|---|---|---:|---:|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        if len(r) == 3:
            print(f"| {r[0]} | {r[1]}: {r[2]} | | | | | | | | |")
        else:
            print(f"| {r[0]} | {r[1]} | {r[2]} | {r[3]:.1f} | {r[4]:,} | {r[5]:.0f} | {r[6]:.3f} | {r[7]:,.0f}{r[10]} "
                  f"| {r[8]:.3f} | {r[9]:.1f} |")


if __name__ == "__main__":
    main()
