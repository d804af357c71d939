"""DRAM bytes of a fused step and of the same chain unfused, measured, from an
ncu launch list of `bench.py --profile-steps`.

The CODA article (d9bl.com, §4.3) credits part of the fused kernels' gain to
the memory traffic they save; this module turns a measurement of that traffic
into per-step totals.  The profile run executes, after its warm-up, one fused
step and then one unfused step, each preceded by a full L2 flush (a 256 MiB
fill, then a 256 MiB read) and followed by a read-only pass over 256 MiB.
Captured with

    ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \\
        --clock-control none --cache-control none --csv --log-file traffic.csv \\
        python bench.py --workload W --profile-steps --warmup 3

every launch is one pass with no cache flush by ncu, so the library kernels of
a step read and write exactly what they would in the benchmark.  Outputs still
dirty in L2 when a step's last kernel ends are written back during the
read-only pass that follows it: that pass writes nothing of its own, so its
DRAM writes are the step's remaining writes.  A step's DRAM bytes are then its
kernels' reads and writes plus that pass's writes.

    python -m gemm_epilogue_transformer_tmem_gb300.traffic W traffic.csv \\
        [--json profiles/traffic.json] [--md profiles/dram_traffic_W.md] [--command "..."]

With --launches the CSV is a plain launch list (gpu__time_duration.sum of every
launch of a bench run) and the output is each kernel's launches, total time and
share of the total.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
KERNEL_SOURCES = ["coda_gemm_kernel.cuh", "coda_ops.cuh", "coda_ptx.cuh", "coda_internal.h", "coda_sequences.h",
                  "coda_api.cu"]
# which GEMM launch of a fused step is the dominant one (most flops); the
# others have one GEMM
DOMINANT_GEMM = {"llama": 2}

_SCALE = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
          "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3, "second": 1e6,
          "ns": 1e-3, "us": 1.0, "ms": 1e3, "s": 1e6}


def kernel_hash() -> str:
    """Hash of the kernel and planner sources with comments and whitespace
    removed: a committed traffic figure stays valid while only the prose around
    the code changes, and is void once the code changes."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(HERE, "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def read_launches(text: str) -> list[dict]:
    """Launches in capture order: name, DRAM bytes read and written, duration (us)."""
    lines = text.splitlines()
    start = next((i for i, ln in enumerate(lines) if ln.startswith('"ID"')), None)
    if start is None:
        raise ValueError("no ncu CSV header in the log")
    rows = csv.DictReader(io.StringIO("\n".join(lines[start:])))
    by_id: dict[int, dict] = {}
    for r in rows:
        try:
            i = int(r["ID"])
        except (KeyError, ValueError):
            continue
        d = by_id.setdefault(i, {"id": i, "name": r["Kernel Name"], "read": 0.0, "write": 0.0, "us": 0.0})
        val = float(str(r["Metric Value"]).replace(",", ""))
        unit = r.get("Metric Unit", "")
        v = val * _SCALE.get(unit, 1.0)
        m = r["Metric Name"]
        if m == "dram__bytes_read.sum":
            d["read"] = v
        elif m == "dram__bytes_write.sum":
            d["write"] = v
        elif m == "gpu__time_duration.sum":
            d["us"] = v
    return [by_id[i] for i in sorted(by_id)]


def is_library(name: str) -> bool:
    """Kernels of this library (the rest are the flush passes of the harness)."""
    return not any(s in name for s in ("at::native", "vectorized_elementwise", "reduce_kernel", "elementwise_kernel",
                                       "FillFunctor"))


def split_steps(launches: list[dict]):
    """(fused kernels, fused write-back pass, unfused kernels, unfused write-back
    pass): the last two runs of library kernels and the pass after each."""
    segs = []
    i = 0
    n = len(launches)
    while i < n:
        if is_library(launches[i]["name"]):
            j = i
            while j < n and is_library(launches[j]["name"]):
                j += 1
            wb = launches[j] if j < n else None
            segs.append((launches[i:j], wb))
            i = j
        else:
            i += 1
    if len(segs) < 2 or segs[-1][1] is None or segs[-2][1] is None:
        raise ValueError("launch list does not end with a fused and an unfused step, each followed by a pass")
    return segs[-2][0], segs[-2][1], segs[-1][0], segs[-1][1]


def summarize(workload: str, launches: list[dict], command: str = "") -> tuple[dict, str]:
    fused, fwb, unfused, uwb = split_steps(launches)

    def tot(ks, wb):
        r = sum(k["read"] for k in ks)
        w = sum(k["write"] for k in ks) + wb["write"]
        return r, w

    fr, fw = tot(fused, fwb)
    ur, uw = tot(unfused, uwb)
    gemms = [k for k in fused if k["name"].startswith("coda_gemm_epilogue_kernel") or
             "coda_gemm_epilogue_kernel" in k["name"].split("(")[0]]
    dom = gemms[DOMINANT_GEMM.get(workload, 0)] if gemms else None
    entry = {
        "kernel_hash": kernel_hash(),
        "fused_step_bytes": int(round(fr + fw)), "fused_step_read": int(round(fr)),
        "fused_step_write": int(round(fw)), "fused_writeback": int(round(fwb["write"])),
        "unfused_step_bytes": int(round(ur + uw)), "unfused_step_read": int(round(ur)),
        "unfused_step_write": int(round(uw)), "unfused_writeback": int(round(uwb["write"])),
        "dominant_kernel": dom["name"].split("(")[0] if dom else None,
        "dominant_kernel_bytes": int(round(dom["read"] + dom["write"])) if dom else None,
        "source": f"profiles/dram_traffic_{workload}.md",
    }
    out = [f"# DRAM traffic per step: {workload}, fused against unfused (measured)", ""]
    if command:
        out += ["Command (one GB300; the same command exited 0 without ncu just before):", "", "```", command, "```",
                ""]
    out += [f"Kernel sources hash `{entry['kernel_hash']}`.  Bytes in MB (10^6).  `write-back` is the DRAM writes of "
            "the read-only pass after the step: the step's outputs still dirty in L2 when it ended.", ""]
    for title, ks, wb, r, w in (("fused step", fused, fwb, fr, fw), ("unfused step", unfused, uwb, ur, uw)):
        out += [f"## {title}", "", "| kernel | DRAM read MB | DRAM write MB | us (ncu) |", "|---|---|---|---|"]
        for k in ks:
            nm = k["name"].split("(")[0]
            nm = nm if len(nm) < 90 else nm[:87] + "..."
            out.append(f"| `{nm}` | {k['read'] / 1e6:.1f} | {k['write'] / 1e6:.1f} | {k['us']:.1f} |")
        out.append(f"| write-back (after the step) | - | {wb['write'] / 1e6:.1f} | - |")
        out.append(f"| **total** | **{r / 1e6:.1f}** | **{w / 1e6:.1f}** | "
                   f"{sum(k['us'] for k in ks):.1f} |")
        out.append("")
    out.append(f"Fused step {entry['fused_step_bytes'] / 1e6:.1f} MB against unfused "
               f"{entry['unfused_step_bytes'] / 1e6:.1f} MB "
               f"({entry['unfused_step_bytes'] / max(entry['fused_step_bytes'], 1):.2f}x).")
    return entry, "\n".join(out) + "\n"


def launch_shares(launches: list[dict], command: str = "") -> str:
    """Per kernel (name without its argument list): launches, total time, share."""
    agg: dict[str, list] = {}
    for k in launches:
        nm = k["name"].split("(")[0]
        a = agg.setdefault(nm, [0, 0.0])
        a[0] += 1
        a[1] += k["us"]
    total = sum(v[1] for v in agg.values()) or 1.0
    out = ["# Launch list (ncu gpu__time_duration.sum; cold-cache, serialised: compare shares)", ""]
    if command:
        out += ["Command (one GB300; the same command exited 0 without ncu just before):", "", "```", command, "```", ""]
    out += ["| kernel | launches | total us | share |", "|---|---|---|---|"]
    for nm, (n, us) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        short = nm if len(nm) < 100 else nm[:97] + "..."
        out.append(f"| `{short}` | {n} | {us:.1f} | {100.0 * us / total:.1f}% |")
    out.append(f"| **all** | {sum(v[0] for v in agg.values())} | {total:.1f} | 100% |")
    return "\n".join(out) + "\n"


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("csv")
    ap.add_argument("--json", help="traffic.json to update with this workload's entry")
    ap.add_argument("--md", help="markdown summary to write")
    ap.add_argument("--command", default="", help="the ncu command line, recorded in the summary")
    ap.add_argument("--launches", action="store_true", help="summarise a plain launch list instead")
    a = ap.parse_args(argv)
    with open(a.csv, encoding="utf-8", errors="replace") as f:
        launches = read_launches(f.read())
    if a.launches:
        md = launch_shares(launches, a.command)
        if a.md:
            with open(a.md, "w") as f:
                f.write(md)
        else:
            sys.stdout.write(md)
        return 0
    entry, md = summarize(a.workload, launches, a.command)
    if a.json:
        d = {}
        if os.path.exists(a.json):
            with open(a.json) as f:
                d = json.load(f)
        d[a.workload] = entry
        with open(a.json, "w") as f:
            json.dump(d, f, indent=1)
            f.write("\n")
    if a.md:
        with open(a.md, "w") as f:
            f.write(md)
    else:
        sys.stdout.write(md)
    print(json.dumps(entry))
    return 0


if __name__ == "__main__":
    sys.exit(main())
