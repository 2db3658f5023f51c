"""Summary of an Nsight Compute capture: one Markdown table per captured launch
with the counters the kernels' roofline readings use (duration, DRAM bytes and
throughput, the tensor / FMA / ALU / XU pipes, issue, warps, L2 hit rate,
registers, launch shape) and the top issue-stall reasons.

  python -m roofline_benchmarking_gb300.ncu_summary REPORT.ncu-rep [--stalls N]
  python -m roofline_benchmarking_gb300.ncu_summary RAW.csv

A ``.ncu-rep`` is read through ``ncu -i REPORT --page raw --csv`` (counters
only); a ``.csv`` is that export already made. Sources (web pages): the
GPU-Roofline page ("Python Hierarchical Roofline Module": DRAM bytes and
duration from ncu counters) and the kbench page ("Implementation details": Nsight
Compute on each kernel).
"""
from __future__ import annotations

import argparse
import csv
import io
import shutil
import subprocess
import sys

# (label, metric, scale, format): value shown = float(metric) * scale
METRICS = [
    ("gpu__time_duration (cold L2, serialised)", "gpu__time_duration.sum", None, "{:.1f} us"),
    ("dram__bytes_read.sum", "dram__bytes_read.sum", None, "{:.1f} MB"),
    ("dram__bytes_write.sum", "dram__bytes_write.sum", None, "{:.1f} MB"),
    ("sm__pipe_tensor_cycles_active (% of peak, active)",
     "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", 1.0, "{:.2f} %"),
    ("sm__pipe_fma_cycles_active (% of peak, active)",
     "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active", 1.0, "{:.2f} %"),
    ("sm__pipe_alu_cycles_active (% of peak, active)",
     "sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active", 1.0, "{:.2f} %"),
    ("sm__inst_executed_pipe_xu (% of peak, active)",
     "sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active", 1.0, "{:.2f} %"),
    ("smsp__issue_active (% of peak, active)", "smsp__issue_active.avg.pct_of_peak_sustained_active", 1.0,
     "{:.2f} %"),
    ("sm__warps_active (% of peak, active)", "sm__warps_active.avg.pct_of_peak_sustained_active", 1.0, "{:.2f} %"),
    ("lts__t_sector_hit_rate", "lts__t_sector_hit_rate.pct", 1.0, "{:.2f} %"),
    ("gpu__dram_throughput (% of peak, elapsed)", "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", 1.0,
     "{:.2f} %"),
    ("SM clock", "sm__cycles_elapsed.avg.per_second", None, "{:.2f} GHz"),
    ("smsp__inst_executed.sum", "smsp__inst_executed.sum", 1.0, "{:,.0f} warp instructions"),
    ("launch__registers_per_thread", "launch__registers_per_thread", 1.0, "{:.0f}"),
]
STALL_PREFIX = "smsp__average_warps_issue_stalled_"
STALL_SUFFIX = "_per_issue_active.ratio"

# the units ncu reports for time, bytes and frequency, to the ones shown
_TIME = {"nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0, "us": 1.0, "msecond": 1e3, "ms": 1e3, "second": 1e6, "s": 1e6}
_BYTES = {"byte": 1e-6, "Kbyte": 1e-3, "Mbyte": 1.0, "Gbyte": 1e3, "Tbyte": 1e6,
          "KB": 1e-3, "MB": 1.0, "GB": 1e3}
_FREQ = {"hz": 1e-9, "khz": 1e-6, "mhz": 1e-3, "ghz": 1.0}


def _number(text: str) -> float | None:
    try:
        return float(text.replace(",", ""))
    except (AttributeError, ValueError):
        return None


def _scaled(value: float, unit: str, metric: str) -> float | None:
    if metric == "gpu__time_duration.sum":
        f = _TIME.get(unit)
    elif metric.startswith("dram__bytes"):
        f = _BYTES.get(unit)
    elif metric.endswith("per_second"):
        f = _FREQ.get(unit.lower())
    else:
        f = 1.0
    return None if f is None else value * f


def parse_raw_csv(text: str) -> list[dict]:
    """Rows of ``ncu --page raw --csv``: a header of metric names, a row of units,
    then one row per captured launch. Returns one dict per launch with the kernel
    name, launch shape, the METRICS values in display units (None if absent) and
    the stall ratios by reason."""
    rows = list(csv.reader(io.StringIO(text)))
    # skip anything ncu printed before the header (==PROF== lines and the like)
    start = next((i for i, r in enumerate(rows) if r and r[0] == "ID"), None)
    if start is None or len(rows) < start + 2:
        return []
    hdr, units = rows[start], rows[start + 1]
    col = {h: i for i, h in enumerate(hdr)}
    out = []
    for r in rows[start + 2:]:
        if len(r) != len(hdr):
            continue
        launch = {"kernel": r[col["Kernel Name"]] if "Kernel Name" in col else "",
                  "grid": r[col["Grid Size"]] if "Grid Size" in col else "",
                  "block": r[col["Block Size"]] if "Block Size" in col else "", "values": {}, "stalls": {}}
        for label, metric, _, _ in METRICS:
            v = _number(r[col[metric]]) if metric in col else None
            launch["values"][metric] = None if v is None else _scaled(v, units[col[metric]], metric)
        for h, i in col.items():
            if h.startswith(STALL_PREFIX) and h.endswith(STALL_SUFFIX):
                v = _number(r[i])
                if v is not None:
                    launch["stalls"][h[len(STALL_PREFIX):-len(STALL_SUFFIX)]] = v
        out.append(launch)
    return out


def render(launches: list[dict], stalls: int = 6) -> str:
    md = []
    for n, L in enumerate(launches):
        md.append(f"### launch {n}: `{L['kernel']}`, grid {L['grid']} x block {L['block']}")
        md.append("")
        md.append("| metric | value |")
        md.append("|---|---|")
        v = L["values"]
        for label, metric, _, fmt in METRICS:
            if v.get(metric) is not None:
                md.append(f"| {label} | {fmt.format(v[metric])} |")
        rd, wr = v.get("dram__bytes_read.sum"), v.get("dram__bytes_write.sum")
        if rd is not None and wr is not None:
            md.append(f"| traffic (read + write) | {rd + wr:.1f} MB |")
            t = v.get("gpu__time_duration.sum")
            if t:
                md.append(f"| DRAM bytes / duration | {(rd + wr) * 1e6 / (t * 1e-6) / 1e9:.0f} GB/s |")
        if L["stalls"] and stalls > 0:
            md.append("")
            md.append("| stall reason | cycles per issued instruction |")
            md.append("|---|---|")
            for name, ratio in sorted(L["stalls"].items(), key=lambda x: -x[1])[:stalls]:
                md.append(f"| {name} | {ratio:.2f} |")
        md.append("")
    return "\n".join(md)


def export_csv(report: str) -> str:
    ncu = shutil.which("ncu") or "/usr/local/cuda/bin/ncu"
    r = subprocess.run([ncu, "-i", report, "--page", "raw", "--csv"], capture_output=True, text=True)
    if r.returncode != 0:
        raise SystemExit(f"ncu -i {report} failed: {r.stderr.strip()[-500:]}")
    return r.stdout


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("source", help="an .ncu-rep report or the CSV of `ncu -i REPORT --page raw --csv`")
    p.add_argument("--stalls", type=int, default=6, help="stall reasons listed per launch")
    args = p.parse_args(argv)
    text = open(args.source).read() if args.source.endswith(".csv") else export_csv(args.source)
    launches = parse_raw_csv(text)
    if not launches:
        print("no launch found", file=sys.stderr)
        return 1
    print(render(launches, args.stalls))
    return 0


if __name__ == "__main__":
    sys.exit(main())
