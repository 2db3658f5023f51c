"""Hierarchical instruction roofline of the library's kernels, from ncu counters.

Sources (web pages): the GPU-Roofline-Python page ("Python Hierarchical
Roofline Module"), section "Metrics Used": the number of instructions a kernel
executes, the global and shared transactions at L1, the L2 transactions and
the HBM transactions; instruction intensity = (instructions / 32) /
transactions and performance = (instructions / 32) / (1e9 x run time) in warp
GIPS. The method is Ding and Williams, "An Instruction Roofline Model for
GPUs" (2019), which the page cites: one point per memory level, each against
min(peak warp GIPS, intensity x that level's transaction rate).

Counters (ncu metric names on sm_103):
  instructions  smsp__thread_inst_executed.sum (thread level; / 32 = warp level)
  L1 global     l1tex__t_sectors_pipe_lsu_mem_global_op_{ld,st,atom,red}.sum
  L1 shared     l1tex__data_pipe_lsu_wavefronts_mem_shared_op_{ld,st,atom}.sum
  L2            lts__t_sectors_op_{read,write,atom,red}.sum
  HBM           dram__sectors_{read,write}.sum
A transaction is a 32-byte sector (a wavefront for shared memory). Beyond the
page: the sectors TMA moves from L2 into shared memory
(l1tex__m_xbar2l1tex_read_sectors_mem_global_op_tma_ld.sum) are reported too,
because the tensor-core kernel's loads bypass the LSU path the page's L1
metrics count, and tensor-core operand reads from shared memory appear in no
LSU counter at all.

Ceilings come from ncu's own peak rates (metric.sum.peak_sustained x the
unit's clock, metric.avg.per_second) and, for HBM, also from the measured copy
bandwidth / 32 bytes. Run times come from CUDA events outside the profiler
(``run --time``); a label that launches several kernels (the naive variant)
splits its event time by the kernels' shares of ncu's gpu__time_duration.

  python -m roofline_benchmarking_gb300.iroofline metrics        # the --metrics list
  python -m roofline_benchmarking_gb300.iroofline run            # one launch of each kernel (run under ncu)
  python -m roofline_benchmarking_gb300.iroofline run --time T.json   # CUDA-event times, no profiler
  python -m roofline_benchmarking_gb300.iroofline report --counters C.csv --times T.json [--out DIR]
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import re
import statistics
import sys

from .roofline import instruction_intensity, warp_gips

LEVELS = {
    "L1 global": ["l1tex__t_sectors_pipe_lsu_mem_global_op_ld.sum", "l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum",
                  "l1tex__t_sectors_pipe_lsu_mem_global_op_atom.sum",
                  "l1tex__t_sectors_pipe_lsu_mem_global_op_red.sum"],
    "L1 shared": ["l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld.sum",
                  "l1tex__data_pipe_lsu_wavefronts_mem_shared_op_st.sum",
                  "l1tex__data_pipe_lsu_wavefronts_mem_shared_op_atom.sum"],
    "L2": ["lts__t_sectors_op_read.sum", "lts__t_sectors_op_write.sum", "lts__t_sectors_op_atom.sum",
           "lts__t_sectors_op_red.sum"],
    "HBM": ["dram__sectors_read.sum", "dram__sectors_write.sum"],
    "TMA L2->smem": ["l1tex__m_xbar2l1tex_read_sectors_mem_global_op_tma_ld.sum"],
}
INSTRUCTIONS = "smsp__thread_inst_executed.sum"
WARP_INSTRUCTIONS = "smsp__inst_executed.sum"
DURATION = "gpu__time_duration.sum"

# Peak rates per level: (sectors-per-cycle metric, cycles-per-second metric).
CEILINGS = {
    "inst": ("smsp__inst_executed.sum.peak_sustained", "sm__cycles_elapsed.avg.per_second"),
    "L1 global": ("l1tex__t_sectors.sum.peak_sustained", "l1tex__cycles_elapsed.avg.per_second"),
    "L1 shared": ("l1tex__data_pipe_lsu_wavefronts.sum.peak_sustained", "l1tex__cycles_elapsed.avg.per_second"),
    "L2": ("lts__t_sectors.sum.peak_sustained", "lts__cycles_elapsed.avg.per_second"),
    "HBM": ("dram__sectors.sum.peak_sustained", "dram__cycles_elapsed.avg.per_second"),
    "TMA L2->smem": ("lts__t_sectors.sum.peak_sustained", "lts__cycles_elapsed.avg.per_second"),
}
SECTOR_BYTES = 32


def metric_names() -> list[str]:
    names = [INSTRUCTIONS, WARP_INSTRUCTIONS, DURATION]
    for ms in LEVELS.values():
        names += ms
    for a, b in CEILINGS.values():
        names += [a, b]
    out = []
    for n in names:
        if n not in out:
            out.append(n)
    return out


# --------------------------------------------------------------------------
# parsing ncu's CSV (``ncu --csv --metrics ... --log-file F``: one row per
# launch and metric)
# --------------------------------------------------------------------------
_TIME_UNITS = {"nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0, "ns": 1e-9, "us": 1e-6,
               "ms": 1e-3, "s": 1.0}
_RATE_UNITS = {"cycle/second": 1.0, "cycle/nsecond": 1e9, "cycle/usecond": 1e6, "cycle/msecond": 1e3,
               "Hz": 1.0, "Khz": 1e3, "KHz": 1e3, "kHz": 1e3, "Mhz": 1e6, "MHz": 1e6, "Ghz": 1e9, "GHz": 1e9}


def short_kernel_name(name: str) -> str:
    """'void ns::(anonymous namespace)::k<128>(const float *, int)' -> 'k<128>'."""
    s = name.strip()
    if s.startswith("void "):
        s = s[5:]
    for anon in ("(anonymous namespace)::", "<unnamed>::", "unnamed>::"):
        s = s.replace(anon, "")
    depth, cut = 0, len(s)
    for i, ch in enumerate(s):  # drop the argument list (the first '(' outside template brackets)
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif ch == "(" and depth == 0 and i > 0:
            cut = i
            break
    s = s[:cut]
    depth, start = 0, 0
    for i, ch in enumerate(s):  # drop namespaces (the last '::' outside template brackets)
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif ch == ":" and depth == 0 and i + 1 < len(s) and s[i + 1] == ":":
            start = i + 2
    return s[start:]


def _value(raw: str, unit: str, metric: str) -> float:
    v = float(raw.replace(",", ""))
    if metric == DURATION:
        return v * _TIME_UNITS.get(unit, 1e-9)
    if metric.endswith(".per_second"):
        return v * _RATE_UNITS.get(unit, 1.0)
    return v


def parse_ncu_csv(text: str) -> list[dict]:
    """Launches in order: [{'id', 'kernel', 'name', 'metrics': {metric: value}}].
    Time is in seconds and clock rates in cycles per second."""
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    if not lines:
        return []
    rows = list(csv.reader(io.StringIO("\n".join(lines))))
    hdr = rows[0]
    col = {h: i for i, h in enumerate(hdr)}
    for need in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value"):
        if need not in col:
            raise ValueError(f"not an ncu --csv metrics log: column {need!r} missing")
    launches: dict[int, dict] = {}
    for r in rows[1:]:
        if len(r) != len(hdr) or r[col["ID"]] == "ID":
            continue
        lid = int(r[col["ID"]])
        ent = launches.setdefault(lid, {"id": lid, "name": r[col["Kernel Name"]],
                                        "kernel": short_kernel_name(r[col["Kernel Name"]]), "metrics": {}})
        m = r[col["Metric Name"]]
        try:
            ent["metrics"][m] = _value(r[col["Metric Value"]], r[col["Metric Unit"]], m)
        except ValueError:
            continue
    return [launches[k] for k in sorted(launches)]


def aggregate(launches: list[dict]) -> dict[str, dict]:
    """Per kernel: launch count and the mean per launch of every metric."""
    out: dict[str, dict] = {}
    for ln in launches:
        e = out.setdefault(ln["kernel"], {"launches": 0, "sums": {}})
        e["launches"] += 1
        for k, v in ln["metrics"].items():
            e["sums"][k] = e["sums"].get(k, 0.0) + v
    for e in out.values():
        e["mean"] = {k: v / e["launches"] for k, v in e["sums"].items()}
    return out


# --------------------------------------------------------------------------
# the roofline points
# --------------------------------------------------------------------------
def level_transactions(mean: dict) -> dict[str, float]:
    return {lvl: sum(mean.get(m, 0.0) for m in ms) for lvl, ms in LEVELS.items()}


def ceilings(mean: dict, hbm_gbs: float | None = None) -> dict[str, float]:
    """Peak warp GIPS ('inst') and each level's peak transactions per second
    (GTXN/s), from ncu's peak rates; 'HBM measured' from a measured copy
    bandwidth in GB/s."""
    out = {}
    for key, (rate, clock) in CEILINGS.items():
        if rate in mean and clock in mean:
            out[key] = mean[rate] * mean[clock] / 1e9
    if hbm_gbs:
        out["HBM measured"] = hbm_gbs / SECTOR_BYTES
    return out


def roofline_points(mean: dict, seconds: float, ceil: dict) -> dict:
    """Intensity, attainable GIPS and the binding level for one kernel."""
    inst = mean.get(INSTRUCTIONS, 0.0)
    gips = warp_gips(inst, seconds)
    peak = ceil.get("inst")
    levels = {}
    for lvl, txn in level_transactions(mean).items():
        if txn <= 0:
            continue
        ii = instruction_intensity(inst, txn)
        bw = ceil.get("HBM measured" if lvl == "HBM" and "HBM measured" in ceil else lvl)
        att = None
        if peak is not None and bw is not None:
            att = min(peak, ii * bw)
        levels[lvl] = {"transactions": txn, "intensity": ii, "ceiling_gtxn_s": bw, "attainable_gips": att,
                       "achieved_gtxn_s": txn / seconds / 1e9}
    bound, att = None, None
    bounded = {k: v for k, v in levels.items() if v["attainable_gips"] is not None and k != "TMA L2->smem"}
    if bounded:
        bound = min(bounded, key=lambda k: bounded[k]["attainable_gips"])
        att = bounded[bound]["attainable_gips"]
        if peak is not None and att >= peak:
            bound = "instruction issue"  # every level's memory ceiling lies above the peak
    return {"warp_instructions": inst / 32.0, "warp_gips": gips, "peak_warp_gips": peak, "levels": levels,
            "bound": bound, "attainable_gips": att, "frac": (gips / att) if att else None}


# --------------------------------------------------------------------------
# the kernels: one launch each (under ncu), or CUDA-event times (without)
# --------------------------------------------------------------------------
def _plan():
    """(label, kernel-name regex, callable factory). Factories build inputs on
    the device and return (launch, bench) closures."""
    import torch

    from . import inputs, kbattn
    V = kbattn.Variant

    def attn(w, variant):
        def make():
            q, k, v = (t.cuda() for t in inputs.make_qkv(w))
            o = torch.empty_like(q)
            ws = None
            if variant == V.NAIVE:
                n = kbattn.kb_attn_workspace_bytes(w.B, w.H, w.S, w.d, kbattn.DType.F32, variant)
                ws = torch.empty(n, dtype=torch.uint8, device="cuda")

            def launch():
                if ws is None:
                    kbattn.kb_attn_fwd(q, k, v, o, causal=w.causal, scale=w.scale, variant=variant)
                else:
                    kbattn.kb_attn_fwd_ws(q, k, v, o, ws, causal=w.causal, scale=w.scale, variant=variant)

            def bench(iters):
                return kbattn.kb_attn_bench(q, k, v, o, w.causal, w.scale, variant, warmup=5, iters=iters,
                                            workspace=ws)
            return launch, bench
        return make

    def hbm(op):
        def make():
            n = inputs.TRIAD_N // 8  # 256 MiB arrays: larger than L2, a few hundred MB on the device
            a = torch.empty(n, dtype=torch.float32, device="cuda")
            b = torch.ones(n, dtype=torch.float32, device="cuda")
            c = torch.full((n,), 2.0, dtype=torch.float32, device="cuda")
            out = torch.zeros(1, dtype=torch.float32, device="cuda")

            def launch():
                kbattn.kb_hbm_bench(op, a, b, c, 3.0, out, block=256, warmup=0, iters=1)

            def bench(iters):
                return kbattn.kb_hbm_bench(op, a, b, c, 3.0, out, block=256, warmup=5, iters=iters)
            return launch, bench
        return make

    H = kbattn.HbmOp
    return [
        ("tc " + inputs.BF16_CAUSAL_S4096.name, r"attn_tc_kernel<128", attn(inputs.BF16_CAUSAL_S4096, V.TC)),
        ("tc " + inputs.BF16_S2048_D64.name, r"attn_tc64_kernel", attn(inputs.BF16_S2048_D64, V.TC)),
        ("tc " + inputs.BF16_CAUSAL_D256.name, r"attn_tc256_kernel", attn(inputs.BF16_CAUSAL_D256, V.TC)),
        ("naive " + inputs.F32_S1024.name, r"naive_", attn(inputs.F32_S1024, V.NAIVE)),
        ("fused " + inputs.F32_S1024.name, r"fused_row", attn(inputs.F32_S1024, V.FUSED)),
        ("flash " + inputs.F32_S1024.name, r"flash_f32", attn(inputs.F32_S1024, V.FLASH)),
        ("fixedpoint " + inputs.Q15_S1024.name, r"q15_attn", attn(inputs.Q15_S1024, V.FIXEDPOINT)),
        ("triad 256 MiB", r"TriadOp", hbm(H.TRIAD)),
        ("copy 256 MiB", r"CopyOp", hbm(H.COPY)),
        ("write 256 MiB", r"FillOp", hbm(H.WRITE)),
        ("read 256 MiB", r"read_kernel", hbm(H.READ)),
    ]


def run(times_out: str | None, seconds: float = 0.2) -> int:
    import torch

    from . import build, kbattn
    if not torch.cuda.is_available():
        print("needs a CUDA GPU", file=sys.stderr)
        return 2
    build.build()
    kbattn.load()
    times = {}
    for label, pattern, make in _plan():
        launch, bench = make()
        if times_out is None:
            launch()
            torch.cuda.synchronize()
        else:
            probe = statistics.median(bench(3))
            iters = max(5, min(2000, int(seconds / max(probe * 1e-3, 1e-6))))
            ms = bench(iters)
            times[label] = {"pattern": pattern, "ms": statistics.median(ms), "iters": iters}
        if kbattn.kb_check_device_error() != kbattn.Status.OK:
            raise RuntimeError(f"device error in {label}")
        torch.cuda.empty_cache()
    if times_out is not None:
        with open(times_out, "w") as f:
            json.dump(times, f, indent=1)
    return 0


def report(counters_path: str, times_path: str, out_dir: str | None, hbm_gbs: float | None) -> list[dict]:
    launches = parse_ncu_csv(open(counters_path).read())
    kernels = aggregate(launches)
    times = json.load(open(times_path))
    rows = []
    for label, t in times.items():
        pat = re.compile(t["pattern"])
        mine = {k: v for k, v in kernels.items() if pat.search(k)}
        if not mine:
            continue
        total = sum(v["mean"].get(DURATION, 0.0) * v["launches"] for v in mine.values())
        for kname, v in mine.items():
            share = (v["mean"].get(DURATION, 0.0) * v["launches"] / total) if total > 0 else 1.0 / len(mine)
            # one call of the label launches each of its kernels once
            sec = t["ms"] * 1e-3 * share
            ceil = ceilings(v["mean"], hbm_gbs)
            pts = roofline_points(v["mean"], sec, ceil)
            rows.append({"label": label, "kernel": kname, "seconds": sec, "time_share": share, **pts,
                         "ceilings": ceil})
    if out_dir:
        os.makedirs(out_dir, exist_ok=True)
        with open(os.path.join(out_dir, "iroofline.json"), "w") as f:
            json.dump(rows, f, indent=1)
        with open(os.path.join(out_dir, "iroofline.md"), "w") as f:
            f.write(markdown(rows) + "\n")
    return rows


def _fmt(x, spec):
    return "-" if x is None else format(x, spec)


def markdown(rows: list[dict]) -> str:
    out = ["| label | kernel | time us | warp inst | warp GIPS | peak GIPS | level | txn | intensity "
           "(warp inst/txn) | achieved GTXN/s | ceiling GTXN/s | attainable GIPS |",
           "|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        first = True
        for lvl, p in r["levels"].items():
            mark = " (bound)" if lvl == r["bound"] else ""
            head = (f"| {r['label']} | {r['kernel']} | {r['seconds'] * 1e6:.1f} | {r['warp_instructions']:.4g} | "
                    f"{r['warp_gips']:.1f} | {_fmt(r['peak_warp_gips'], '.0f')} ") if first else "| | | | | | "
            out.append(head + f"| {lvl}{mark} | {p['transactions']:.4g} | {p['intensity']:.3g} | "
                       f"{p['achieved_gtxn_s']:.1f} | {_fmt(p['ceiling_gtxn_s'], '.1f')} | "
                       f"{_fmt(p['attainable_gips'], '.1f')} |")
            first = False
    return "\n".join(out)


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = p.add_subparsers(dest="cmd", required=True)
    sub.add_parser("metrics", help="print the comma-separated metric list for ncu --metrics")
    r = sub.add_parser("run", help="one launch of each kernel, or CUDA-event times with --time")
    r.add_argument("--time", default=None, help="write median event times (ms) per label to this JSON file")
    r.add_argument("--seconds", type=float, default=0.2)
    rp = sub.add_parser("report")
    rp.add_argument("--counters", required=True)
    rp.add_argument("--times", required=True)
    rp.add_argument("--out", default=None)
    rp.add_argument("--hbm-gbs", type=float, default=None, help="measured copy GB/s (default: measured peaks)")
    a = p.parse_args(argv)
    if a.cmd == "metrics":
        print(",".join(metric_names()))
        return 0
    if a.cmd == "run":
        return run(a.time, a.seconds)
    hbm = a.hbm_gbs
    if hbm is None:
        from . import roofline as rf
        hbm = rf.load_measured_peaks()[0]["hbm_gbs"]
    print(markdown(report(a.counters, a.times, a.out, hbm)))
    return 0


if __name__ == "__main__":
    sys.exit(main())
