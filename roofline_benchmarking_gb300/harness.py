"""Measurement harness: every workload x variant of the attention library and
the four HBM kernels, timed with CUDA events around each launch, placed on the
roofline, with SM clocks sampled during each row. One schema for all rows,
written as CSV, Markdown and JSON lines.

  python -m roofline_benchmarking_gb300.harness [--only SUBSTR] [--out DIR]
                                                [--seconds S] [--quick] [--sweep] [--resume]
                                                [--config NAMES] [--variant NAMES]
                                                [--warmup W] [--iters N] [--size-mb MB]

Every row is appended to ``checkpoint.jsonl`` in the output directory as soon as
it is measured; ``--resume`` reuses the rows found there (a run that was cut off
keeps what it finished) and measures only the missing ones, then writes the
outputs from all of them.

``--sweep`` runs only the kbench page's sequence sweep (section "Running") with
the three fp32 variants, and the same sweep widened to S = 16384 on the
tensor-core path (bf16, d = 64 and 128), and writes their tables (the fp32
variants' speed-up over the naive one per S; the tensor-core kernels' fraction
of the measured bf16 peak per S) to ``sweep.md`` beside the other outputs.

Sources (web pages): the kbench page, "Implementation details" (events around
the kernel only, configurable warm-up, mean / p50 / p99 / min, achieved GFLOP/s
and effective GB/s) and "Analysis" (each kernel placed against min(compute
ceiling, intensity x bandwidth ceiling)); the TileOPs "Hardware Microbenchmarks"
README, "Methodology" (Triad, copy, read-only and write-only; 100 warm-up
launches, 5 runs of 200 timed launches, best and median, block sizes
128/256/512 -- plus 1024 here -- on 2 GiB arrays).

Correctness is not checked here (the harness is product code and never runs
the oracle); the parity of every row is covered by the GPU tests.
"""
from __future__ import annotations

import argparse
import csv
import json
import math
import os
import statistics
import sys
import time

import torch

from . import inputs, kbattn
from . import roofline as rf
from .clocks import ClockSampler, gpu_id_for_smi

ATTN_VARIANTS = {"f32": [kbattn.Variant.NAIVE, kbattn.Variant.FUSED, kbattn.Variant.FLASH],
                 "bf16": [kbattn.Variant.TC], "f16": [kbattn.Variant.TC], "q15": [kbattn.Variant.FIXEDPOINT]}

FIELDS = ["kernel", "workload", "variant", "dtype", "block", "p50_ms", "min_ms", "mean_ms", "p99_ms", "tflops",
          "gbs", "bound", "attainable", "roofline_unit", "roofline_frac", "sm_mhz", "clock_reasons", "iters"]


def _stats(ms: list[float]) -> dict:
    s = sorted(ms)
    return {"p50_ms": statistics.median(s), "min_ms": s[0], "mean_ms": statistics.mean(s),
            "p99_ms": s[min(len(s) - 1, int(math.ceil(0.99 * len(s))) - 1)], "iters": len(s)}


def naive_score_bytes(w: inputs.Workload) -> float:
    """Score traffic of the three-pass variant: pass 1 writes each visible score,
    pass 2 reads it twice and writes it once, pass 3 reads it once."""
    visible = w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S
    return 5.0 * 4.0 * w.N * visible


def row_clock(clocks: dict) -> tuple:
    """The SM clock and throttle reasons of a row: the median of the samples
    taken while the row ran; a row shorter than one sampling period has none
    (its neighbours' samples would mostly show the idle clock between rows)."""
    if clocks.get("window") != "timed region":
        return None, "no sample (row shorter than one clock sample)"
    return clocks["sm_mhz"], "+".join(clocks["reasons"]) or "none"


def attention_row(w, variant, peaks, dev_info, seconds, sampler, bandwidth_gbs: float, warmup: int = 10,
                  iters: int = 0) -> dict:
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    o = torch.empty_like(q)
    ws = None
    if variant == kbattn.Variant.NAIVE:
        nbytes = kbattn.kb_attn_workspace_bytes(w.B, w.H, w.S, w.d, kbattn.DType.F32, variant)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if iters <= 0:  # as many launches as fill `seconds`
        probe = kbattn.kb_attn_bench(q, k, v, o, w.causal, w.scale, variant, warmup=3, iters=3, workspace=ws)
        iters = max(10, min(5000, int(seconds / max(statistics.median(probe) * 1e-3, 1e-6))))
    t0 = time.time()
    ms = kbattn.kb_attn_bench(q, k, v, o, w.causal, w.scale, variant, warmup=warmup, iters=iters, workspace=ws)
    t1 = time.time()
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise RuntimeError(f"device error in {w.name} {variant.name}")
    st = _stats(ms)
    clocks = sampler.summary(t0, t1)
    sec = st["p50_ms"] * 1e-3
    tflops = w.flops / sec / 1e12
    io = w.io_bytes
    if variant == kbattn.Variant.TC:
        compute, bound = peaks["bf16_tflops"], "tensor"
        traffic = io
    elif variant == kbattn.Variant.FIXEDPOINT:
        # integer path: multiply-adds counted like FMAs (2 operations each)
        compute = rf.int32_mad_peak_gops(dev_info["sm_count"], dev_info["sm_clock_khz"] / 1e3) / 1e3
        bound = "alu"
        traffic = io
    else:
        # fp32 CUDA-core peak: SMs x 128 lanes x 2 FLOP x the device's maximum clock
        compute = rf.fp32_peak_gflops(dev_info["sm_count"], dev_info["sm_clock_khz"] / 1e3) / 1e3
        bound = "fp32"
        traffic = io + (naive_score_bytes(w) if variant == kbattn.Variant.NAIVE else 0.0)
    intensity = w.flops / traffic
    attainable = rf.attainable(intensity, compute * 1e3, bandwidth_gbs) / 1e3
    if attainable < compute:
        bound = "hbm"
    return {"kernel": "attention", "workload": w.name, "variant": variant.name, "dtype": w.dtype, "block": "",
            **st, "tflops": tflops, "gbs": traffic / sec / 1e9, "bound": bound, "attainable": attainable,
            "roofline_unit": "TFLOP/s", "roofline_frac": tflops / attainable, "sm_mhz": row_clock(clocks)[0],
            "clock_reasons": row_clock(clocks)[1]}


GRAPH_LAUNCHES = 200


def graph_row(w, variant, base: dict, sampler) -> dict:
    """The same problem as ``base`` timed as one CUDA graph of 200 captured
    launches (kbench page, "Implementation details": the launch cost of tiny
    problems); the per-launch statistics are graph times / 200."""
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    o = torch.empty_like(q)
    t0 = time.time()
    ms = kbattn.kb_attn_bench_graph(q, k, v, o, w.causal, w.scale, variant, launches=GRAPH_LAUNCHES,
                                    warmup=5, iters=50)
    t1 = time.time()
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise RuntimeError(f"device error in {w.name} {variant.name} graph")
    st = _stats([x / GRAPH_LAUNCHES for x in ms])
    st["iters"] = len(ms) * GRAPH_LAUNCHES
    sec = st["p50_ms"] * 1e-3
    tflops = w.flops / sec / 1e12
    clocks = sampler.summary(t0, t1)
    row = dict(base)
    row.update({**st, "variant": f"{variant.name}+graph{GRAPH_LAUNCHES}", "tflops": tflops,
                "gbs": base["gbs"] * base["p50_ms"] / st["p50_ms"],
                "roofline_frac": tflops / base["attainable"], "sm_mhz": row_clock(clocks)[0],
                "clock_reasons": row_clock(clocks)[1]})
    return row


def hbm_rows(peaks, dev_info, quick, sampler, only, size_mb: int = 0) -> list[dict]:
    n = inputs.TRIAD_N if not quick else inputs.TRIAD_N // 8
    if size_mb > 0:
        n = size_mb * (1 << 20) // 4
    a = torch.empty(n, dtype=torch.float32, device="cuda")
    b = torch.ones(n, dtype=torch.float32, device="cuda")
    c = torch.full((n,), 2.0, dtype=torch.float32, device="cuda")
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    theo = rf.theoretical_dram_gbs(dev_info["mem_clock_khz"] / 1e3, dev_info["mem_bus_width_bits"])
    rows = []
    runs, iters, warm = (5, 200, 100) if not quick else (2, 20, 5)
    for op in kbattn.HbmOp:
        name = op.name.lower()
        if only and only not in name:
            continue
        nbytes = kbattn.HBM_BYTES_PER_ELEMENT[op] * n
        for block in (128, 256, 512, 1024):
            kbattn.kb_hbm_bench(op, a, b, c, 3.0, out, block=block, warmup=warm, iters=1)
            t0 = time.time()
            per_run = [kbattn.kb_hbm_bench(op, a, b, c, 3.0, out, block=block, warmup=0, iters=iters)
                       for _ in range(runs)]
            t1 = time.time()
            clocks = sampler.summary(t0, t1)
            allms = [x for r in per_run for x in r]
            st = _stats(allms)
            gbs_runs = [nbytes / (statistics.mean(r) * 1e-3) / 1e9 for r in per_run]
            best = max(gbs_runs)
            rows.append({"kernel": name, "workload": f"{n * 4 >> 20} MiB arrays", "variant": name,
                         "dtype": "f32", "block": block, **st, "tflops": 0.0, "gbs": best, "bound": "hbm",
                         "attainable": theo, "roofline_unit": "GB/s", "roofline_frac": best / theo,
                         "sm_mhz": row_clock(clocks)[0], "clock_reasons": row_clock(clocks)[1],
                         "gbs_median_of_runs": statistics.median(gbs_runs),
                         "frac_of_measured_copy": best / peaks["hbm_gbs"]})
    del a, b, c
    torch.cuda.empty_cache()
    return rows


def _mhz(x) -> str:
    return "n/a" if x is None else f"{x}"


CHECKPOINT = "checkpoint.jsonl"


def row_key(row: dict) -> tuple:
    """What identifies a row across runs: kernel, workload, variant, block."""
    return (row.get("kernel"), row.get("workload"), row.get("variant"), str(row.get("block", "")))


def append_checkpoint(out_dir: str, row: dict) -> None:
    """Append one finished row to the checkpoint file (one JSON object per line)."""
    os.makedirs(out_dir, exist_ok=True)
    with open(os.path.join(out_dir, CHECKPOINT), "a") as f:
        f.write(json.dumps(row) + "\n")
        f.flush()
        os.fsync(f.fileno())


def load_checkpoint(out_dir: str) -> dict:
    """Rows of an earlier run's checkpoint by row_key (the last copy of a key
    wins); a line cut short by an interrupted write, or any other line that is
    not a complete row, is ignored."""
    rows = {}
    try:
        with open(os.path.join(out_dir, CHECKPOINT)) as f:
            for line in f:
                try:
                    r = json.loads(line)
                except ValueError:
                    continue
                if isinstance(r, dict) and "kernel" in r and "workload" in r and "variant" in r:
                    rows[row_key(r)] = r
    except OSError:
        pass
    return rows


def write_outputs(rows, out_dir, meta):
    os.makedirs(out_dir, exist_ok=True)
    with open(os.path.join(out_dir, "results.jsonl"), "w") as f:
        f.write(json.dumps({"meta": meta}) + "\n")
        for r in rows:
            f.write(json.dumps(r) + "\n")
    with open(os.path.join(out_dir, "results.csv"), "w", newline="") as f:
        wr = csv.DictWriter(f, fieldnames=FIELDS, extrasaction="ignore")
        wr.writeheader()
        wr.writerows(rows)
    md = [f"Device: {meta['device']} ({meta['sms']} SMs); peaks: {meta['peaks_source']} "
          f"bf16 {meta['peaks']['bf16_tflops']} TFLOP/s, copy {meta['peaks']['hbm_gbs']} GB/s; attention bandwidth roof "
          f"{meta['attention_bandwidth_gbs']:.0f} GB/s ({meta['attention_bandwidth_source']}); "
          f"theoretical HBM {meta['theoretical_hbm_gbs']:.0f} GB/s; fp32 FMA peak {meta['fp32_peak_tflops']:.1f} TFLOP/s.",
          "",
          "| kernel | workload | variant | block | p50 ms | min ms | p99 ms | TFLOP/s | GB/s | bound | attainable | frac | SM MHz |",
          "|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        md.append(f"| {r['kernel']} | {r['workload']} | {r['variant']} | {r['block']} | {r['p50_ms']:.4f} | "
                  f"{r['min_ms']:.4f} | {r['p99_ms']:.4f} | {r['tflops']:.2f} | {r['gbs']:.0f} | {r['bound']} | "
                  f"{r['attainable']:.1f} {r['roofline_unit']} | {r['roofline_frac']:.3f} | {_mhz(r['sm_mhz'])} |")
    with open(os.path.join(out_dir, "results.md"), "w") as f:
        f.write("\n".join(md) + "\n")
    return "\n".join(md)


def tc_sweep_table(rows) -> str | None:
    """The tensor-core sweep (16 heads, bf16, d = 64 and 128, S = 128 ... 16384):
    per d and S the median time, TFLOP/s, the fraction of the measured bf16
    peak and the algorithmic GB/s (Q, K, V and O once)."""
    names = {w.name: w for w in inputs.TC_SWEEP}
    by = {r["workload"]: r for r in rows if r["workload"] in names and r["kernel"] == "attention"}
    if not by:
        return None
    md = ["| d | S | p50 ms | TFLOP/s | frac of measured bf16 peak | GB/s | SM MHz |", "|---|---|---|---|---|---|---|"]
    for w in inputs.TC_SWEEP:
        r = by.get(w.name)
        if r is not None:
            md.append(f"| {w.d} | {w.S} | {r['p50_ms']:.4f} | {r['tflops']:.1f} | {r['roofline_frac']:.3f} | "
                      f"{r['gbs']:.0f} | {_mhz(r['sm_mhz'])} |")
    return "\n".join(md)


def sweep_table(rows) -> str | None:
    """The kbench page's sequence sweep (16 heads, d = 64, fp32) as the page
    reports it: per S and variant the median time, GFLOP/s, effective GB/s
    (naive: with its modelled score traffic) and the speed-up over the naive
    variant; the page's "Expected results" give naive 1.0x, fused ~2.2x and
    flash ~4.7x at S = 2048 on its own (unnamed) GPU."""
    names = {w.name: w for w in inputs.KBENCH_SWEEP}
    by = {(r["workload"], r["variant"]): r for r in rows if r["workload"] in names and r["kernel"] == "attention"}
    if not by:
        return None
    md = ["| S | variant | p50 ms | GFLOP/s | effective GB/s | speed-up over naive | frac of FMA roof |",
          "|---|---|---|---|---|---|---|"]
    for w in inputs.KBENCH_SWEEP:
        base = by.get((w.name, "NAIVE"))
        for v in ("NAIVE", "FUSED", "FLASH"):
            r = by.get((w.name, v))
            if r is None:
                continue
            up = f"{base['p50_ms'] / r['p50_ms']:.2f}x" if base else ""
            md.append(f"| {w.S} | {v} | {r['p50_ms']:.4f} | {r['tflops'] * 1e3:.0f} | {r['gbs']:.0f} | {up} | "
                      f"{r['roofline_frac']:.3f} |")
    return "\n".join(md)


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--only", default="", help="run only rows whose workload, variant or kernel contains this")
    p.add_argument("--out", default="harness_out")
    p.add_argument("--seconds", type=float, default=0.5, help="timed seconds per attention row")
    p.add_argument("--quick", action="store_true", help="small HBM arrays and few repetitions")
    p.add_argument("--no-hbm", action="store_true")
    p.add_argument("--no-attention", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="only the kbench page's sequence sweep (fp32, 16 heads, d = 64, S = 128 ... 2048) and its "
                        "tensor-core widening (bf16, d = 64 and 128, S = 128 ... 16384); no HBM rows unless "
                        "--with-hbm")
    p.add_argument("--with-hbm", action="store_true", help="with --sweep: run the HBM kernels too")
    p.add_argument("--resume", action="store_true",
                   help="reuse the rows in OUT/checkpoint.jsonl and measure only the missing ones")
    p.add_argument("--config", default="", help="comma-separated workload names (default: all, or the sweep's)")
    p.add_argument("--variant", default="",
                   help="comma-separated variants: NAIVE, FUSED, FLASH, TC, FIXEDPOINT (default: each workload's all)")
    p.add_argument("--warmup", type=int, default=10, help="untimed launches before each attention row")
    p.add_argument("--iters", type=int, default=0,
                   help="timed launches per attention row (default: as many as fill --seconds)")
    p.add_argument("--size-mb", type=int, default=0, help="MiB per HBM-kernel array (default 2048; --quick 256)")
    args = p.parse_args(argv)
    if args.sweep and not args.with_hbm:
        args.no_hbm = True
    return args


def attention_plan(args) -> list:
    """The (workload, variant) pairs a run measures, in order; raises on an
    unknown workload or variant name."""
    if args.no_attention:
        return []
    todo = list(inputs.KBENCH_SWEEP + inputs.TC_SWEEP) if args.sweep else list(inputs.WORKLOADS.values())
    if args.config:
        names = [n.strip() for n in args.config.split(",") if n.strip()]
        unknown = [n for n in names if n not in inputs.WORKLOADS]
        if unknown:
            raise SystemExit(f"unknown workload(s) {unknown}; known: {sorted(inputs.WORKLOADS)}")
        todo = [inputs.WORKLOADS[n] for n in names]
    wanted = None
    if args.variant:
        wanted = [n.strip().upper() for n in args.variant.split(",") if n.strip()]
        bad = [n for n in wanted if n not in kbattn.Variant.__members__ or n == "AUTO"]
        if bad:
            raise SystemExit(f"unknown variant(s) {bad}")
    only = args.only.lower()
    plan = []
    for w in todo:
        for variant in ATTN_VARIANTS[w.dtype]:
            if wanted is not None and variant.name not in wanted:
                continue
            if only and only not in w.name.lower() and only not in variant.name.lower():
                continue
            plan.append((w, variant))
    return plan


def main(argv=None) -> int:
    args = parse_args(argv)
    plan = attention_plan(args)  # unknown names fail here, before anything is measured
    if not torch.cuda.is_available():
        print("the harness needs a CUDA GPU", file=sys.stderr)
        return 2
    from . import build
    build.build()
    kbattn.load()
    dev = torch.cuda.current_device()
    info = kbattn.kb_device_info(dev)
    peaks, src = rf.load_measured_peaks()
    sampler = ClockSampler(gpu_id_for_smi(dev))
    sampler.start()
    time.sleep(0.3)
    rows, hbm = [], []
    only = args.only.lower()
    done = load_checkpoint(args.out) if args.resume else {}
    if not args.resume and os.path.exists(os.path.join(args.out, CHECKPOINT)):
        os.remove(os.path.join(args.out, CHECKPOINT))
    try:
        # the HBM kernels first: the best STREAM Triad of this run is the attention rows'
        # bandwidth roof (the measured copy figure when the HBM rows are not run)
        if not args.no_hbm:
            earlier = [r for r in done.values() if r["kernel"] != "attention"]
            if any(r["kernel"] == "triad" for r in earlier):
                hbm = earlier  # the HBM rows of the interrupted run, Triad included
            else:
                for r in hbm_rows(peaks, info, args.quick, sampler, only, args.size_mb):
                    hbm.append(r)
                    append_checkpoint(args.out, r)
                    print(json.dumps(r), flush=True)
        triad = [r["gbs"] for r in hbm if r["kernel"] == "triad"]
        bandwidth = max(triad) if triad else peaks["hbm_gbs"]
        bw_source = "best STREAM Triad of this run" if triad else "measured copy bandwidth (no Triad run)"
        for w, variant in plan:
            base = done.get(("attention", w.name, variant.name, ""))
            if base is None:
                base = attention_row(w, variant, peaks, info, args.seconds, sampler, bandwidth, args.warmup,
                                     args.iters)
                append_checkpoint(args.out, base)
                print(json.dumps(base), flush=True)
            rows.append(base)
            if w.flops < 1e8:  # launch-bound sizes: also timed as a CUDA graph
                g = done.get(("attention", w.name, f"{variant.name}+graph{GRAPH_LAUNCHES}", ""))
                if g is None:
                    g = graph_row(w, variant, base, sampler)
                    append_checkpoint(args.out, g)
                    print(json.dumps(g), flush=True)
                rows.append(g)
        rows += hbm
    finally:
        sampler.stop()
    meta = {"device": info["name"], "sms": info["sm_count"], "peaks": peaks, "peaks_source": src,
            "attention_bandwidth_gbs": bandwidth, "attention_bandwidth_source": bw_source,
            "theoretical_hbm_gbs": rf.theoretical_dram_gbs(info["mem_clock_khz"] / 1e3, info["mem_bus_width_bits"]),
            "fp32_peak_tflops": rf.fp32_peak_gflops(info["sm_count"], info["sm_clock_khz"] / 1e3) / 1e3}
    print(write_outputs(rows, args.out, meta))
    sweep = "\n\n".join(s for s in (sweep_table(rows), tc_sweep_table(rows)) if s)
    if sweep:
        with open(os.path.join(args.out, "sweep.md"), "w") as f:
            f.write(sweep + "\n")
        print(sweep)
    return 0


if __name__ == "__main__":
    sys.exit(main())
