#!/usr/bin/env python
"""Attention-forward benchmark: one JSON line on stdout (rank 0).

A step is one kb_attn_fwd call over the whole workload (default: bf16 causal
B=4 H=16 S=4096 d=128, seed 2, normal(0,1) rounded to bf16), i.e. one pass of
the tensor-core hot path: TMA staging, S = Q K^T on tcgen05, online softmax,
O += P V, normalisation and the bf16 store.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl ours (default): W untimed steps, then exactly K steps between CUDA
events on the launching stream with a barrier and a device synchronise on both
sides; the max over ranks is reported. value = FLOPs of all ranks / time.
Also reported: the roofline fraction of the kernel (per-launch CUDA events;
the bandwidth roof is the STREAM Triad measured in the same run), a sustained
rate from ~2 s of back-to-back launches right after the timed region with the
SM clocks nvidia-smi sampled over both, the end-to-end rate through the
library's host-to-host call kb_attn_fwd_host with pinned host buffers (copies
inside the timed region), the Triad ceiling itself and the CPU oracle on a
bounded row sample.

--impl reference: the CPU oracle (the method's plain definition, one host core,
double precision) timed on a bounded row sample of the same workload per step.

Under torchrun each rank runs the whole workload on its own GPU (replicas,
weak scaling): attention heads are independent and no data moves between GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, B4 H16 S4096 d128 causal) and % of roofline"
HEADLINE = "bf16_causal_b4h16s4096d128"


def metric_for(w) -> str:
    return METRIC if w.name == HEADLINE else f"attention fwd TFLOP/s ({w.name}) and % of roofline"
UNIT = "TFLOP/s"
TC_SOURCES = ["attn_tc.cu", "tc_ptx.cuh"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_tc_bf16_causal_b4h16s4096d128.md")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of the CPU baseline")
    p.add_argument("--reference-seconds", type=float, default=120.0,
                   help="total oracle time budget of --impl reference")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--soak-seconds", type=float, default=2.0,
                   help="back-to-back launches after the timed region for the sustained rate and clocks (0: none)")
    p.add_argument("--no-triad", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--oracle-table", action="store_true",
                   help="time the CPU oracle on every workload (bounded row samples, one thread and all "
                        "host threads) and print a Markdown table instead of the JSON line")
    p.add_argument("--oracle-seconds", type=float, default=10.0, help="oracle time budget per workload and mode")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        import torch.distributed as dist
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def aggregate_tflops(flops_per_replica: float, world: int, ms_per_step: float) -> float:
    """Whole-job rate: every rank runs the whole workload (replicas), and the
    step time is the maximum over ranks."""
    return flops_per_replica * world / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------------------- clocks
from roofline_benchmarking_gb300.clocks import ClockSampler, gpu_id_for_smi  # noqa: E402


# ----------------------------------------------------------------------------- helpers
def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in TC_SOURCES:
        with open(os.path.join(ROOT, "roofline_benchmarking_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(expected_hash: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source and on this workload; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    mh = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    mw = re.search(r"profiled_workload:\s*(\S+)", text)
    if not mh or not mt or not mw or mh.group(1) != expected_hash or mw.group(1) != workload:
        return None
    return float(mt.group(1))


def host_cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        if m:
            return m.group(1).strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def workload_config(w, extra=None) -> dict:
    dist = (f"uniform[-1,1]" if w.dist == "uniform" else
            f"Q,K normal(0,{w.sigma_qk:g}), V normal(0,{w.sigma_v:g})")
    rounded = {"bf16": " rounded to bf16", "f16": " rounded to fp16", "q15": " rounded to Q15"}.get(w.dtype, "")
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "d": w.d, "causal": w.causal,
           "dtype": w.dtype, "seed": w.seed, "distribution": dist + rounded,
           "scale": "1/sqrt(d)", "flops_per_step": w.flops}
    if extra:
        cfg.update(extra)
    return cfg


L2_BYTES = int(126.5 * 2**20)  # GB300's L2


def flushes_l2(w) -> bool:
    """Whether the timed steps flush L2 between them: when a step's inputs and
    output fit in L2 (else they are larger than L2 and evict each other)."""
    return w.io_bytes <= L2_BYTES


def bench_config(w, world: int) -> dict:
    """The workload as both arms print it (identical dicts, so the two lines
    describe the same job): shape, draws, the L2 policy and the parallelism."""
    io = w.io_bytes / 2**20
    return workload_config(w, {
        "l2": (f"flushed: a {2 * L2_BYTES / 2**20:.0f} MiB write before each timed step, outside its CUDA events "
               f"(the step's inputs and output, {io:.1f} MiB, fit in the 126.5 MiB L2); ms_per_step is the mean "
               f"of the per-step event times" if flushes_l2(w) else
               f"no flush: each step's inputs and output ({io:.0f} MiB) exceed the 126.5 MiB L2"),
        "parallelism": f"replicas x{world} (each GPU runs the whole workload; no collective)"})


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def kernel_for(w, sms: int) -> dict:
    """The library kernel that runs workload ``w`` (one launch per step unless
    noted), what bounds it, and the peak it is measured against."""
    if w.dtype in ("bf16", "f16"):
        name = (f"attn_tc256_kernel<{w.dtype}>" if w.d == 256 else
                f"attn_tc64_kernel<{w.dtype}>" if w.d <= 64 else f"attn_tc_kernel<128,{w.dtype}>")
        return {"kernel": name, "bound": "tensor", "launches_per_step": 1, "peak_key": "bf16_tflops",
                "peak_note": ("measured bf16 burst (cuBLAS 8192^3)" if w.dtype == "bf16" else
                              "measured bf16 burst (cuBLAS 8192^3) x 1, the nominal fp16:bf16 dense ratio")}
    if w.dtype == "q15":
        return {"kernel": "q15_attn_kernel", "bound": "alu", "launches_per_step": 1, "peak_key": None,
                "peak_note": "integer multiply-add lanes: SMs x 64 dp2a lanes x 2 x max SM clock"}
    # the library splits the heavier causal query tiles over two blocks on small grids
    # (N * ceil(S / 64) <= 2 x SMs, S >= 256) and merges them in a second launch
    tiles = (w.S + 63) // 64
    split = w.causal and tiles >= 4 and w.N * tiles <= 2 * sms
    name = "flash_f32x2_kernel" if w.d <= 64 else "flash_f32_kernel"
    return {"kernel": name + (" + flash_merge_kernel" if split else ""), "bound": "alu",
            "launches_per_step": 2 if split else 1, "peak_key": None,
            "peak_note": "fp32 FMA: SMs x 128 lanes x 2 x max SM clock"}


# ----------------------------------------------------------------------------- CPU oracle
def widen(q, k, v):
    """Q, K, V as float64 numpy arrays (exact) for the oracle."""
    import oracle
    orc = oracle.get()
    return tuple(orc._f64(t) for t in (q, k, v))


def oracle_sample(w, q64, k64, v64, seconds: float, seed: int = 0, gpu_out=None):
    """Rows of the workload evaluated by the oracle until `seconds` elapse.
    q64, k64, v64 come from widen(). Returns (flops, elapsed, rows, parity or None)."""
    import numpy as np
    import torch

    import oracle
    from roofline_benchmarking_gb300 import inputs

    heads, rows = inputs.sample_rows(w, per_head=min(w.S, 512), seed=seed)
    perm = torch.randperm(len(heads), generator=torch.Generator().manual_seed(seed))
    heads, rows = heads[perm].numpy(), rows[perm].numpy()
    orc = oracle.get()
    done, flops, elapsed = 0, 0.0, 0.0
    chunk = 4
    outs = []
    while done < len(heads) and elapsed < seconds:
        h, r = heads[done:done + chunk], rows[done:done + chunk]
        t0 = time.perf_counter()
        o = orc.attn_rows(q64, k64, v64, w.causal, w.scale, h, r)
        elapsed += time.perf_counter() - t0
        outs.append(o)
        vis = (r + 1) if w.causal else np.full(len(r), w.S)
        flops += float(np.sum(4.0 * vis * w.d))
        done += len(h)
    parity = None
    if gpu_out is not None and done:
        got = gpu_out.view(w.N, w.S, w.d)[torch.from_numpy(heads[:done]).cuda(),
                                           torch.from_numpy(rows[:done]).cuda()].float().cpu().numpy()
        diff = np.abs(got - np.concatenate(outs))
        parity = {"rows": int(done), "max_abs": float(diff.max()), "mean_abs": float(diff.mean())}
    return flops, elapsed, int(done), parity


def oracle_threads_rate(w, q64, k64, v64, seconds: float, threads: int, seed: int = 0):
    """The oracle on the same seeded row sample, split over `threads` host
    threads (the oracle's ctypes calls release the GIL). Returns (flops, wall
    seconds, rows)."""
    import concurrent.futures as cf

    import numpy as np
    import torch

    import oracle
    from roofline_benchmarking_gb300 import inputs

    heads, rows = inputs.sample_rows(w, per_head=min(w.S, 512), seed=seed)
    perm = torch.randperm(len(heads), generator=torch.Generator().manual_seed(seed))
    heads, rows = heads[perm].numpy(), rows[perm].numpy()
    orc = oracle.get()
    parts = [(heads[t::threads], rows[t::threads]) for t in range(threads)]
    chunk = max(4, int(4e6 / (4.0 * w.S * w.d)))  # rows per call: a few MFLOP, so Python overhead stays small

    def work(part):
        h_all, r_all = part
        done, flops, t0 = 0, 0.0, time.perf_counter()
        while done < len(h_all) and time.perf_counter() - t0 < seconds:
            h, r = h_all[done:done + chunk], r_all[done:done + chunk]
            orc.attn_rows(q64, k64, v64, w.causal, w.scale, h, r)
            vis = (r + 1) if w.causal else np.full(len(r), w.S)
            flops += float(np.sum(4.0 * vis * w.d))
            done += len(h)
        return flops, done

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(work, parts))
    wall = time.perf_counter() - t0
    return sum(f for f, _ in res), wall, sum(n for _, n in res)


def oracle_table(args) -> int:
    """The CPU oracle's rate on every workload: a time-bounded seeded row sample
    on one thread and on all host threads, with the full-problem time
    extrapolated by the exact FLOP count of the visible keys."""
    import numpy as np

    import oracle
    from roofline_benchmarking_gb300 import inputs

    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    print(f"Host CPU: {host_cpu_model()}; {threads} threads available; budget {args.oracle_seconds:g} s per "
          f"workload and mode.\n")
    print("| workload | rows evaluated (1 thread) | of all rows | 1 thread GFLOP/s | full problem, 1 thread (s) | "
          f"{threads} threads GFLOP/s | full problem, {threads} threads (s) |")
    print("|---|---|---|---|---|---|---|")
    for w in (inputs.SINGLE_HEAD_F32, inputs.F32_S1024, inputs.F32_S1024_CAUSAL, inputs.BF16_CAUSAL_S4096,
              inputs.BF16_S2048_D64, inputs.BF16_CAUSAL_S16384, inputs.BF16_CAUSAL_D256):
        q64, k64, v64 = widen(*inputs.make_qkv(w))
        vis_total = w.N * (w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S)
        full_flops = 4.0 * w.d * vis_total
        f1, t1, n1, _ = oracle_sample(w, q64, k64, v64, args.oracle_seconds, seed=7)
        fm, tm, _ = oracle_threads_rate(w, q64, k64, v64, args.oracle_seconds, threads, seed=7)
        r1, rm = f1 / t1, fm / tm
        print(f"| {w.name} | {n1} | {n1 / (w.N * w.S):.2%} | {r1 / 1e9:.2f} | {full_flops / r1:.1f} | "
              f"{rm / 1e9:.2f} | {full_flops / rm:.1f} |", flush=True)
    # the Q15 fixed-point model, whole problem, one thread
    orc = oracle.get()
    for w in (inputs.Q15_SINGLE_HEAD, inputs.Q15_S1024, inputs.Q15_S1024_CAUSAL):
        q, k, v = inputs.make_qkv(w)
        t0 = time.perf_counter()
        orc.attn_q15(q, k, v, w.causal, w.scale)
        t = time.perf_counter() - t0
        vis_total = w.N * (w.S * (w.S + 1) / 2 if w.causal else float(w.S) * w.S)
        ops = 4.0 * w.d * vis_total
        print(f"| {w.name} (Q15 model, integer ops) | {w.N * w.S} | 100.00% | {ops / t / 1e9:.2f} | {t:.2f} | - | - |",
              flush=True)
    del np
    return 0


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, d: Dist):
    if d.rank != 0:
        return 0
    import numpy as np  # noqa: F401

    from roofline_benchmarking_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    q64, k64, v64 = widen(*inputs.make_qkv(w))
    per_step = max(args.reference_seconds / max(args.steps + args.warmup, 1), 0.05)
    for i in range(args.warmup):
        oracle_sample(w, q64, k64, v64, per_step, seed=1000 + i)
    tot_f, tot_t, tot_rows = 0.0, 0.0, 0
    for i in range(args.steps):
        f, t, n, _ = oracle_sample(w, q64, k64, v64, per_step, seed=i)
        tot_f += f
        tot_t += t
        tot_rows += n
    value = tot_f / tot_t / 1e12
    sample = (f"{tot_rows} seeded (head, query) rows of {w.name} over {args.steps} steps "
              f"(~{per_step:.2f} s of oracle time per step); single thread, float64")
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "cores_available": host_cores(),
                         "kind": "oracle", "sample": sample, "rows_per_step": tot_rows / args.steps,
                         "cpu": host_cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def triad_ceiling(kbattn, dev_info) -> dict:
    """STREAM Triad over three 2 GiB fp32 arrays; the TileOPs protocol: 100
    warm-up launches, then 5 runs of 200 timed launches, per block size
    (128/256/512 as on the page, plus 1024); the best run calibrates."""
    import torch

    from roofline_benchmarking_gb300 import inputs
    from roofline_benchmarking_gb300 import roofline as rf

    n = inputs.TRIAD_N
    a = torch.empty(n, dtype=torch.float32, device="cuda")
    b = torch.ones(n, dtype=torch.float32, device="cuda")
    c = torch.full((n,), 2.0, dtype=torch.float32, device="cuda")
    nbytes = 3.0 * n * 4
    best, per_block = 0.0, {}
    for block in (128, 256, 512, 1024):
        kbattn.kb_triad_bench(a, b, c, 3.0, block=block, warmup=100, iters=1)
        runs = []
        for _ in range(5):
            ms = kbattn.kb_triad_bench(a, b, c, 3.0, block=block, warmup=0, iters=200)
            runs.append(nbytes / (statistics.mean(ms) * 1e-3) / 1e9)
        per_block[block] = {"best_gbs": max(runs), "median_gbs": statistics.median(runs)}
        best = max(best, max(runs))
    ok = bool((a[:1024] == 7.0).all())
    theo = rf.theoretical_dram_gbs(dev_info["mem_clock_khz"] / 1e3, dev_info["mem_bus_width_bits"])
    del a, b, c
    torch.cuda.empty_cache()
    return {"best_gbs": best, "per_block": per_block, "theoretical_gbs": theo,
            "calibration": rf.calibration(best, theo), "bytes_per_launch": nbytes, "check_7": ok,
            "theoretical_formula": "2 x memory clock x bus width / 8 (device attributes)"}


def soak(step, stream, seconds: float, ms_per_step: float, sampler) -> dict:
    """Back-to-back steps for about ``seconds`` right after the timed region, with
    the clock sampler running: the sustained rate under the power cap, next to
    the burst figure of the short timed region."""
    import torch

    n = max(1, int(math.ceil(seconds / max(ms_per_step * 1e-3, 1e-6))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    return {"launches": n, "ms_per_launch": e0.elapsed_time(e1) / n, "seconds": t1 - t0,
            "clocks": sampler.summary(t0, t1), "window": (t0, t1)}


def run_ours(args, d: Dist):
    import torch

    from roofline_benchmarking_gb300 import build as kb_build
    from roofline_benchmarking_gb300 import inputs, kbattn
    from roofline_benchmarking_gb300 import roofline as rf

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the attention library has no CPU path)")
    torch.cuda.set_device(d.local_rank)
    d.init("nccl")
    kb_build.build()
    kbattn.load()
    w = inputs.WORKLOADS[args.workload]
    dev = torch.cuda.current_device()
    info = kbattn.kb_device_info(dev)
    stream = torch.cuda.current_stream()
    kinfo = kernel_for(w, info["sm_count"])

    qh, kh, vh = inputs.make_qkv(w)
    q, k, v = (t.cuda() for t in (qh, kh, vh))
    o = torch.empty_like(q)
    variant = {"f32": kbattn.Variant.FLASH, "q15": kbattn.Variant.FIXEDPOINT}.get(w.dtype, kbattn.Variant.TC)

    def step():
        kbattn.kb_attn_fwd(q, k, v, o, causal=w.causal, scale=w.scale, variant=variant, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise SystemExit("device error during warm-up")

    sampler = ClockSampler(gpu_id_for_smi(dev))
    sampler.start()
    time.sleep(0.35)  # let the sampler attach before the timed region
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # a workload that fits in L2 gets an L2 flush (a write twice the L2's size) before each step
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if flushes_l2(w) else None
    d.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    t_begin.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    d.barrier()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # with flushes, the steps' own device time (the flushes sit between the events)
    total_ms = sum(launch_ms) if flush is not None else t_begin.elapsed_time(t_end)
    del flush
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise SystemExit("device error in the timed region")
    sus = soak(step, stream, args.soak_seconds, total_ms / K, sampler) if args.soak_seconds > 0 else None
    sampler.stop()
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise SystemExit("device error in the soak")
    narrow = sampler.summary(h0, h1)
    if sus is not None:
        # the timed region (milliseconds long) and the seconds of the same kernel after it
        clocks = sampler.summary(h0 - 0.3, sus["window"][1])
        clocks["window"] = f"timed region and the {sus['seconds']:.1f} s soak of the same kernel right after it"
    else:
        clocks = dict(narrow)
    clocks["timed_region_only"] = narrow

    total_ms = d.max(total_ms)
    ms_per_step = total_ms / K
    value = aggregate_tflops(w.flops, d.world, ms_per_step)

    peaks, src = rf.load_measured_peaks()
    mean_launch_s = statistics.mean(launch_ms) * 1e-3
    achieved = w.flops / mean_launch_s / 1e12
    intensity = w.flops / w.io_bytes
    if kinfo["bound"] == "tensor":
        peak, peak_sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
        peak_source = f"{src} {kinfo['peak_note']}"
    else:
        peak = rf.fp32_peak_gflops(info["sm_count"], info["sm_clock_khz"] / 1e3) / 1e3
        peak_sus, peak_source = None, kinfo["peak_note"]
    roof = {
        "kernel": kinfo["kernel"], "bound": kinfo["bound"], "achieved": achieved,
        "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_source,
        "frac_of_sustained_peak": achieved / peak_sus if peak_sus else None,
        "traffic": None, "algorithmic_flops_per_launch": w.flops, "algorithmic_bytes_per_launch": w.io_bytes,
        "intensity_flop_per_byte": intensity,
        "launch_ms": {"mean": statistics.mean(launch_ms), "p50": statistics.median(launch_ms),
                      "min": min(launch_ms), "p99": sorted(launch_ms)[int(0.99 * (K - 1))]},
        "timing": "CUDA events around each launch on the launching stream",
    }
    if kinfo["kernel"].startswith("attn_tc_kernel<128,bf16>"):
        traffic = profiled_traffic(kernel_source_hash(), w.name)
        if traffic is not None:
            roof["traffic"] = traffic
    if sus is not None:
        sus_tf = w.flops / (sus["ms_per_launch"] * 1e-3) / 1e12
        c = sus["clocks"]
        roof["sustained"] = {
            "launches": sus["launches"], "seconds": sus["seconds"], "ms_per_launch": sus["ms_per_launch"],
            "achieved": sus_tf, "frac_of_sustained_peak": sus_tf / peak_sus if peak_sus else None,
            "frac_of_burst_peak": sus_tf / peak, "sm_mhz": c["sm_mhz"], "sm_max_mhz": c["sm_max_mhz"],
            "power_w_median": c.get("power_w_median"), "power_w_max": c.get("power_w_max"),
            "reasons": c["reasons"], "clock_samples": c["samples"],
            "timing": "CUDA events around the whole back-to-back run on the launching stream"}

    line = {
        "metric": metric_for(w), "value": value, "unit": UNIT, "n_gpus": d.world, "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": bench_config(w, d.world),
        "device": {"name": info["name"], "sms": info["sm_count"], "variant": variant.name},
        "clocks": clocks, "gpu_launches": K * kinfo["launches_per_step"], "roofline": roof,
    }

    if not args.no_e2e:
        line["e2e"] = e2e_rate(args, w, qh, kh, vh, q, k, v, o, variant, d)

    triad = None
    if d.rank == 0 and not args.no_triad and d.world == 1:
        triad = line["triad"] = triad_ceiling(kbattn, info)
    # the bandwidth roof: this run's STREAM Triad, else the measured copy figure
    if triad is not None:
        bw, bw_src = triad["best_gbs"], "STREAM Triad measured in this run"
    else:
        bw, bw_src = peaks["hbm_gbs"], f"{src} copy bandwidth (no Triad in this run)"
    roof["bandwidth_gbs"] = bw
    roof["bandwidth_source"] = bw_src
    roof["attainable"] = rf.attainable(intensity, peak * 1e3, bw) / 1e3
    roof["frac_of_attainable"] = achieved / roof["attainable"]

    if d.rank == 0 and d.world == 1 and not args.no_cpu_baseline:
        f, t, n, parity = oracle_sample(w, *widen(qh, kh, vh), args.cpu_seconds, seed=0, gpu_out=o)
        line["cpu_baseline"] = {
            "value": f / t / 1e12, "unit": UNIT, "cores": 1, "cores_available": host_cores(), "kind": "oracle",
            "sample": f"{n} seeded (head, query) rows of {w.name} ({t:.1f} s, single thread, float64)",
            "cpu": host_cpu_model(), "parity_of_sampled_rows": parity}

    if d.rank == 0:
        print(json.dumps(line), flush=True)
    d.close()
    return 0


def e2e_rate(args, w, qh, kh, vh, q, k, v, o, variant, d: Dist) -> dict:
    """The same metric through the library's host-to-host call
    kb_attn_fwd_host: every step copies its Q, K, V from pinned host buffers
    into device staging buffers, runs the forward pass and copies O back into a
    pinned host buffer, all inside the library call on one stream. Consecutive
    steps alternate between two streams, each with its own device buffers and
    host output buffer, so one step's copies overlap its neighbour's kernel.
    The timed region runs from before the first step's input copy to after the
    last step's output copy."""
    import torch

    from roofline_benchmarking_gb300 import kbattn

    o_ref = o.clone()  # the device-resident run's output, for a bit-exact check below
    qp, kp, vp = (t.pin_memory() for t in (qh, kh, vh))
    op = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    dev = [(q, k, v, o), tuple(torch.empty_like(t) for t in (q, k, v, o))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def step(i):
        sl = i % 2
        dq, dk, dv, do = dev[sl]
        kbattn.kb_attn_fwd_host(qp, kp, vp, op[sl], dq, dk, dv, do, causal=w.causal, scale=w.scale,
                                variant=variant, stream=streams[sl])

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    K = max(args.e2e_steps, 1)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    last = torch.cuda.Event()
    d.barrier()
    torch.cuda.synchronize()
    t0.record(streams[0])
    streams[1].wait_event(t0)
    for i in range(K):
        step(i)
    last.record(streams[(K - 1) % 2])
    other = streams[K % 2]
    other.wait_event(last)
    t1.record(other)
    torch.cuda.synchronize()
    d.barrier()
    ms = d.max(t0.elapsed_time(t1)) / K
    if kbattn.kb_check_device_error() != kbattn.Status.OK:
        raise SystemExit("device error in the end-to-end region")
    same = bool(torch.equal(op[(K - 1) % 2], o_ref.cpu()))
    h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
    d2h = op[0].numel() * op[0].element_size()
    return {"value": aggregate_tflops(w.flops, d.world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": K, "host_buffers": "pinned",
            "api": "kb_attn_fwd_host (host-to-host C-ABI call)",
            "pipelining": "steps alternate over 2 streams and 2 device buffer sets; copies overlap the "
                          "neighbouring step's kernel",
            "output_equals_device_run": same}


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_table:
        return oracle_table(args)
    d = Dist()
    if args.impl == "reference":
        return run_reference(args, d)
    return run_ours(args, d)


if __name__ == "__main__":
    sys.exit(main())
