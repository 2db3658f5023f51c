"""The benchmark's one-line JSON contract: every key the line carries, with
its type and unit, for the reference arm (the oracle on the host cores; runs
on CPU) and for the library's own arm (GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config"}


def run_bench(*args, timeout=600):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                       timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]  # exactly one line on stdout
    return json.loads(lines[0])


def check_common(line, steps, warmup, dtype):
    assert BASE_KEYS <= set(line), BASE_KEYS - set(line)
    assert line["steps"] == steps and line["warmup"] == warmup and line["n_gpus"] == 1
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["config"]["workload"] == "bf16_causal_b4h16s4096d128"
    assert line["dtype"] == dtype and line["data"] == "synthetic"  # the arithmetic type of the arm


def test_reference_arm_line():
    import bench
    from roofline_benchmarking_gb300 import inputs
    line = run_bench("--impl", "reference", "--steps", "2", "--warmup", "1", "--reference-seconds", "1.5")
    check_common(line, 2, 1, "f64")
    assert line["impl"] == "reference"
    # the same config dict the library's arm prints for this workload
    assert line["config"] == json.loads(json.dumps(bench.bench_config(inputs.BF16_CAUSAL_S4096, 1)))
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert cb["cores_available"] >= cb["cores"] and cb["rows_per_step"] > 0
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_roofline_kernel_follows_the_workload():
    import bench
    from roofline_benchmarking_gb300 import inputs
    want = {"bf16_causal_b4h16s4096d128": ("attn_tc_kernel<128,bf16>", "tensor"),
            "bf16_b16h12s2048d64": ("attn_tc64_kernel<bf16>", "tensor"),
            "f16_b16h12s2048d64": ("attn_tc64_kernel<f16>", "tensor"),
            "bf16_causal_b2h16s4096d256": ("attn_tc256_kernel<bf16>", "tensor"),
            "f32_b1h8s1024d64": ("flash_f32x2_kernel", "alu"),
            "f32_b1h8s1024d64_causal": ("flash_f32x2_kernel + flash_merge_kernel", "alu")}
    for name, (kernel, bound) in want.items():
        k = bench.kernel_for(inputs.WORKLOADS[name], 152)
        assert (k["kernel"], k["bound"]) == (kernel, bound), name
    assert bench.kernel_for(inputs.F32_S1024_CAUSAL, 152)["launches_per_step"] == 2
    assert bench.metric_for(inputs.BF16_CAUSAL_S4096) == bench.METRIC


@pytest.mark.gpu
def test_library_arm_line():
    line = run_bench("--steps", "5", "--warmup", "3", "--e2e-steps", "3", "--cpu-seconds", "1", "--no-triad",
                     "--soak-seconds", "0.5")
    check_common(line, 5, 3, "bf16")
    assert line.get("impl", "ours") != "reference"
    r = line["roofline"]
    assert r["kernel"] == "attn_tc_kernel<128,bf16>"
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert r["achieved"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    assert r["bandwidth_source"].endswith("(no Triad in this run)") and r["attainable"] > 0
    sus = r["sustained"]
    assert sus["launches"] >= 1 and sus["achieved"] > 0 and sus["clock_samples"] >= 1
    c = line["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list) and "timed_region_only" in c
    assert line["gpu_launches"] >= 5
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "TFLOP/s" and e2e["output_equals_device_run"] is True
    assert e2e["h2d_bytes_per_step"] == 3 * 4 * 16 * 4096 * 128 * 2  # Q, K, V in bf16
    assert e2e["d2h_bytes_per_step"] == 4 * 16 * 4096 * 128 * 2      # O
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0


@pytest.mark.gpu
def test_library_arm_line_names_the_d64_kernel():
    line = run_bench("--workload", "bf16_b16h12s2048d64", "--steps", "3", "--warmup", "3", "--no-e2e",
                     "--no-cpu-baseline", "--no-triad", "--soak-seconds", "0")
    assert line["config"]["workload"] == "bf16_b16h12s2048d64"
    assert line["roofline"]["kernel"] == "attn_tc64_kernel<bf16>"
    assert line["roofline"]["traffic"] is None  # the committed capture is of another workload


def test_profiled_traffic_only_for_the_captured_workload_and_source():
    import bench
    h = bench.kernel_source_hash()
    traffic = bench.profiled_traffic(h, bench.HEADLINE)
    assert traffic is not None and traffic > 0  # the committed capture is of the current source
    assert bench.profiled_traffic(h, "bf16_causal_b1h32s16384d128_sharp") is None
    assert bench.profiled_traffic("0" * 16, bench.HEADLINE) is None


def test_l2_policy_in_the_config():
    import bench
    from roofline_benchmarking_gb300 import inputs
    big = bench.bench_config(inputs.BF16_CAUSAL_S4096, 1)["l2"]
    assert big.startswith("no flush") and "256 MiB" in big and not bench.flushes_l2(inputs.BF16_CAUSAL_S4096)
    small = bench.bench_config(inputs.F32_S1024, 1)["l2"]
    assert small.startswith("flushed") and bench.flushes_l2(inputs.F32_S1024)
