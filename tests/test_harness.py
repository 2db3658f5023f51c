"""Host logic of the measurement harness (no GPU): the naive variant's score
traffic model, the one-schema CSV / Markdown / JSON output and the row
checkpoint that ``--resume`` reads."""
import csv
import json

import pytest

from roofline_benchmarking_gb300 import harness, inputs


def test_naive_score_traffic_model():
    w = inputs.F32_S1024                      # 8 heads, S = 1024, all S^2 scores visible
    assert harness.naive_score_bytes(w) == 5 * 4 * 8 * 1024 * 1024
    wc = inputs.F32_S1024_CAUSAL              # the lower triangle including the diagonal
    assert harness.naive_score_bytes(wc) == 5 * 4 * 8 * (1024 * 1025 / 2)


def test_outputs_share_one_schema(tmp_path):
    row = {k: 0 for k in harness.FIELDS}
    row.update(kernel="attention", workload="w", variant="TC", dtype="bf16", block="", p50_ms=0.2, min_ms=0.19,
               mean_ms=0.2, p99_ms=0.21, tflops=1200.0, gbs=1000.0, bound="tensor", attainable=1961.8,
               roofline_unit="TFLOP/s", roofline_frac=0.61, sm_mhz=1900.0, clock_reasons="none", iters=10)
    meta = {"device": "GPU", "sms": 152, "peaks": {"bf16_tflops": 1961.8, "hbm_gbs": 6655.3}, "peaks_source": "measured",
            "theoretical_hbm_gbs": 7928.0, "fp32_peak_tflops": 80.5, "attention_bandwidth_gbs": 7262.3,
            "attention_bandwidth_source": "best STREAM Triad of this run"}
    md = harness.write_outputs([row, dict(row, kernel="triad", block=256)], str(tmp_path), meta)
    assert md.count("\n| ") == 3 and "0.610" in md and "7262 GB/s (best STREAM Triad of this run)" in md
    lines = (tmp_path / "results.jsonl").read_text().splitlines()
    assert json.loads(lines[0])["meta"]["sms"] == 152 and len(lines) == 3
    rows = list(csv.DictReader(open(tmp_path / "results.csv")))
    assert [r["kernel"] for r in rows] == ["attention", "triad"] and list(rows[0]) == harness.FIELDS


def test_kbench_sequence_sweep_table():
    # the page's sweep: 16 heads, d = 64, fp32, S = 128 ... 2048
    assert [w.S for w in inputs.KBENCH_SWEEP] == [128, 256, 512, 1024, 2048]
    assert all((w.B, w.H, w.d, w.dtype, w.causal) == (1, 16, 64, "f32", False) for w in inputs.KBENCH_SWEEP)
    assert all(inputs.WORKLOADS[w.name] is w for w in inputs.KBENCH_SWEEP)
    w = inputs.KBENCH_SWEEP[-1]
    rows = [{"kernel": "attention", "workload": w.name, "variant": v, "p50_ms": ms, "tflops": w.flops / ms / 1e9,
             "gbs": 1.0, "roofline_frac": 0.5} for v, ms in (("NAIVE", 2.0), ("FUSED", 1.0), ("FLASH", 0.5))]
    rows.append(dict(rows[0], workload=inputs.F32_S1024.name))  # not a sweep row: ignored
    md = harness.sweep_table(rows)
    lines = md.splitlines()[2:]
    assert len(lines) == 3
    assert lines[0].startswith("| 2048 | NAIVE | 2.0000 |") and "| 1.00x |" in lines[0]
    assert "| 2.00x |" in lines[1] and "| 4.00x |" in lines[2]
    assert harness.sweep_table([rows[-1]]) is None


def test_tensor_core_sweep_table():
    assert [w.S for w in inputs.TC_SWEEP] == [128, 256, 512, 1024, 2048, 4096, 8192, 16384] * 2
    assert [w.d for w in inputs.TC_SWEEP] == [64] * 8 + [128] * 8
    assert all((w.B, w.H, w.dtype, w.causal) == (1, 16, "bf16", False) for w in inputs.TC_SWEEP)
    assert all(inputs.WORKLOADS[w.name] is w for w in inputs.TC_SWEEP)
    w = inputs.TC_SWEEP[-1]
    row = {"kernel": "attention", "workload": w.name, "variant": "TC", "p50_ms": 1.5, "tflops": 1466.0,
           "gbs": 179.0, "roofline_frac": 0.747, "sm_mhz": 1950.0}
    lines = harness.tc_sweep_table([row, dict(row, workload=inputs.F32_S1024.name)]).splitlines()
    assert len(lines) == 3 and lines[2] == "| 128 | 16384 | 1.5000 | 1466.0 | 0.747 | 179 | 1950.0 |"
    assert harness.tc_sweep_table([dict(row, workload="other")]) is None


@pytest.mark.gpu
def test_harness_runs_a_quick_sweep(tmp_path):
    assert harness.main(["--only", "f32_b1h1s64d32", "--no-hbm", "--seconds", "0.02",
                         "--out", str(tmp_path)]) == 0
    rows = [json.loads(x) for x in (tmp_path / "results.jsonl").read_text().splitlines()[1:]]
    assert {r["variant"] for r in rows} == {"NAIVE", "FUSED", "FLASH", "NAIVE+graph200", "FUSED+graph200",
                                            "FLASH+graph200"}
    assert all(r["p50_ms"] > 0 and 0 < r["roofline_frac"] < 2 for r in rows)


def test_checkpoint_keeps_finished_rows_and_ignores_a_cut_line(tmp_path):
    out = str(tmp_path)
    a = {"kernel": "attention", "workload": "w1", "variant": "TC", "block": "", "p50_ms": 0.2}
    g = dict(a, variant="TC+graph200", p50_ms=0.1)
    t1 = {"kernel": "triad", "workload": "2048 MiB arrays", "variant": "triad", "block": 256, "gbs": 7000.0}
    t2 = dict(t1, block=512, gbs=7100.0)
    for r in (a, g, t1, t2):
        harness.append_checkpoint(out, r)
    harness.append_checkpoint(out, dict(a, p50_ms=0.25))          # a later copy of the same row wins
    with open(tmp_path / harness.CHECKPOINT, "a") as f:
        f.write('{"kernel": "attention", "workload": "w2", "vari')  # a write cut off by an interruption
        f.write("\n[1, 2, 3]\n")                                   # not a row
    done = harness.load_checkpoint(out)
    assert set(done) == {("attention", "w1", "TC", ""), ("attention", "w1", "TC+graph200", ""),
                         ("triad", "2048 MiB arrays", "triad", "256"), ("triad", "2048 MiB arrays", "triad", "512")}
    assert done[("attention", "w1", "TC", "")]["p50_ms"] == 0.25
    assert harness.row_key(t1) == ("triad", "2048 MiB arrays", "triad", "256")
    assert harness.load_checkpoint(str(tmp_path / "missing")) == {}


def test_run_plan_from_the_flags():
    plan = harness.attention_plan(harness.parse_args([]))
    every = [(w.name, v.name) for w in inputs.WORKLOADS.values() for v in harness.ATTN_VARIANTS[w.dtype]]
    assert [(w.name, v.name) for w, v in plan] == every
    plan = harness.attention_plan(harness.parse_args(["--config", "f32_b1h8s1024d64,bf16_b16h12s2048d64",
                                                      "--variant", "flash,TC"]))
    assert [(w.name, v.name) for w, v in plan] == [("f32_b1h8s1024d64", "FLASH"), ("bf16_b16h12s2048d64", "TC")]
    plan = harness.attention_plan(harness.parse_args(["--config", "f32_b1h8s1024d64", "--only", "naive"]))
    assert [v.name for _, v in plan] == ["NAIVE"]
    sweep = harness.attention_plan(harness.parse_args(["--sweep", "--variant", "FUSED"]))
    assert [w.S for w, _ in sweep] == [128, 256, 512, 1024, 2048]
    assert harness.attention_plan(harness.parse_args(["--no-attention"])) == []
    args = harness.parse_args(["--warmup", "3", "--iters", "50", "--size-mb", "64"])
    assert (args.warmup, args.iters, args.size_mb) == (3, 50, 64)
    with pytest.raises(SystemExit):
        harness.attention_plan(harness.parse_args(["--config", "no_such_workload"]))
    with pytest.raises(SystemExit):
        harness.attention_plan(harness.parse_args(["--variant", "AUTO"]))


def test_row_clock_needs_a_sample_inside_the_row():
    inside = {"window": "timed region", "sm_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert harness.row_clock(inside) == (2070.0, "sw_power_cap")
    assert harness.row_clock(dict(inside, reasons=[])) == (2070.0, "none")
    near = {"window": "timed region +- 0.3 s", "sm_mhz": 120.0, "reasons": []}
    mhz, why = harness.row_clock(near)
    assert mhz is None and "no sample" in why
