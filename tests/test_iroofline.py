"""Host logic of the hierarchical instruction roofline (GPU-Roofline-Python
page, "Metrics Used"): parsing ncu's per-launch CSV, per-kernel aggregation,
the intensity and warp-GIPS points per memory level and the binding level."""
import pytest

from roofline_benchmarking_gb300 import iroofline as ir

HDR = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
       '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')


def row(lid, kernel, metric, unit, value):
    return (f'"{lid}","1","python3","h","{kernel}","1","7","(256, 1, 1)","(8, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"')


K1 = "void kb::(anonymous namespace)::stream_kernel<256, kb::(anonymous namespace)::TriadOp>(float *, unsigned long)"
K2 = "kb::attn_tc_kernel<128>(CUtensorMap_st, int)"


def fixture():
    lines = ["==PROF== Connected to process 1", HDR]
    for lid, k, dur, inst in ((0, K1, "10.0", "3,200,000"), (1, K2, "200", "64,000,000"), (2, K1, "12.0", "3,200,000")):
        lines += [row(lid, k, "gpu__time_duration.sum", "usecond", dur),
                  row(lid, k, "smsp__thread_inst_executed.sum", "inst", inst),
                  row(lid, k, "dram__sectors_read.sum", "sector", "200,000"),
                  row(lid, k, "dram__sectors_write.sum", "sector", "100,000"),
                  row(lid, k, "lts__t_sectors_op_read.sum", "sector", "250,000"),
                  row(lid, k, "lts__t_sectors_op_write.sum", "sector", "100,000"),
                  row(lid, k, "smsp__inst_executed.sum.peak_sustained", "inst/cycle", "608"),
                  row(lid, k, "sm__cycles_elapsed.avg.per_second", "cycle/second", "2,000,000,000"),
                  row(lid, k, "dram__sectors.sum.peak_sustained", "sector/cycle", "62"),
                  row(lid, k, "dram__cycles_elapsed.avg.per_second", "cycle/nsecond", "4")]
    lines.append("==PROF== Disconnected from process 1")
    return "\n".join(lines)


def test_kernel_names_are_shortened():
    assert ir.short_kernel_name(K1) == "stream_kernel<256, kb::TriadOp>"
    assert ir.short_kernel_name(K2) == "attn_tc_kernel<128>"
    assert ir.short_kernel_name("void unnamed>::naive_pv_kernel<64>(const float *, int)") == "naive_pv_kernel<64>"


def test_parse_and_aggregate():
    launches = ir.parse_ncu_csv(fixture())
    assert [ln["id"] for ln in launches] == [0, 1, 2]
    assert launches[0]["metrics"]["gpu__time_duration.sum"] == pytest.approx(10e-6)
    assert launches[0]["metrics"]["smsp__thread_inst_executed.sum"] == 3.2e6
    assert launches[0]["metrics"]["dram__cycles_elapsed.avg.per_second"] == pytest.approx(4e9)
    agg = ir.aggregate(launches)
    tri = agg["stream_kernel<256, kb::TriadOp>"]
    assert tri["launches"] == 2
    assert tri["mean"]["gpu__time_duration.sum"] == pytest.approx(11e-6)
    assert agg["attn_tc_kernel<128>"]["launches"] == 1


def test_points_ceilings_and_bound():
    mean = ir.aggregate(ir.parse_ncu_csv(fixture()))["stream_kernel<256, kb::TriadOp>"]["mean"]
    ceil = ir.ceilings(mean, hbm_gbs=6400.0)
    assert ceil["inst"] == pytest.approx(608 * 2.0)           # warp GIPS
    assert ceil["HBM"] == pytest.approx(62 * 4.0)             # GTXN/s from ncu's peak rate
    assert ceil["HBM measured"] == pytest.approx(6400.0 / 32)
    pts = ir.roofline_points(mean, 1e-5, ceil)
    assert pts["warp_instructions"] == pytest.approx(1e5)
    assert pts["warp_gips"] == pytest.approx(1e5 / 1e9 / 1e-5)  # 10 warp GIPS
    hbm = pts["levels"]["HBM"]
    assert hbm["transactions"] == 300000 and hbm["intensity"] == pytest.approx(1e5 / 3e5)
    assert hbm["attainable_gips"] == pytest.approx(min(1216, (1 / 3) * 200))
    assert "L2" in pts["levels"] and pts["levels"]["L2"]["ceiling_gtxn_s"] is None  # no L2 peak in the fixture
    assert pts["bound"] == "HBM" and pts["frac"] == pytest.approx(10 / (200 / 3))


def test_metric_list_covers_every_level():
    names = ir.metric_names()
    for ms in ir.LEVELS.values():
        assert set(ms) <= set(names)
    assert ir.INSTRUCTIONS in names and ir.DURATION in names and len(names) == len(set(names))


def test_compute_bound_kernel_reports_instruction_issue():
    mean = {ir.INSTRUCTIONS: 32e9, "dram__sectors_read.sum": 1e6, "smsp__inst_executed.sum.peak_sustained": 608,
            "sm__cycles_elapsed.avg.per_second": 2e9}
    pts = ir.roofline_points(mean, 1.0, ir.ceilings(mean, hbm_gbs=6400.0))
    assert pts["bound"] == "instruction issue" and pts["attainable_gips"] == pytest.approx(1216)
    assert pts["warp_gips"] == pytest.approx(1.0) and pts["frac"] == pytest.approx(1.0 / 1216)
