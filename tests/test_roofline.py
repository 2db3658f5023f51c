"""The roofline arithmetic against the worked numbers the pages print
(tests/golden/roofline_worked_examples.txt, each line cites its page)."""
import os

import pytest

from roofline_benchmarking_gb300 import roofline as rf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "roofline_worked_examples.txt")


def golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, args, want, tol, source = (x.strip() for x in line.split("|"))
        kw = {k: float(v) for k, v in (a.split("=") for a in args.split())}
        cases.append(pytest.param(name, kw, float(want), float(tol), id=f"{name}:{source}"))
    return cases


def evaluate(name, kw):
    if name == "calibration":
        return rf.calibration(kw["measured_gbs"], kw["theoretical_gbs"])
    if name == "fp32_peak":
        return rf.fp32_peak_gflops(int(kw["sms"]), kw["clock_mhz"])
    if name == "utilisation":
        return kw["achieved"] / rf.fp32_peak_gflops(int(kw["sms"]), kw["clock_mhz"])
    if name == "clock_from_throughput":
        return rf.clock_from_throughput(kw["gflops"], int(kw["sms"]))
    if name == "dram_theoretical":
        return rf.theoretical_dram_gbs(kw["mem_clock_mhz"], int(kw["bus_width_bits"]))
    raise KeyError(name)


@pytest.mark.parametrize("name,kw,want,tol", golden_cases())
def test_worked_examples(name, kw, want, tol):
    assert abs(evaluate(name, kw) - want) <= tol


def test_attention_work_convention():
    # 4 B H S^2 d, halved when causal: the headline workload is 2.749e11 FLOP
    assert rf.attention_flops(4, 16, 4096, 128, True) == 4 * 4 * 16 * 4096 ** 2 * 128 / 2
    assert abs(rf.attention_flops(4, 16, 4096, 128, True) - 2.749e11) < 1e8
    assert rf.attention_flops(1, 8, 1024, 64, False) == 2 * rf.attention_flops(1, 8, 1024, 64, True)
    assert rf.attention_io_bytes(4, 16, 4096, 128, 2) == 256 * 2 ** 20


def test_roofline_ceilings():
    # below the ridge the bandwidth ceiling binds, above it the compute ceiling
    peak, bw = 1949.4e3, 6685.8  # GFLOP/s, GB/s
    ridge = rf.ridge_point(peak, bw)
    assert 291 < ridge < 292
    assert rf.attainable(ridge / 2, peak, bw) == pytest.approx(peak / 2)
    assert rf.attainable(2 * ridge, peak, bw) == peak
    assert rf.roofline_fraction(peak / 4, 2 * ridge, peak, bw) == pytest.approx(0.25)


def test_instruction_roofline_units():
    # 32 instructions = one warp instruction; 1e9 warp instructions in 1 s = 1 GIPS
    assert rf.instruction_intensity(3200, 10) == 10
    assert rf.warp_gips(32e9, 1.0) == 1.0


def test_measured_peaks_loader(tmp_path):
    p = tmp_path / "peaks.json"
    p.write_text('{"hbm_gbs": 6685.8, "bf16_tflops": 1949.4, "bf16_tflops_sustained": 1739.7}')
    peaks, src = rf.load_measured_peaks(str(p))
    assert src == "measured" and peaks["bf16_tflops"] == 1949.4
    peaks, src = rf.load_measured_peaks(str(tmp_path / "absent.json"))
    assert src == "fallback" and peaks == rf.FALLBACK_PEAKS
