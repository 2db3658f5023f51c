"""Roofline arithmetic: peak formulas, calibration and roofline fractions.

Sources (web pages):
 - TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth" / "Output":
   calibration = best measured Triad bandwidth / theoretical bandwidth.
 - "microbench" results page (martins3.github.io, GPU section on compute
   throughput): FP32 peak = SMs x CUDA cores per SM x 2 FLOP per FMA x clock,
   and theoretical DRAM bandwidth = 2 x memory clock x bus width / 8.
 - kbench page, section "Analysis" (scripts/roofline.py): each kernel is placed
   against min(compute ceiling, intensity x bandwidth ceiling).
 - GPU-Roofline-Python page, section "Metrics Used": instruction intensity =
   (instructions / 32) / transactions and performance = (instructions / 32) /
   (1e9 x time) in warp GIPS.
"""
from __future__ import annotations

import json
import os

# FP32 lanes per SM assumed by the peak formula (the microbench page's value;
# CUDA does not expose it).
CUDA_CORES_PER_SM = 128

# Used only when the measured-peaks file is absent (one earlier GB300 measurement).
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def theoretical_dram_gbs(mem_clock_mhz: float, bus_width_bits: int) -> float:
    """2 transfers per memory clock x bus width in bytes (GB/s, 1e9 bytes)."""
    return 2.0 * mem_clock_mhz * 1e6 * bus_width_bits / 8.0 / 1e9


def fp32_peak_gflops(sms: int, clock_mhz: float, cores_per_sm: int = CUDA_CORES_PER_SM) -> float:
    """SMs x FP32 lanes per SM x 2 FLOP (one FMA) x clock."""
    return sms * cores_per_sm * 2.0 * clock_mhz * 1e6 / 1e9


# Integer multiply-add lanes per SM per clock, the roof of the Q15 kernel. That
# kernel forms each 16-bit x 16-bit product of its scores and weighted sums with
# one dp2a lane-operation (two 16 x 8-bit products on the split operands), so its
# bound is the dp2a issue rate. Measured on GB300 with independent dp2a, IMAD and
# FFMA chains in one run: dp2a and IMAD each issue 65.6 lanes per SM per clock
# where FFMA issues 128, i.e. half the FP32 lanes (64).
INT32_MAD_PER_SM = 64


def int32_mad_peak_gops(sms: int, clock_mhz: float, lanes_per_sm: int = INT32_MAD_PER_SM) -> float:
    """SMs x integer multiply-add lanes per SM x 2 operations (one multiply-add) x clock."""
    return sms * lanes_per_sm * 2.0 * clock_mhz * 1e6 / 1e9


def clock_from_throughput(gflops: float, sms: int, cores_per_sm: int = CUDA_CORES_PER_SM) -> float:
    """The same formula solved for the clock (MHz) a measured FP32 rate implies."""
    return gflops * 1e9 / (sms * cores_per_sm * 2.0) / 1e6


def calibration(measured_gbs: float, theoretical_gbs: float) -> float:
    return measured_gbs / theoretical_gbs


def attainable(intensity: float, compute_peak: float, bandwidth: float) -> float:
    """min(compute peak, intensity x bandwidth); units follow the arguments
    (e.g. FLOP/B x GB/s = GFLOP/s)."""
    return min(compute_peak, intensity * bandwidth)


def ridge_point(compute_peak: float, bandwidth: float) -> float:
    """Intensity where the two ceilings meet."""
    return compute_peak / bandwidth


def roofline_fraction(achieved: float, intensity: float, compute_peak: float, bandwidth: float) -> float:
    return achieved / attainable(intensity, compute_peak, bandwidth)


def instruction_intensity(instructions: float, transactions: float) -> float:
    """Warp-level instructions per memory transaction (hierarchical instruction roofline)."""
    return (instructions / 32.0) / transactions


def warp_gips(instructions: float, seconds: float) -> float:
    return (instructions / 32.0) / (1e9 * seconds)


def attention_flops(B: int, H: int, S: int, d: int, causal: bool) -> float:
    """4 B H S^2 d, halved for causal (QK^T and PV, 2 FLOP per MAC; the
    diagonal's extra half tile and the softmax are not counted)."""
    f = 4.0 * B * H * S * S * d
    return f / 2 if causal else f


def attention_io_bytes(B: int, H: int, S: int, d: int, elem_bytes: int) -> float:
    """Q, K, V read once and O written once."""
    return 4.0 * B * H * S * d * elem_bytes


def load_measured_peaks(path: str | None = None) -> tuple[dict, str]:
    """(peaks, source): the measured-peaks file at the repository root if
    present ("measured"), else FALLBACK_PEAKS ("fallback")."""
    if path is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            data = json.load(f)
        peaks = {k: float(data[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}
        return peaks, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"
