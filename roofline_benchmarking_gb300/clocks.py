"""SM clocks and throttle reasons sampled with nvidia-smi while a region runs.

Clocks are never set or reset here: they are only read, so that every number
can be reported next to the clock it was measured at.
"""
from __future__ import annotations

import os
import statistics
import subprocess
import threading
import time

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampled every 100 ms in a background process; each line is
    stamped with the host time it was read."""

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:  # the timed region was shorter than one sampling period
            inside = [s for t, s in self.samples if t0 - 0.3 <= t <= t1 + 0.3]
            window = "timed region +- 0.3 s"
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(inside), "window": window}
        sm, smax, power = [], [], []
        reasons = set()
        for s in inside:
            try:
                sm.append(float(s[1]))
                smax.append(float(s[2]))
                power.append(float(s[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(REASON_NAMES, s[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if sm:
            out["sm_mhz"] = statistics.median(sm)
            out["sm_max_mhz"] = max(smax)
            out["power_w_max"] = max(power)
            out["power_w_median"] = statistics.median(power)
        out["reasons"] = sorted(reasons)
        return out


def gpu_id_for_smi(device: int) -> str:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        return ids[device] if device < len(ids) else str(device)
