"""The ncu capture summary (no GPU): parsing of the raw-page CSV export, unit
scaling and the rendered table."""
import csv
import io

from roofline_benchmarking_gb300 import ncu_summary


def _csv(rows):
    buf = io.StringIO()
    csv.writer(buf, quoting=csv.QUOTE_ALL).writerows(rows)
    return buf.getvalue()


def test_raw_csv_to_table():
    hdr = ["ID", "Kernel Name", "Block Size", "Grid Size", "gpu__time_duration.sum", "dram__bytes_read.sum",
           "dram__bytes_write.sum", "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
           "sm__cycles_elapsed.avg.per_second", "smsp__inst_executed.sum",
           "smsp__average_warps_issue_stalled_wait_per_issue_active.ratio",
           "smsp__average_warps_issue_stalled_barrier_per_issue_active.ratio",
           "smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio"]
    units = ["", "", "", "", "nsecond", "Kbyte", "Mbyte", "%", "Mhz", "inst", "", "", ""]
    row = ["0", "kernel_a<0>(int)", "(384, 1, 1)", "(152, 1, 1)", "225,696", "152,665.856", "34.653184", "42.95",
           "1,913.69", "113,085,424", "1.18", "1.04", "0.90"]
    text = "==PROF== Connected to process 1\n" + _csv([hdr, units, row, ["short", "row"]])
    launches = ncu_summary.parse_raw_csv(text)
    assert len(launches) == 1
    L = launches[0]
    assert (L["kernel"], L["grid"], L["block"]) == ("kernel_a<0>(int)", "(152, 1, 1)", "(384, 1, 1)")
    v = L["values"]
    assert abs(v["gpu__time_duration.sum"] - 225.696) < 1e-9          # ns -> us
    assert abs(v["dram__bytes_read.sum"] - 152.665856) < 1e-9          # KB -> MB
    assert abs(v["dram__bytes_write.sum"] - 34.653184) < 1e-9
    assert abs(v["sm__cycles_elapsed.avg.per_second"] - 1.91369) < 1e-9  # MHz -> GHz
    assert v["sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active"] is None  # not captured
    assert L["stalls"] == {"wait": 1.18, "barrier": 1.04, "long_scoreboard": 0.90}
    md = ncu_summary.render(launches, stalls=2)
    assert "| gpu__time_duration (cold L2, serialised) | 225.7 us |" in md
    assert "| traffic (read + write) | 187.3 MB |" in md
    assert "| DRAM bytes / duration | 830 GB/s |" in md
    assert "| smsp__inst_executed.sum | 113,085,424 warp instructions |" in md
    assert "| wait | 1.18 |" in md and "| barrier | 1.04 |" in md and "long_scoreboard" not in md
    assert "pipe_alu" not in md


def test_no_launch_in_the_export():
    assert ncu_summary.parse_raw_csv("==PROF== nothing profiled\n") == []
    assert ncu_summary.parse_raw_csv(_csv([["ID", "Kernel Name"], ["", ""]])) == []
