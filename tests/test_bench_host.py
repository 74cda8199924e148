"""Host-side pieces of bench.py that run without a GPU: argument parsing of the
workload options, the reference (oracle) arm's JSON line, and the DRAM-traffic
table lookup."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parse_ints():
    import bench
    assert bench.parse_ints("16,64,64,421,421,12,12", 7) == [16, 64, 64, 421, 421, 12, 12]
    with pytest.raises(SystemExit):
        bench.parse_ints("1,2,3", 5)


def test_measured_traffic_reads_the_table():
    import bench
    # every row of the table parses; a kernel never captured gives None
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    rows = [l for l in open(path) if l.startswith("| B")]
    assert rows
    for line in rows:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        t = bench.measured_traffic(cells[0], cells[1], cells[2])
        assert t == float(cells[3]) + float(cells[4])
    assert bench.measured_traffic("B16_C64_128x128_m32", "no_such_kernel", "fp32") is None


def test_reference_arm_prints_one_json_line():
    # the oracle arm runs on the host; a custom small shape keeps it to seconds
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "3", "--shape", "2,4,4,16,16,4,4"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "samples/s"
    assert d["config"]["workload"] == "B2_C4x4_16x16_m4x4"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
