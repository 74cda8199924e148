"""Host-side pieces of bench.py that run without a GPU: argument parsing of the
workload options, the reference (oracle) arm's JSON line, the kernel roofline
arithmetic and the DRAM-traffic record (ingest from an ncu CSV, lookup, stale
sources)."""
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


def test_kernel_roofline_follows_the_layer_bytes():
    """The dominant kernel's fraction is recomputable from the line: bytes are
    the kernel's share of x + y + w only (the contraction: w), the spectra in
    the workspace are reported beside them, and the contraction's flops are
    held against the path's compute peak."""
    import bench
    from fourier_neural_spectral_gb300 import synth
    cfg = synth.CONFIGS["B16_C64_128x128_m32"]
    peaks = {"hbm_gbs": 6795.5, "bf16_tflops": 1959.3, "sm_max_mhz": 2070.0}
    w = cfg.w_bytes()
    mix = {"name": "mix_wide", "bytes": w + cfg.x_bytes() // 4 + cfg.y_bytes() // 4,
           "flops": cfg.gemm_flops()}
    r = bench.kernel_roofline(mix, 0.03543, cfg, peaks, 152, "fp32")
    fma = 152 * 128 * 2 * 2070e6 / 1e12
    assert r["io_bytes_per_launch"] == w
    assert r["workspace_bytes_per_launch"] == mix["bytes"] - w
    # 67.1 MB at 6795.5 GB/s = 9.9 us; 1.07 GFLOP at 80.5 TFLOP/s = 13.3 us: FMA binds
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - cfg.gemm_flops() / 0.03543e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / fma) < 1e-12
    tc = dict(mix, name="mix_tcm_3xtf32")
    r = bench.kernel_roofline(tc, 0.012, cfg, peaks, 152, "fp32")
    assert r["bound"] == "hbm" and abs(r["frac"] - w / 0.012e-3 / 1e9 / 6795.5) < 1e-12
    assert abs(r["compute_peak_tflops"] - 1959.3 * bench.TF32_PER_BF16 / 3) < 1e-9
    fwd = {"name": "fwd_fused", "bytes": cfg.x_bytes() + 16777216, "flops": 123}
    r = bench.kernel_roofline(fwd, 0.034, cfg, peaks, 152, "fp32")
    assert r["bound"] == "hbm" and r["io_bytes_per_launch"] == cfg.x_bytes()
    assert r["flops_per_launch"] == 0  # transform arithmetic is not in the roofline
    assert bench.kernel_io_bytes("inv_fused", cfg) == cfg.y_bytes()
    assert bench.kernel_io_bytes("zero_X", cfg) == 0


def test_traffic_ingest_and_stale_sources(tmp_path):
    """An ncu CSV ingested into the traffic file gives the median bytes per
    launch; an entry whose kernel sources changed since reads as None."""
    import json
    import bench
    csv = tmp_path / "launches.csv"
    head = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    body = ""
    for i, (rd, wr) in enumerate([(100, 10), (300, 30), (200, 20)]):
        k = "void fno::(anonymous namespace)::mix_wide_kernel<16, 0>(CUtensorMap, ...)"
        body += f'"{i}","{k}","dram__bytes_read.sum","byte","{rd}"\n'
        body += f'"{i}","{k}","dram__bytes_write.sum","byte","{wr}"\n'
    body += '"9","void fno::(anonymous namespace)::fwd_fused_kernel<128, 128, 32, 32>(...)",' \
            '"dram__bytes_read.sum","Mbyte","67.1"\n'
    body += '"9","void fno::(anonymous namespace)::fwd_fused_kernel<128, 128, 32, 32>(...)",' \
            '"dram__bytes_write.sum","Kbyte","2"\n'
    csv.write_text("==PROF== noise\n" + head + body)
    out = tmp_path / "traffic.json"
    added = bench.ingest_ncu(str(csv), "W", "fp32", "ncu ...", path=str(out))
    assert {e["kernel"] for e in added} == {"mix_wide", "fwd_fused"}
    assert bench.measured_traffic("W", "mix_wide", "fp32", path=str(out)) == 220.0
    assert abs(bench.measured_traffic("W", "fwd_fused", "fp32", path=str(out)) - 67.102e6) < 1e-3
    assert bench.measured_traffic("W", "inv_fused", "fp32", path=str(out)) is None
    data = json.loads(out.read_text())
    data["captures"][0]["sources"]["common.cuh"] = "0" * 64   # the kernel changed since
    out.write_text(json.dumps(data))
    k0 = data["captures"][0]["kernel"]
    assert bench.measured_traffic("W", k0, "fp32", path=str(out)) is None


def test_kernel_patterns_pick_one_name_each():
    import re
    import bench
    demangled = {
        "mix_tcm_kernel<16, 3>": "mix_tcm_3xtf32", "mix_tcm_kernel<8, 1>": "mix_tcm_tf32",
        "mix_tc_kernel<3>": "mix_tc_3xtf32", "mix_tc_kernel<1>": "mix_tc_tf32",
        "fwd_fused_kernel<128, 128, 32, 32>": "fwd_fused", "inv_big_kernel<2048, 64, true>":
        "inv_fused", "mix_wide_kernel<16, 0>": "mix_wide", "layer_persistent_kernel<64, 16, 16>":
        "layer_persistent", "dft_rows_gemm_kernel<64, 4, true, true>": "dft_rows",
        "dft_rows_gemm_kernel<64, 2, false, false>": "dft_irows",
        "dft_frows_kernel<24>": "dft_rows", "dft_irows_kernel": "dft_irows",
        "dft_cols_gemm_kernel<true>": "dft_cols", "dft_cols_gemm_kernel<false>": "dft_icols",
        "dft_cols_gemm_kernel<1>": "dft_cols", "dft_cols_gemm_kernel<0>": "dft_icols",
        "dft_rows_gemm_kernel<32, 4, 1, 1>": "dft_rows", "dft_rows_gemm_kernel<64, 2, 0, 0>": "dft_irows",
        "block_tc_kernel<64>": "block_tc", "block_epilogue_kernel<8>": "block_fp32",
    }
    for name, want in demangled.items():
        hits = [k for k, (rx, _) in bench.KERNEL_SOURCES.items()
                if re.search(rx, "void fno::(anonymous namespace)::" + name + "(...)")]
        assert hits == [want], (name, hits)


def test_committed_traffic_file_parses():
    import json
    import bench
    data = json.load(open(bench.TRAFFIC_JSON))
    for e in data["captures"]:
        assert e["kernel"] in bench.KERNEL_SOURCES
        assert e["read_bytes"] >= 0 and e["write_bytes"] >= 0


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
