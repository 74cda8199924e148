"""Benchmark of the FNO 2D spectral-convolution layer (libfnospec) on GB300.

One step = one call of the whole layer (forward transforms, per-mode channel
contraction, inverse transforms) over one batch of the workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--precision fp32|tf32|3xtf32] [--impl ours|reference]

Prints one JSON line on rank 0.  `--impl reference` times the double-precision
oracle (plain single-threaded C++) on the host cores instead, on a bounded
sample of the same workload.  With N > 1 (torchrun) each rank runs its own
replica of the workload on its own GPU (weak scaling, no collective on the data
path); rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from fourier_neural_spectral_gb300 import synth  # noqa: E402

METRIC = "FNO spectral-conv samples/s at 128² C=64; % of HBM/tensor roofline"
UNIT = "samples/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "sm_max_mhz": 2070.0}, "fallback"


def fp32_fma_peak_tflops(sm_mhz: float, sms: int) -> float:
    """FP32 FMA peak: SMs x 128 lanes x 2 flops x clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


# dense TF32 tensor rate relative to dense bf16 (nominal 1.1 against 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25


def device_sms(dev) -> int:
    import torch
    return int(torch.cuda.get_device_properties(dev).multi_processor_count)


def kernel_io_bytes(name: str, cfg) -> int:
    """The share of the layer's algorithmic bytes (x read, y written, w read:
    the roofline's definition) that kernel `name` moves; the rest of its bytes
    are the spectra X, Z (and T) in the plan's workspace."""
    if name.startswith(("fwd_fused", "fwd_rows", "dft_rows", "dft1_fwd", "rows1d_fwd")):
        return cfg.x_bytes()
    if name.startswith(("inv_fused", "inv_rows", "dft_irows", "dft1_inv", "rows1d_inv")):
        return cfg.y_bytes()
    if name.startswith("mix"):
        return cfg.w_bytes()
    if name.startswith("layer_persistent"):  # the whole layer in one launch
        return cfg.x_bytes() + cfg.y_bytes() + cfg.w_bytes()
    return 0


def kernel_roofline(kinfo, ms: float, cfg, peaks: dict, sms: int, precision: str):
    """Roofline of one kernel from its algorithmic bytes and flops: bytes are
    its share of x + y + w (kernel_io_bytes) at the measured HBM copy peak;
    flops (the mode contraction only; the transforms' arithmetic is secondary)
    at the FP32 FMA peak, or at the TF32 tensor peak divided by the number of
    TF32 products per fp32 product (3 for split TF32) on the tensor path.
    Whichever takes longer binds; frac = that time / the measured time."""
    hbm = float(peaks["hbm_gbs"])
    clock = float(peaks.get("sm_max_mhz", 2070.0))
    io = kernel_io_bytes(kinfo["name"], cfg)
    t = ms * 1e-3
    t_bytes = io / (hbm * 1e9)
    flops = kinfo["flops"] if kinfo["name"].startswith(("mix", "layer_persistent")) else 0
    tensor = "_tc" in kinfo["name"] or "tcgen05" in kinfo["name"]
    if tensor:
        split = 3 if "3xtf32" in kinfo["name"] else 1
        cpeak = float(peaks["bf16_tflops"]) * TF32_PER_BF16 / split
        ckind = f"tf32 tensor peak = measured bf16 x {TF32_PER_BF16:.3f} / {split}"
    else:
        cpeak = fp32_fma_peak_tflops(clock, sms)
        ckind = f"fp32 FMA peak = {sms} SMs x 128 x 2 x {clock:.0f} MHz"
    t_flops = flops / (cpeak * 1e12) if flops else 0.0
    if t_bytes >= t_flops:
        r = {"bound": "hbm", "achieved": io / t / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        r = {"bound": "tensor" if tensor else "alu", "achieved": flops / t / 1e12, "peak": cpeak,
             "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r.update({"kernel": kinfo["name"], "ms_per_launch": ms, "io_bytes_per_launch": io,
              "workspace_bytes_per_launch": kinfo["bytes"] - io,
              "flops_per_launch": flops, "t_bytes_us": t_bytes * 1e6,
              "t_flops_us": t_flops * 1e6, "compute_peak_tflops": cpeak,
              "compute_peak_kind": ckind})
    return r


# ---------------------------------------------------- measured DRAM traffic ---
# profiles/dram_traffic.json holds per-launch DRAM bytes of the kernels, one
# entry per (workload, kernel, precision), written by `--ingest-ncu` from the
# CSV of an ncu capture with dram__bytes_read.sum and dram__bytes_write.sum.
# Each entry records the SHA-256 of the source files its kernel is built from;
# a lookup whose sources have changed since returns None.

TRAFFIC_JSON = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "fourier_neural_spectral_gb300", "csrc")
# plan kernel name -> (regex on the demangled ncu kernel name, source files)
_COMMON = ["common.cuh", "internal.h"]
KERNEL_SOURCES = {
    "fwd_fused": (r"\b(fwd_fused_kernel|fwd_big_kernel)\b",
                  ["stages_fused.cu", "stages_big.cu", "fused_columns.cuh", "fft_reg.cuh",
                   "tma.cuh", "fused_rows.cuh"] + _COMMON),
    "inv_fused": (r"\b(inv_fused_kernel|inv_big_kernel)\b",
                  ["stages_fused.cu", "stages_big.cu", "fused_columns.cuh", "fft_reg.cuh",
                   "tma.cuh", "fused_rows.cuh"] + _COMMON),
    "zero_X": (r"\bzero_kernel\b", ["stages_fused.cu"] + _COMMON),
    "mix_wide": (r"\bmix_wide_kernel\b", ["mix_wide.cu", "tma.cuh"] + _COMMON),
    "mix_tma": (r"\bmix_tma_kernel\b", ["mix_tma.cu", "tma.cuh"] + _COMMON),
    "mix_tc_tf32": (r"\bmix_tc_kernel<1>", ["mix_tc.cu", "tcgen05.cuh", "tma.cuh"] + _COMMON),
    "mix_tc_3xtf32": (r"\bmix_tc_kernel<3>", ["mix_tc.cu", "tcgen05.cuh", "tma.cuh"] + _COMMON),
    "mix_tcm_3xtf32": (r"\bmix_tcm_kernel<\d+, 3>", ["mix_tcm.cu", "tcgen05.cuh", "tma.cuh"] + _COMMON),
    "mix_tcm_tf32": (r"\bmix_tcm_kernel<\d+, 1>", ["mix_tcm.cu", "tcgen05.cuh", "tma.cuh"] + _COMMON),
    "layer_persistent": (r"\blayer_persistent_kernel\b",
                         ["layer_persistent.cu", "fused_rows.cuh", "fused_columns.cuh",
                          "fft_reg.cuh", "tma.cuh"] + _COMMON),
    # ncu prints a bool template argument as 1 / 0
    "dft_rows": (r"\b(dft_rows_gemm_kernel<[0-9]+, [0-9]+, (true|1),|dft_frows_kernel<)",
                 ["stages_dft.cu", "tma.cuh"] + _COMMON),
    "dft_irows": (r"\b(dft_rows_gemm_kernel<[0-9]+, [0-9]+, (false|0),|dft_irows_kernel\b)",
                  ["stages_dft.cu", "tma.cuh"] + _COMMON),
    "dft_cols": (r"\bdft_cols_gemm_kernel<(true|1)>", ["stages_dft.cu"] + _COMMON),
    "dft_icols": (r"\bdft_cols_gemm_kernel<(false|0)>", ["stages_dft.cu"] + _COMMON),
    "block_tc": (r"\bblock_tc_kernel<", ["block_tc.cu", "tcgen05.cuh", "tma.cuh"] + _COMMON),
    "block_fp32": (r"\bblock_epilogue_kernel<", ["block.cu", "tma.cuh"] + _COMMON),
}


def source_hashes(kernel: str) -> dict:
    import hashlib
    files = KERNEL_SOURCES.get(kernel, (None, sorted(os.listdir(CSRC))))[1]
    out = {}
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            out[f] = hashlib.sha256(fh.read()).hexdigest()
    return out


def measured_traffic(workload: str, kernel: str, precision: str, path: str = TRAFFIC_JSON):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    ingested ncu captures, or None if never captured or if its sources changed
    since the capture."""
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    for e in data.get("captures", []):
        if (e["workload"], e["kernel"], e["precision"]) == (workload, kernel, precision):
            try:
                if source_hashes(kernel) != e["sources"]:
                    return None
            except OSError:
                return None
            return float(e["read_bytes"]) + float(e["write_bytes"])
    return None


def ingest_ncu(csv_path: str, workload: str, precision: str, command: str,
               path: str = TRAFFIC_JSON) -> list:
    """Read an ncu --csv capture (one row per launch and metric: columns
    "Kernel Name", "Metric Name", "Metric Value") and record the median DRAM
    read and write bytes per launch of every known kernel in it."""
    import csv
    import re
    rows = {}
    with open(csv_path, newline="") as f:
        lines = [l for l in f if l.startswith('"')]  # skip ncu's ==PROF== lines
    for r in csv.DictReader(lines):
        name, metric = r.get("Kernel Name", ""), r.get("Metric Name", "")
        if metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        unit = (r.get("Metric Unit") or "byte").lower()
        scale = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9}.get(unit, 1)
        val = float(str(r["Metric Value"]).replace(",", "")) * scale
        for k, (rx, _) in KERNEL_SOURCES.items():
            if re.search(rx, name):
                rows.setdefault(k, {}).setdefault(metric, []).append(val)
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    caps = [e for e in data.get("captures", [])
            if not (e["workload"] == workload and e["precision"] == precision and e["kernel"] in rows)]
    added = []
    for k, m in sorted(rows.items()):
        rd, wr = m.get("dram__bytes_read.sum", []), m.get("dram__bytes_write.sum", [])
        if not rd or not wr:
            continue
        e = {"workload": workload, "kernel": k, "precision": precision,
             "read_bytes": statistics.median(rd), "write_bytes": statistics.median(wr),
             "launches": len(rd), "command": command, "sources": source_hashes(k)}
        caps.append(e)
        added.append(e)
    data = {"about": "DRAM bytes per launch (ncu dram__bytes_read.sum / dram__bytes_write.sum, "
                     "median over the captured launches), written by bench.py --ingest-ncu",
            "captures": sorted(caps, key=lambda e: (e["workload"], e["kernel"], e["precision"]))}
    with open(path, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")
    return added


# ----------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ NVTX ---

class nvtx_range:
    """An NVTX range around a region of the bench (seen by Nsight tools; a no-op
    cost otherwise)."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        import torch
        torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        import torch
        torch.cuda.nvtx.range_pop()
        return False


# ------------------------------------------------------------ distributed ---

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_value(world: int, batch: int, steps: int, elapsed_ms_max: float) -> float:
    """Whole-job samples/s: every rank runs its own replica of the workload
    (weak scaling), timed by the slowest rank."""
    return world * batch * steps / (elapsed_ms_max / 1e3)


# ---------------------------------------------------------- oracle (host) ---

def oracle_sample_batch(cfg, budget: float = 2.5e9) -> int:
    """Batch rows per oracle sample, bounded by `budget` multiply-adds
    (2.5e9 is roughly 5-15 s of single-threaded host work)."""
    per_sample = cfg.Cin * (cfg.H * cfg.W * cfg.m2 + 2 * cfg.m1 * cfg.H * cfg.m2) \
        + cfg.Cout * (cfg.H * cfg.W * cfg.m2 + 2 * cfg.m1 * cfg.H * cfg.m2) \
        + cfg.Cin * cfg.Cout * cfg.nmodes
    return max(1, min(cfg.B, int(budget // per_sample)))


def time_oracle(cfg, reps: int = 1):
    """Time the oracle, single-threaded, on a bounded sample of the workload
    (the first `nb` batch rows).  Returns (samples/s, sample description)."""
    import oracle
    oracle.build()
    nb = oracle_sample_batch(cfg)
    x, w = synth.make_inputs(cfg)
    xs = np.ascontiguousarray(x[:nb].astype(np.float64))
    wc = w.astype(np.float64).view(np.complex128)[..., 0]
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.spectral_conv2d(xs, wc, cfg.m1, cfg.m2)
    dt = (time.perf_counter() - t0) / reps
    return nb / dt, dt, f"oracle on {nb} of {cfg.B} batch rows ({cfg.name}), {dt:.2f} s per call"


def run_reference(args, cfg):
    rank, world, _ = dist_info()
    if rank != 0:
        return  # the oracle arm runs on rank 0 only; other ranks exit without work
    import oracle
    oracle.build()
    nb = oracle_sample_batch(cfg, budget=3e8)  # about 1-2 s of host work per step
    x, w = synth.make_inputs(cfg)
    xs = np.ascontiguousarray(x[:nb].astype(np.float64))
    wc = w.astype(np.float64).view(np.complex128)[..., 0]
    for _ in range(args.warmup):
        oracle.spectral_conv2d(xs[:1], wc, cfg.m1, cfg.m2)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.spectral_conv2d(xs, wc, cfg.m1, cfg.m2)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = nb * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, "f64-oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{nb} of {cfg.B} batch rows per step",
                         "host": platform.machine(), "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_dict(cfg, precision):
    return {"workload": cfg.name, "B": cfg.B, "Cin": cfg.Cin, "Cout": cfg.Cout, "H": cfg.H,
            "W": cfg.W, "m1": cfg.m1, "m2": cfg.m2, "precision": precision,
            "global_batch": cfg.B, "x": "N(0,1)" if not cfg.smooth else "smooth-ish",
            "w": "re,im ~ U[0,1)/(Cin*Cout)", "seed": 0}


# ------------------------------------------------------------- ours (GPU) ---

def run_ours(args, cfg):
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__ as g
    g.build()
    from fourier_neural_spectral_gb300 import fnospec

    peaks, peak_kind = read_peaks()
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2, args.precision)
    if args.single_launch != "auto":
        plan.fno_plan_set_single_launch(args.single_launch == "on")
    step_bytes = cfg.algorithmic_bytes()
    # rotate over enough distinct (x, w, y) sets that no buffer is still in L2
    # when it is used again (every step touches a different set)
    nsets = max(1, min(8, -(-3 * L2_BYTES // step_bytes) + 1)) if step_bytes < 3 * L2_BYTES else 1
    x0, w0 = synth.make_inputs(cfg)
    xs = [torch.from_numpy(x0).to(dev)]
    ws = [torch.from_numpy(w0).to(dev)]
    for k in range(1, nsets):
        xs.append(torch.roll(xs[0], shifts=k, dims=0).contiguous())
        ws.append((ws[0] * (1.0 + 0.01 * k)).contiguous())
    ys = [torch.empty((cfg.B, cfg.Cout, cfg.H, cfg.W), dtype=torch.float32, device=dev)
          for _ in range(nsets)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        j = i % nsets
        plan.fno_plan_execute(xs[j], ws[j], ys[j], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after warm-up")

    # The timed steps run back to back with no event between their kernels
    # (an event recorded between two kernels keeps the second from starting in
    # the first one's tail); the per-kernel breakdown and the latency
    # percentiles come from separate steps with per-kernel events armed.
    nk = plan.launches
    nbreak = max(3, min(args.steps, 20))
    evsets = []
    for _ in range(nbreak):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        for e in evs:
            e.record(stream)  # materialise the CUDA events
        evsets.append(evs)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with nvtx_range(f"timed steps: {cfg.name}"):
        t_start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    status = plan.fno_get_device_status()
    if status != fnospec.FNO_OK:
        raise RuntimeError(f"device status {status} after timed steps")
    with nvtx_range("per-kernel breakdown steps"):
        for i in range(nbreak):
            plan.fno_plan_record_events(evsets[i])
            step(args.warmup + args.steps + i)
        plan.fno_plan_record_events(None)
        torch.cuda.synchronize(dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after the breakdown steps")

    per_step = [evs[0].elapsed_time(evs[-1]) for evs in evsets]
    per_kernel = [[evs[k].elapsed_time(evs[k + 1]) for evs in evsets] for k in range(nk)]
    ms_per_step = elapsed_ms / args.steps
    value = aggregate_value(world, cfg.B, args.steps, elapsed_ms)

    # dominant kernel and its roofline (the kernel with the largest mean time)
    kmean = [statistics.mean(v) for v in per_kernel]
    kdom = int(np.argmax(kmean))
    kinfo = plan.kernels[kdom]
    hbm = float(peaks["hbm_gbs"])
    sms = device_sms(dev)
    roofline = kernel_roofline(kinfo, kmean[kdom], cfg, peaks, sms, args.precision)
    roofline["traffic"] = measured_traffic(cfg.name, kinfo["name"], args.precision)
    roofline["peak_kind"] = (f"{peak_kind} (hbm_gbs, STREAM-style copy)"
                             if roofline["bound"] == "hbm" else roofline["compute_peak_kind"])
    # the layer roofline: slower of (x + y + w bytes at HBM peak) and the mode
    # contraction flops at the compute peak of the path
    fp32_peak = fp32_fma_peak_tflops(float(peaks.get("sm_max_mhz", 2070.0)), sms)
    t_hbm = step_bytes / (hbm * 1e9)
    t_gemm = cfg.gemm_flops() / (fp32_peak * 1e12)
    t_roof = max(t_hbm, t_gemm)
    step_s = ms_per_step * 1e-3
    layer = {"bound": "hbm" if t_hbm >= t_gemm else "fp32-fma",
             "bytes_per_step": step_bytes, "gemm_flops_per_step": cfg.gemm_flops(),
             "t_roof_us": t_roof * 1e6, "t_step_us": step_s * 1e6,
             "frac": t_roof / step_s, "achieved_gbs": step_bytes / step_s / 1e9,
             "peak_gbs": hbm, "fp32_peak_tflops_at_max_clock": fp32_peak}

    kernels = [{"name": plan.kernels[k]["name"], "ms": kmean[k],
                "share": kmean[k] / sum(kmean),
                "gbs": plan.kernels[k]["bytes"] / (kmean[k] * 1e-3) / 1e9}
               for k in range(nk)]

    # end to end through the public calls: every step copies its x from pinned
    # host memory, runs fno_plan_execute and copies its y back to pinned host
    # memory.  Serialised on one stream first; then pipelined, with the copies
    # on two copy streams and two device buffer sets, so that the copies of one
    # step overlap the layer of its neighbours (event dependencies keep every
    # buffer from being rewritten before its last reader is done).
    xh = torch.from_numpy(x0).pin_memory()
    yh = [torch.empty((cfg.B, cfg.Cout, cfg.H, cfg.W), dtype=torch.float32).pin_memory()
          for _ in range(2)]
    xd = [torch.empty_like(xs[0]) for _ in range(2)]
    yd = [torch.empty_like(ys[0]) for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        xd[0].copy_(xh, non_blocking=True)
        plan.fno_plan_execute(xd[0], ws[0], yd[0], stream=stream)
        yh[0].copy_(yd[0], non_blocking=True)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    with nvtx_range("end to end, serialised"):
        e0.record(stream)
        for _ in range(e2e_steps):
            xd[0].copy_(xh, non_blocking=True)
            plan.fno_plan_execute(xd[0], ws[0], yd[0], stream=stream)
            yh[0].copy_(yd[0], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    serial_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    serial_value = aggregate_value(world, cfg.B, e2e_steps, serial_ms)

    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):
        for e in (ev_in[b], ev_done[b], ev_out[b]):
            e.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    nvtx_e2e = nvtx_range("end to end, pipelined copies")
    nvtx_e2e.__enter__()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e2e_steps):
        b = i % 2
        s_in.wait_event(ev_done[b])           # the layer two steps back has read xd[b]
        with torch.cuda.stream(s_in):
            xd[b].copy_(xh, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])          # yd[b] was copied out two steps back
        plan.fno_plan_execute(xd[b], ws[0], yd[b], stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            yh[b].copy_(yd[b], non_blocking=True)
        ev_out[b].record(s_out)
    stream.wait_event(ev_out[(e2e_steps - 1) % 2])
    stream.wait_event(ev_out[e2e_steps % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    nvtx_e2e.__exit__(None, None, None)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after the end-to-end steps")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = aggregate_value(world, cfg.B, e2e_steps, e2e_ms)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, sample = time_oracle(cfg)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
               "host": platform.machine(), "host_cores": os.cpu_count()}

    if rank == 0:
        pct = np.percentile(per_step, [10, 50, 90]).tolist()
        dtype = {"fp32": "f32", "tf32": "f32 (tf32 mode contraction)",
                 "3xtf32": "f32 (3xtf32 mode contraction)"}[args.precision]
        l2 = (f"inputs rotate over {nsets} buffer sets ({nsets * step_bytes / 1e6:.0f} MB) > L2"
              if nsets > 1 else f"one step moves {step_bytes / 1e6:.0f} MB > L2")
        if nsets * step_bytes < 2 * L2_BYTES:
            l2 = f"working set {nsets * step_bytes / 1e6:.1f} MB is L2-resident (small case)"
        cfgd = config_dict(cfg, args.precision)
        cfgd["l2"] = l2
        cfgd["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "latency_ms": {"p10": pct[0], "p50": pct[1], "p90": pct[2]},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype, "data": "synthetic (seeded SplitMix64 inputs, random weights)",
            "config": cfgd, "roofline": roofline, "layer_roofline": layer,
            "kernels": kernels, "kernel_breakdown_steps": nbreak, "plan": plan.description,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": cfg.x_bytes(),
                    "d2h_bytes_per_step": cfg.y_bytes(), "steps": e2e_steps,
                    "serialised_value": serial_value,
                    "note": "every step copies its x from pinned host memory and its y back to "
                            "pinned host memory around fno_plan_execute; value: copies on two "
                            "copy streams overlapping the neighbouring steps' layer (two device "
                            "buffer sets); serialised_value: one stream, no overlap; w resident"},
            "gpu_launches": nk * args.steps,
            "clocks": clk,
            "context": "fused-operator page quotes 42 ms -> 11.3 ms per 128x128 FNO step "
                       "on A100 (whole model, not this layer)",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours_block(args, cfg):
    """Time fno_block_execute (spectral layer + pointwise branch + bias + GELU)
    on the workload; one JSON line.  Algorithmic bytes: x read, y written, w and
    w_pw read; flops: the mode contraction plus the pointwise branch
    (2*B*Cin*Cout*H*W); roofline = max(bytes / HBM peak, flops / FP32 peak)."""
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    from fourier_neural_spectral_gb300 import fnospec

    peaks, peak_kind = read_peaks()
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
    step_bytes = cfg.algorithmic_bytes() + 4 * cfg.Cin * cfg.Cout
    nsets = max(1, min(8, -(-3 * L2_BYTES // step_bytes) + 1)) if step_bytes < 3 * L2_BYTES else 1
    x0, w0 = synth.make_inputs(cfg)
    xs = [torch.from_numpy(x0).to(dev)]
    for k in range(1, nsets):
        xs.append(torch.roll(xs[0], shifts=k, dims=0).contiguous())
    wt = torch.from_numpy(w0).to(dev)
    gen = torch.Generator(device=dev).manual_seed(0)
    wpw = torch.randn((cfg.Cout, cfg.Cin), device=dev, generator=gen) / cfg.Cin ** 0.5
    bias = torch.randn((cfg.Cout,), device=dev, generator=gen)
    ys = [torch.empty((cfg.B, cfg.Cout, cfg.H, cfg.W), dtype=torch.float32, device=dev)
          for _ in range(nsets)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        j = i % nsets
        plan.fno_block_execute(xs[j], wt, wpw, bias, ys[j], "gelu", stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after warm-up")
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after timed steps")
    ms_per_step = elapsed_ms / args.steps
    hbm = float(peaks["hbm_gbs"])
    flops = cfg.gemm_flops() + 2 * cfg.B * cfg.Cin * cfg.Cout * cfg.H * cfg.W
    fp32_peak = fp32_fma_peak_tflops(float(peaks.get("sm_max_mhz", 2070.0)), device_sms(dev))
    t_roof = max(step_bytes / (hbm * 1e9), flops / (fp32_peak * 1e12))
    if rank == 0:
        cfgd = config_dict(cfg, "fp32")
        cfgd["pass"] = "FNO block: gelu(layer(x, w) + w_pw x + bias)"
        line = {
            "metric": "FNO block samples/s", "value":
                aggregate_value(world, cfg.B, args.steps, elapsed_ms),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfgd,
            "layer_roofline": {"bytes_per_step": step_bytes, "flops_per_step": flops,
                               "t_roof_us": t_roof * 1e6, "t_step_us": ms_per_step * 1e3,
                               "frac": t_roof / (ms_per_step * 1e-3), "peak_gbs": hbm,
                               "fp32_peak_tflops_at_max_clock": fp32_peak,
                               "peak_kind": peak_kind},
            "plan": plan.description, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours_backward(args, cfg):
    """Time fno_plan_backward (both gradients) on the workload; one JSON line.

    Algorithmic bytes per step: x and gy read, w read (adjoint contraction),
    gx and gw written.  Flops: the adjoint contraction and the weight gradient,
    8*B*Cin*Cout*nm each."""
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import __graft_entry__ as g
    g.build()
    from fourier_neural_spectral_gb300 import fnospec

    peaks, peak_kind = read_peaks()
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
    step_bytes = 2 * cfg.x_bytes() + cfg.y_bytes() + 2 * cfg.w_bytes()
    nsets = max(1, min(8, -(-3 * L2_BYTES // step_bytes) + 1)) if step_bytes < 3 * L2_BYTES else 1
    x0, w0 = synth.make_inputs(cfg)
    xs = [torch.from_numpy(x0).to(dev)]
    for k in range(1, nsets):
        xs.append(torch.roll(xs[0], shifts=k, dims=0).contiguous())
    wt = torch.from_numpy(w0).to(dev)
    gen = torch.Generator(device=dev).manual_seed(0)
    gys = [torch.randn((cfg.B, cfg.Cout, cfg.H, cfg.W), device=dev, generator=gen)
           for _ in range(nsets)]  # dL/dy: seeded N(0,1)
    gxs = [torch.empty_like(xs[0]) for _ in range(nsets)]
    gws = [torch.empty_like(wt) for _ in range(nsets)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        j = i % nsets
        plan.fno_plan_backward(xs[j], wt, gys[j], gxs[j], gws[j], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after warm-up")
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after timed steps")
    ms_per_step = elapsed_ms / args.steps
    hbm = float(peaks["hbm_gbs"])
    t_roof = step_bytes / (hbm * 1e9)
    if rank == 0:
        cfgd = config_dict(cfg, "fp32")
        cfgd["pass"] = "backward (dL/dx and dL/dw)"
        line = {
            "metric": "FNO spectral-conv backward samples/s", "value":
                aggregate_value(world, cfg.B, args.steps, elapsed_ms),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfgd,
            "layer_roofline": {"bound": "hbm", "bytes_per_step": step_bytes,
                               "t_roof_us": t_roof * 1e6, "t_step_us": ms_per_step * 1e3,
                               "frac": t_roof / (ms_per_step * 1e-3), "peak_gbs": hbm,
                               "peak_kind": peak_kind},
            "plan": plan.description, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours_1d(args):
    """The 1D layer (fno_plan_create_1d) on x [B, Cin, L]: forward steps timed
    like the 2D headline (inputs rotated past L2, CUDA events on the stream,
    per-kernel breakdown from separate event-armed steps), the oracle's 1D
    layer timed on the host as the CPU baseline."""
    import torch
    import __graft_entry__ as g
    g.build()
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, L, m = args.shape1d
    name = f"1D_B{B}_C{Cin}x{Cout}_L{L}_m{m}"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = read_peaks()
    hbm = float(peaks["hbm_gbs"])
    plan = fnospec.Plan1d(B, Cin, Cout, L, m, args.precision)
    step_bytes = 4 * B * Cin * L + 4 * B * Cout * L + 8 * Cin * Cout * m
    nsets = max(1, min(8, -(-3 * L2_BYTES // step_bytes) + 1)) if step_bytes < 3 * L2_BYTES else 1
    x0 = synth.normal_f32((B, Cin, L), seed=0, stream=1)
    w0 = synth.uniform_f32((Cin, Cout, m, 2), scale=1.0 / (Cin * Cout), seed=0, stream=2)
    xs = [torch.from_numpy(x0).to(dev)]
    ws = [torch.from_numpy(w0).to(dev)]
    for k in range(1, nsets):
        xs.append(torch.roll(xs[0], shifts=k, dims=0).contiguous())
        ws.append((ws[0] * (1.0 + 0.01 * k)).contiguous())
    ys = [torch.empty((B, Cout, L), dtype=torch.float32, device=dev) for _ in range(nsets)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        j = i % nsets
        plan.fno_plan_execute(xs[j], ws[j], ys[j], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    nk = plan.launches
    nbreak = max(3, min(args.steps, 20))
    evsets = []
    for _ in range(nbreak):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        for e in evs:
            e.record(stream)
        evsets.append(evs)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    for i in range(nbreak):
        plan.fno_plan_record_events(evsets[i])
        step(args.warmup + args.steps + i)
    plan.fno_plan_record_events(None)
    torch.cuda.synchronize(dev)
    if plan.fno_get_device_status() != fnospec.FNO_OK:
        raise RuntimeError("device status not clean after the 1D steps")
    ms_per_step = elapsed_ms / args.steps
    kmean = [statistics.mean(evs[k].elapsed_time(evs[k + 1]) for evs in evsets)
             for k in range(nk)]
    kernels = [{"name": plan.kernels[k]["name"], "ms": kmean[k],
                "gbs": plan.kernels[k]["bytes"] / (kmean[k] * 1e-3) / 1e9,
                "tflops": plan.kernels[k]["flops"] / (kmean[k] * 1e-3) / 1e12}
               for k in range(nk)]
    kdom = int(np.argmax(kmean))
    fp32_peak = fp32_fma_peak_tflops(float(peaks.get("sm_max_mhz", 2070.0)), device_sms(dev))
    gemm = 8 * B * Cin * Cout * m
    t_hbm = step_bytes / (hbm * 1e9)
    t_roof = max(t_hbm, gemm / (fp32_peak * 1e12))
    # the direct-DFT transforms' own flops (8 per retained bin and input point
    # forward, 4 per kept bin and output point inverse) at the fp32 peak
    dft_flops = 8 * B * Cin * L * m + 4 * B * Cout * L * m
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        nb = max(1, min(B, int(2.5e9 // ((Cin + Cout) * L * m + Cin * Cout * m))))
        t = time.perf_counter()
        oracle.spectral_conv1d(x0[:nb].astype(np.float64),
                               w0.astype(np.float64).view(np.complex128)[..., 0], m)
        dt = time.perf_counter() - t
        cpu = {"value": nb / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"oracle 1D layer (numpy direct sums) on {nb} of {B} batch rows",
               "host": platform.machine(), "host_cores": os.cpu_count()}
    line = {
        "metric": "FNO 1D spectral-conv samples/s; % of HBM roofline", "value":
        B * args.steps / (elapsed_ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "B": B, "Cin": Cin, "Cout": Cout, "L": L, "m": m,
                   "precision": args.precision, "l2": f"inputs rotate over {nsets} buffer sets"},
        "roofline": {"kernel": kernels[kdom]["name"], "bound": "hbm",
                     "achieved": kernels[kdom]["gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": kernels[kdom]["gbs"] / hbm, "traffic": None,
                     "peak_kind": f"{peak_kind} (hbm_gbs)"},
        "layer_roofline": {"bytes_per_step": step_bytes, "t_roof_us": t_roof * 1e6,
                           "t_step_us": ms_per_step * 1e3, "frac": t_roof / (ms_per_step * 1e-3),
                           "dft_flops_per_step": dft_flops,
                           "dft_t_at_fp32_peak_us": dft_flops / (fp32_peak * 1e12) * 1e6},
        "kernels": kernels, "plan": plan.description, "cpu_baseline": cpu,
        "gpu_launches": nk * args.steps, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def parse_ints(text: str, n: int):
    vals = [int(v) for v in text.split(",")]
    if len(vals) != n:
        raise SystemExit(f"expected {n} comma-separated integers, got {text!r}")
    return vals


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=synth.HEADLINE, choices=synth.CONFIG_ORDER)
    ap.add_argument("--precision", default="fp32", choices=["fp32", "tf32", "3xtf32"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", default="forward",
                    choices=["forward", "backward", "block", "layer1d"],
                    help="forward (the headline), the layer's backward, one FNO block "
                         "(layer + pointwise branch + bias + GELU), or the 1D layer")
    ap.add_argument("--shape", default=None,
                    help="B,Cin,Cout,H,W,m1,m2: a workload other than the named configs "
                         "(any H, W in [2, 4096]); x ~ N(0,1), w ~ U[0,1)/(Cin*Cout)")
    ap.add_argument("--shape1d", default="64,64,64,4096,64",
                    help="B,Cin,Cout,L,m of the 1D layer (--pass layer1d)")
    ap.add_argument("--single-launch", default="auto", choices=["auto", "on", "off"],
                    help="run the layer as one cooperative launch (on), as three launches "
                         "(off), or as the plan chooses (auto)")
    ap.add_argument("--ingest-ncu", metavar="CSV", default=None,
                    help="record the DRAM bytes per launch of an ncu --csv capture of this "
                         "workload (metrics dram__bytes_read.sum, dram__bytes_write.sum) in "
                         "profiles/dram_traffic.json and exit (no GPU needed)")
    ap.add_argument("--ncu-command", default="",
                    help="the command line of that capture, stored with each entry")
    args = ap.parse_args()
    if args.ingest_ncu:
        if args.shape:
            B, Cin, Cout, H, W, m1, m2 = parse_ints(args.shape, 7)
            name = synth.LayerConfig(f"B{B}_C{Cin}x{Cout}_{H}x{W}_m{m1}x{m2}", B, Cin, Cout, H,
                                     W, m1, m2).name
        else:
            name = args.config
        for e in ingest_ncu(args.ingest_ncu, name, args.precision, args.ncu_command):
            print(f"{e['workload']} {e['kernel']} {e['precision']}: read {e['read_bytes']:.0f} "
                  f"write {e['write_bytes']:.0f} bytes per launch ({e['launches']} launches)")
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.pass_ == "layer1d":
        args.shape1d = parse_ints(args.shape1d, 5)
        run_ours_1d(args)
        return
    if args.shape:
        B, Cin, Cout, H, W, m1, m2 = parse_ints(args.shape, 7)
        cfg = synth.LayerConfig(f"B{B}_C{Cin}x{Cout}_{H}x{W}_m{m1}x{m2}", B, Cin, Cout, H, W,
                                m1, m2)
    else:
        cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.pass_ == "backward":
        run_ours_backward(args, cfg)
    elif args.pass_ == "block":
        run_ours_block(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
