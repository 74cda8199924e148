"""The range-checked build (libfnospec_debug.so, FNO_DEBUG): every global store
of the kernels on the execute, stage, backward, single-launch and no-alloc paths
is checked against its launch's output ranges.

Run in a child process with FNO_DEBUG_BOUNDS=1 (the loader then picks the debug
library), so that the release library of this process is never mixed with it.
First, one layer through every kernel family must match the oracle with a clean
device status (no false alarms); then the test hook that shortens each launch's
first output range must be caught: FNO_ERR_DEVICE from fno_get_device_status,
the stores past the shortened range skipped (the output's sentinel survives),
and a clean run once the hook is cleared."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["FNO_ROOT"]); sys.path.insert(0, os.path.join(os.environ["FNO_ROOT"], "tests"))
import numpy as np, torch
import oracle
from fourier_neural_spectral_gb300 import fnospec
from gpu_helpers import errors, f32pairs_to_cplx, rand_layer_inputs, to_dev
assert fnospec.LIB_PATH.endswith("libfnospec_debug.so"), fnospec.LIB_PATH
out = {}
rng = np.random.default_rng(3)

def layer(shape, precision="fp32", single=False):
    B, Cin, Cout, H, W, m1, m2 = shape
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = fnospec.Plan(*shape, precision)
    if single:
        plan.fno_plan_set_single_launch(True)
    y = torch.full((B, Cout, H, W), float("nan"), device="cuda")
    plan.fno_plan_execute(to_dev(x), to_dev(w), y)
    torch.cuda.synchronize()
    st = plan.fno_get_device_status()
    rel, mx = errors(y.cpu().numpy(), oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2))
    return {"status": st, "rel": rel, "max": mx, "plan": plan.description}

out["fused_short"] = layer((2, 16, 16, 128, 128, 32, 32))
out["fused_long_groups"] = layer((1, 4, 4, 512, 512, 16, 16))
out["generic_fft"] = layer((2, 4, 4, 16, 16, 4, 4))
out["direct_dft"] = layer((2, 3, 5, 24, 20, 5, 7))
# the direct-DFT pass kernels: rows of 307 points (every row alignment) and,
# with 39,040 rows, the residue-class forward rows
out["direct_dft_passes"] = layer((4, 32, 2, 305, 307, 6, 3))
out["tensor_memory_3xtf32"] = layer((4, 32, 32, 64, 64, 16, 16), "3xtf32")
out["single_launch"] = layer((2, 8, 8, 64, 64, 16, 16), single=True)

# the FNO block with the tensor-core pointwise branch (its stores are TMA stores,
# not range-checked; in this build its shared-memory layout differs)
shape = B, Cin, Cout, H, W, m1, m2 = (2, 32, 32, 64, 64, 16, 16)
x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
wpw = (rng.standard_normal((Cout, Cin)) / Cin).astype(np.float32)
bias = rng.standard_normal(Cout).astype(np.float32)
plan = fnospec.Plan(*shape)
y = torch.empty((B, Cout, H, W), device="cuda")
plan.fno_block_execute(to_dev(x), to_dev(w), to_dev(wpw), to_dev(bias), y)
torch.cuda.synchronize()
rel, mx = errors(y.cpu().numpy(), oracle.block(x, f32pairs_to_cplx(w), wpw, bias, m1, m2))
out["block_tc"] = {"status": plan.fno_get_device_status(), "rel": rel, "max": mx, "plan": "block"}

# the 1D layer (pruned FFT rows and direct DFTs)
for name, (B, C, L, m) in {"rows1d_fft": (2, 4, 1024, 16), "rows1d_dft": (2, 4, 100, 9)}.items():
    x = rng.standard_normal((B, C, L)).astype(np.float32)
    w = (rng.random((C, C, m, 2)) / (C * C)).astype(np.float32)
    plan = fnospec.Plan1d(B, C, C, L, m)
    y = torch.empty((B, C, L), device="cuda")
    plan.fno_plan_execute(to_dev(x), to_dev(w), y)
    torch.cuda.synchronize()
    rel, mx = errors(y.cpu().numpy(), oracle.spectral_conv1d(x, f32pairs_to_cplx(w), m))
    out[name] = {"status": plan.fno_get_device_status(), "rel": rel, "max": mx, "plan": plan.description}

# the backward (adjoint contraction and weight gradient)
shape = B, Cin, Cout, H, W, m1, m2 = (2, 32, 32, 64, 64, 16, 16)
x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
g = rng.standard_normal((B, Cout, H, W)).astype(np.float32)
plan = fnospec.Plan(*shape)
gx, gw = torch.empty((B, Cin, H, W), device="cuda"), torch.empty((Cin, Cout, 2 * m1, m2, 2), device="cuda")
plan.fno_plan_backward(to_dev(x), to_dev(w), to_dev(g), gx, gw)
torch.cuda.synchronize()
rgx, rgw = oracle.spectral_conv2d_backward(x, f32pairs_to_cplx(w), g, m1, m2)
out["backward"] = {"status": plan.fno_get_device_status(),
                   "rel": max(errors(gx.cpu().numpy(), rgx)[0], errors(f32pairs_to_cplx(gw.cpu().numpy()), rgw)[0]),
                   "max": 0.0, "plan": plan.description}

# the allocation-free entry point
lib = fnospec.load_library()
shape = B, Cin, Cout, H, W, m1, m2 = (2, 4, 4, 32, 32, 8, 8)
x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
y = torch.empty((B, Cout, H, W), device="cuda")
xt, wt = to_dev(x), to_dev(w)  # alive until the kernels have run (raw addresses below)
rc = lib.fno_spectral_conv2d_noalloc(xt.data_ptr(), wt.data_ptr(), y.data_ptr(), *shape,
                                     torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
rel, mx = errors(y.cpu().numpy(), oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2))
out["noalloc"] = {"status": rc, "rel": rel, "max": mx, "plan": "noalloc"}

# the test hook: every launch's first output range 8 bytes short
shape = B, Cin, Cout, H, W, m1, m2 = (2, 8, 8, 64, 64, 16, 16)
x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
plan = fnospec.Plan(*shape)
assert lib.fno_plan_debug_bounds_margin(plan.handle, 8) == fnospec.FNO_OK
y = torch.full((B, Cout, H, W), float("nan"), device="cuda")
plan.fno_plan_execute(to_dev(x), to_dev(w), y)
torch.cuda.synchronize()
tail = y.flatten()[-2:].cpu().numpy().tolist()
out["margin"] = {"status": plan.fno_get_device_status(), "tail_nan": [v != v for v in tail]}
assert lib.fno_plan_debug_bounds_margin(plan.handle, 0) == fnospec.FNO_OK
plan.fno_plan_execute(to_dev(x), to_dev(w), y)
torch.cuda.synchronize()
rel, mx = errors(y.cpu().numpy(), oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2))
out["margin_cleared"] = {"status": plan.fno_get_device_status(), "rel": rel, "max": mx}
print("RESULT " + json.dumps(out))
"""


def test_range_checked_build(cuda_lib):
    from fourier_neural_spectral_gb300 import build, fnospec
    build.build(debug=True)
    env = dict(os.environ, FNO_DEBUG_BOUNDS="1", FNO_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    for name, d in res.items():
        if name in ("margin",):
            continue
        assert d["status"] == fnospec.FNO_OK, (name, d)
        assert d["rel"] <= 1e-5 and d["max"] <= 1e-4, (name, d)
    assert res["margin"]["status"] == fnospec.FNO_ERR_DEVICE, res["margin"]
    assert all(res["margin"]["tail_nan"]), res["margin"]


def test_release_build_has_no_checks(cuda_lib):
    from fourier_neural_spectral_gb300 import fnospec
    if fnospec.LIB_PATH.endswith("libfnospec_debug.so"):
        pytest.skip("this process runs the range-checked build")
    plan = fnospec.Plan(2, 4, 4, 32, 32, 8, 8)
    rc = fnospec.load_library().fno_plan_debug_bounds_margin(plan.handle, 8)
    assert rc == fnospec.FNO_ERR_UNSUPPORTED
