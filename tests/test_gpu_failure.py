"""Failure detection on the GPU without a fault: the forced-timeout hook.

fno_plan_debug_force_timeout makes every bounded device wait of a plan give up
at once, as if its one-second limit had run out.  The kernels then set
FNO_DEVERR_TIMEOUT, let their own bulk copies and tensor-core work finish, free
their tensor memory and return.  Each
case below checks that the call reports FNO_ERR_TIMEOUT through
fno_get_device_status, that the context stays usable, and that the same plan
with the hook cleared again matches the oracle.  The cases cover every kernel
family that waits on an mbarrier: the 32-mode contraction (TMA ring with a
producer warp), the inverse transforms that stage Z by one bulk copy (short and
long rows), the long-row forward that stages row pairs, the tcgen05 contraction
(TMEM accumulators), the direct-DFT inverse rows (bulk-copied twiddle tiles),
the block epilogue and the backward.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import (TF32_REL_L2, assert_fp32_close, errors, f32pairs_to_cplx,
                         rand_layer_inputs, to_dev)

pytestmark = pytest.mark.gpu

CASES = [
    # (B, Cin, Cout, H, W, m1, m2), precision, kernel the waits belong to
    ((2, 64, 64, 128, 128, 32, 32), "fp32", "inv_fused"),    # mix_wide + staged Z
    ((1, 8, 8, 512, 512, 16, 16), "fp32", "fwd_fused"),     # long rows: staged pairs, staged Z
    ((2, 32, 32, 64, 64, 16, 16), "tf32", "mix_tcm"),       # tcgen05, weights in TMEM
    ((32, 32, 32, 16, 16, 4, 4), "tf32", "mix_tc_"),        # tcgen05, operands in smem
    ((2, 8, 8, 30, 50, 6, 9), "fp32", "dft_irows"),          # direct DFT: streamed twiddle tiles
]


def _execute(plan, x, w, Cout):
    import torch
    B, _, H, W = x.shape
    y = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
    plan.fno_plan_execute(to_dev(x), to_dev(w), y)
    return y


@pytest.mark.parametrize("shape,precision,kernel", CASES)
def test_forced_timeout_reports_and_recovers(cuda_lib, shape, precision, kernel):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 77)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, precision)
    assert any(kernel in k["name"] for k in plan.kernels), plan.description
    assert plan.fno_get_device_status() == fnospec.FNO_OK

    plan.fno_plan_debug_force_timeout(True)
    _execute(plan, x, w, Cout)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_ERR_TIMEOUT, plan.description
    # the word was cleared by the read; the context still runs work
    assert plan.fno_get_device_status() == fnospec.FNO_OK

    plan.fno_plan_debug_force_timeout(False)
    y = _execute(plan, x, w, Cout)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    if precision == "fp32":
        assert_fp32_close(y.cpu().numpy(), ref, f"after recovery {shape}")
    else:
        rel, _ = errors(y.cpu().numpy(), ref)
        assert rel <= TF32_REL_L2, f"after recovery {shape}: rel-L2 {rel:.3e}"


def test_forced_timeout_in_backward_and_block(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, H, W, m1, m2 = 2, 64, 64, 128, 128, 32, 32
    rng = np.random.default_rng(91)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    gy = rng.standard_normal((B, Cout, H, W)).astype(np.float32)
    wpw = (rng.standard_normal((Cout, Cin)) / np.sqrt(Cin)).astype(np.float32)
    bias = rng.standard_normal(Cout).astype(np.float32)
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2)
    xt, wt, gyt = to_dev(x), to_dev(w), to_dev(gy)
    gx, gw = torch.empty_like(xt), torch.empty_like(wt)
    y = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")

    plan.fno_plan_debug_force_timeout(True)
    plan.fno_plan_backward(xt, wt, gyt, gx, gw)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_ERR_TIMEOUT
    plan.fno_block_execute(xt, wt, to_dev(wpw), to_dev(bias), y, "gelu")
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_ERR_TIMEOUT

    plan.fno_plan_debug_force_timeout(False)
    plan.fno_plan_backward(xt, wt, gyt, gx, gw)
    plan.fno_block_execute(xt, wt, to_dev(wpw), to_dev(bias), y, "gelu")
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    wc = f32pairs_to_cplx(w)
    ref_gx, ref_gw = oracle.spectral_conv2d_backward(x, wc, gy, m1, m2)
    assert_fp32_close(gx.cpu().numpy(), ref_gx, "dL/dx after recovery")
    assert_fp32_close(f32pairs_to_cplx(gw.cpu().numpy()), ref_gw, "dL/dw after recovery")
    assert_fp32_close(y.cpu().numpy(), oracle.block(x, wc, wpw, bias, m1, m2, "gelu"),
                      "block after recovery")


def test_force_timeout_rejects_null_plan(cuda_lib):
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    assert lib.fno_plan_debug_force_timeout(None, 1) == fnospec.FNO_ERR_INVALID_ARG


def _cudart():
    """The CUDA runtime instance libfnospec is linked against (the one already
    loaded in this process under its soname), for the pending-error cases."""
    import ctypes
    import os
    from fourier_neural_spectral_gb300 import fnospec
    fnospec.load_library()
    try:
        rt = ctypes.CDLL("libcudart.so.13", mode=os.RTLD_NOLOAD | ctypes.RTLD_GLOBAL)
    except OSError:
        rt = ctypes.CDLL("libcudart.so.13")
    for f in ("cudaGetLastError", "cudaPeekAtLastError", "cudaSetDevice", "cudaGetDeviceCount"):
        getattr(rt, f).restype = ctypes.c_int
    return rt


def test_pending_runtime_error_is_reported_before_any_work(cuda_lib):
    """A stream whose host thread holds an unread runtime error: made on the
    host only (cudaSetDevice with an ordinal past the device count, which the
    runtime rejects without touching a GPU).  Every entry point that enqueues
    work returns FNO_ERR_CUDA without enqueuing anything and leaves the error
    pending for its owner; once the caller has read it, the next call is
    correct."""
    import ctypes
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    rt = _cudart()
    shape = B, Cin, Cout, H, W, m1, m2 = 2, 32, 32, 64, 64, 16, 16
    rng = np.random.default_rng(99)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = fnospec.Plan(*shape, "fp32")
    xt, wt = to_dev(x), to_dev(w)
    y = torch.full((B, Cout, H, W), float("nan"), dtype=torch.float32, device="cuda")
    ws_ptr, ws_n = plan._ws(None)
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    assert rt.cudaGetLastError() == 0

    n = ctypes.c_int()
    assert rt.cudaGetDeviceCount(ctypes.byref(n)) == 0
    bad = rt.cudaSetDevice(n.value + 7)
    assert bad != 0 and rt.cudaPeekAtLastError() == bad
    calls = [
        lambda: lib.fno_plan_execute(plan.handle, xt.data_ptr(), wt.data_ptr(), y.data_ptr(),
                                     ws_ptr, ws_n, s),
        lambda: lib.fno_spectral_conv2d(xt.data_ptr(), wt.data_ptr(), y.data_ptr(), *shape, s),
        lambda: lib.fno_spectral_conv2d_noalloc(xt.data_ptr(), wt.data_ptr(), y.data_ptr(),
                                                *shape, s),
        lambda: lib.fno_forward_modes(plan.handle, xt.data_ptr(), y.data_ptr(), ws_ptr, ws_n, s),
    ]
    for call in calls:
        assert call() == fnospec.FNO_ERR_CUDA
        assert rt.cudaPeekAtLastError() == bad  # still the caller's, unread
    assert rt.cudaGetLastError() == bad        # the caller reads (and clears) it
    assert rt.cudaPeekAtLastError() == 0
    torch.cuda.synchronize()
    assert bool(torch.isnan(y).all())          # nothing was enqueued

    assert lib.fno_plan_execute(plan.handle, xt.data_ptr(), wt.data_ptr(), y.data_ptr(), ws_ptr,
                                ws_n, s) == fnospec.FNO_OK
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    assert_fp32_close(y.cpu().numpy(), oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2),
                      "after the pending error was read")


def test_plans_on_every_device_get_their_kernel_limits(cuda_lib):
    """Kernel attributes (the fused kernels' dynamic shared-memory limits) are
    set per device: a plan created on each visible device, after switching the
    current device back and forth, runs the fused 128x128 kernels (over 48 KB of
    shared memory) correctly."""
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    shape = B, Cin, Cout, H, W, m1, m2 = 2, 16, 16, 128, 128, 32, 32
    rng = np.random.default_rng(5)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    n = torch.cuda.device_count()
    for rep in range(2):
        for d in list(range(n)) + [0]:
            with torch.cuda.device(d):
                plan = fnospec.Plan(*shape, "fp32")
                assert "fused" in plan.description
                xt = torch.from_numpy(x).to(f"cuda:{d}")
                wt = torch.from_numpy(w).to(f"cuda:{d}")
                y = torch.empty((B, Cout, H, W), dtype=torch.float32, device=f"cuda:{d}")
                plan.fno_plan_execute(xt, wt, y)
                torch.cuda.synchronize(d)
                assert plan.fno_get_device_status() == fnospec.FNO_OK
                assert_fp32_close(y.cpu().numpy(), ref, f"device {d}")
