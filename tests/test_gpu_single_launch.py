"""The whole layer as one cooperative launch (fno_plan_set_single_launch):
forward transforms, contraction and inverse transforms as three phases of one
persistent grid with grid-wide barriers between them.

Checked against the double-precision oracle on the shapes the path serves
(square planes of 32..256 points, batch up to 16, compiled and run-time mode
counts, the Nyquist column), against the three-launch path, over many
consecutive launches (the barrier counter carries over from launch to launch),
and through the forced-timeout hook (a barrier wait that runs out is reported
and the next launch is correct again)."""
import numpy as np
import pytest

import oracle
from fourier_neural_spectral_gb300 import synth

from gpu_helpers import (assert_fp32_close, f32pairs_to_cplx, rand_layer_inputs, run_layer,
                         to_dev)

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, Cin, Cout, H, W, m1, m2
    (8, 32, 32, 64, 64, 16, 16),     # the 64x64 workload's shape (compiled mode counts)
    (16, 64, 64, 128, 128, 32, 32),  # the 128x128 workload's shape
    (2, 8, 8, 256, 256, 64, 64),     # 256-point rows
    (3, 5, 7, 32, 32, 8, 8),         # smallest planes, ragged channel counts
    (1, 12, 20, 128, 128, 10, 20),   # run-time mode counts, one batch row
    (4, 6, 3, 64, 64, 16, 33),       # Nyquist column kept (m2 = W/2 + 1)
    (16, 3, 9, 32, 32, 16, 17),      # 2*m1 = H and the Nyquist column, full batch tile
]


def single_plan(shape, enable=True):
    from fourier_neural_spectral_gb300 import fnospec
    plan = fnospec.Plan(*shape, "fp32")
    plan.fno_plan_set_single_launch(enable)
    return plan


@pytest.mark.parametrize("shape", SHAPES)
def test_single_launch_matches_oracle(cuda_lib, shape):
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 3)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = single_plan(shape)
    assert plan.launches == 1 and "single-launch" in plan.description, plan.description
    y, _ = run_layer(x, w, m1, m2, plan=plan)
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    rel, mx = assert_fp32_close(y, ref, str(shape))
    y3, _ = run_layer(x, w, m1, m2, plan=single_plan(shape, False))
    assert_fp32_close(y, y3, "against the three-launch path")
    print(f"{shape}: rel-L2 {rel:.2e} max-abs {mx:.2e}")


def test_plans_start_with_three_launches(cuda_lib):
    from fourier_neural_spectral_gb300 import fnospec
    for name in ("B8_C32_64x64_m16_smooth", "B16_C64_128x128_m32"):
        cfg = synth.CONFIGS[name]
        plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
        assert plan.launches == 3, plan.description
        plan.fno_plan_set_single_launch(True)
        assert plan.launches == 1 and plan.kernels[0]["name"] == "layer_persistent"


def test_many_consecutive_launches(cuda_lib):
    """The grid-barrier counter grows by two arrivals per CTA per launch; every
    launch must find it at a multiple of the grid size."""
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    shape = B, Cin, Cout, H, W, m1, m2 = (4, 16, 16, 64, 64, 16, 16)
    rng = np.random.default_rng(8)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = single_plan(shape)
    xt, wt = to_dev(x), to_dev(w)
    ys = [torch.empty((B, Cout, H, W), device="cuda") for _ in range(60)]
    for yt in ys:
        plan.fno_plan_execute(xt, wt, yt)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    first = ys[0].cpu().numpy()
    assert_fp32_close(first, ref, "first launch")
    for yt in ys[1:]:
        assert np.array_equal(yt.cpu().numpy(), first)  # same launch, same arithmetic


def test_forced_barrier_timeout_reports_and_recovers(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    shape = B, Cin, Cout, H, W, m1, m2 = (2, 8, 8, 64, 64, 16, 16)
    rng = np.random.default_rng(9)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    plan = single_plan(shape)
    xt, wt = to_dev(x), to_dev(w)
    y = torch.empty((B, Cout, H, W), device="cuda")
    plan.fno_plan_debug_force_timeout(True)
    for _ in range(3):
        plan.fno_plan_execute(xt, wt, y)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_ERR_TIMEOUT
    plan.fno_plan_debug_force_timeout(False)
    for _ in range(2):
        plan.fno_plan_execute(xt, wt, y)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    assert_fp32_close(y.cpu().numpy(), oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2),
                      "after the forced timeouts")


def test_single_launch_argument_errors(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    unsupported = [
        (17, 4, 4, 64, 64, 16, 16),      # batch above 16
        (2, 4, 4, 64, 128, 16, 16),      # planes that are not square
        (2, 4, 4, 512, 512, 16, 16),     # long rows
        (2, 4, 4, 16, 16, 4, 4),         # rows shorter than 32 points (shape-generic path)
        (2, 4, 4, 60, 60, 8, 8),         # not a power of two
    ]
    for shape in unsupported:
        plan = fnospec.Plan(*shape, "fp32")
        assert lib.fno_plan_set_single_launch(plan.handle, 1) == fnospec.FNO_ERR_UNSUPPORTED
        assert lib.fno_plan_set_single_launch(plan.handle, 0) == fnospec.FNO_OK
    assert lib.fno_plan_set_single_launch(None, 1) == fnospec.FNO_ERR_INVALID_ARG
    plan = fnospec.Plan(2, 4, 4, 64, 64, 16, 16, "fp32")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(plan.launches + 1)]
    plan.fno_plan_record_events(evs)
    assert lib.fno_plan_set_single_launch(plan.handle, 1) == fnospec.FNO_ERR_INVALID_ARG
    plan.fno_plan_record_events(None)
    assert lib.fno_plan_set_single_launch(plan.handle, 1) == fnospec.FNO_OK
    assert plan.launches == 3  # the Python view refreshes only through the method
    plan.fno_plan_set_single_launch(True)
    assert plan.launches == 1
