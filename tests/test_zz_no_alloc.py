"""fno_spectral_conv2d_noalloc: the layer for callers that cannot allocate
device memory (hosts that own every allocation, allocation-free real-time
loops, plugins whose host forbids allocation after start-up).

Its result is checked against the double-precision oracle at the fp32 bounds,
call after call with the static scratch reused (the second call of each shape
gets new inputs, so state left in the scratch by the first would show), and
once more against the plan path.  The two paths differ in their twiddle
tables (the plan rounds host cos/sin computed in double, this entry point
rounds the device's double sincospi), so that comparison uses the fp32 bounds,
not bit equality.  A second call must not change the device's free memory,
and shapes whose scratch does not fit are refused before anything runs.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest

import oracle

from gpu_helpers import (FP32_MAX_ABS, FP32_REL_L2, errors, f32pairs_to_cplx, rand_layer_inputs,
                         to_dev)

pytestmark = pytest.mark.gpu

SHAPES = [
    (2, 4, 4, 16, 16, 4, 4),
    (8, 32, 32, 64, 64, 16, 16),
    (3, 5, 7, 16, 64, 8, 33),    # Nyquist column kept (m2 = W/2 + 1)
    (2, 3, 5, 24, 20, 5, 7),     # sizes that are not powers of two: direct-DFT stages
]


def _noalloc(lib, xt, wt, yt, shape):
    import torch
    B, Cin, Cout, H, W, m1, m2 = shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.fno_spectral_conv2d_noalloc(xt.data_ptr(), wt.data_ptr(), yt.data_ptr(),
                                           B, Cin, Cout, H, W, m1, m2, stream)


@pytest.mark.parametrize("shape", SHAPES)
def test_noalloc_matches_oracle_twice(cuda_lib, shape):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 7)
    for call in range(2):  # two calls in a row: the shared scratch must not leak state
        x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
        xt, wt = to_dev(x), to_dev(w)
        y_new = torch.full((B, Cout, H, W), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = _noalloc(lib, xt, wt, y_new, shape)
        assert rc == fnospec.FNO_OK, fnospec.status_string(rc)
        torch.cuda.synchronize()
        if call == 1:
            # the first call has loaded the kernels; from then on a call takes
            # no device memory at all
            assert torch.cuda.mem_get_info()[0] == free0
        got = y_new.cpu().numpy()
        ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
        rel, mx = errors(got, ref)
        assert rel <= FP32_REL_L2 and mx <= FP32_MAX_ABS, ("oracle", call, rel, mx)
        # the plan path on the same inputs (different twiddle tables: fp32 bounds)
        plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, "fp32")
        y_ref = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
        plan.fno_plan_execute(xt, wt, y_ref)
        torch.cuda.synchronize()
        rel, mx = errors(got, y_ref.cpu().numpy())
        assert rel <= FP32_REL_L2 and mx <= FP32_MAX_ABS, ("plan path", call, rel, mx)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    shape = B, Cin, Cout, H, W, m1, m2 = 16, 64, 64, 128, 128, 32, 32   # ~67 MB of scratch
    x = torch.zeros((B, Cin, H, W), device="cuda")
    w = torch.zeros((Cin, Cout, 2 * m1, m2, 2), device="cuda")
    y = torch.full((B, Cout, H, W), 7.0, device="cuda")
    rc = _noalloc(lib, x, w, y, shape)
    assert rc == fnospec.FNO_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())  # nothing ran
