"""fno_spectral_conv2d_noalloc: the layer for callers that cannot allocate
device memory (hosts that own every allocation, allocation-free real-time
loops).  It must give the same result as the regular plan path, call after
call, with its static scratch reused; shapes that do not fit the scratch are
refused before anything runs.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import FP32_MAX_ABS, FP32_REL_L2, errors, rand_layer_inputs, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    (2, 4, 4, 16, 16, 4, 4),
    (8, 32, 32, 64, 64, 16, 16),
    (3, 5, 7, 16, 64, 8, 33),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_noalloc_matches_plan_path_twice(cuda_lib, shape):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    B, Cin, Cout, H, W, m1, m2 = shape
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, "fp32")
    rng = np.random.default_rng(sum(shape) + 7)
    for call in range(2):  # two calls in a row: the shared scratch must not leak state
        x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
        xt, wt = to_dev(x), to_dev(w)
        y_ref = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
        y_new = torch.full((B, Cout, H, W), float("nan"), dtype=torch.float32, device="cuda")
        plan.fno_plan_execute(xt, wt, y_ref)
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.fno_spectral_conv2d_noalloc(xt.data_ptr(), wt.data_ptr(), y_new.data_ptr(),
                                             B, Cin, Cout, H, W, m1, m2, stream)
        assert rc == fnospec.FNO_OK, fnospec.status_string(rc)
        torch.cuda.synchronize()
        rel, mx = errors(y_new.cpu().numpy(), y_ref.cpu().numpy())
        assert rel <= FP32_REL_L2 and mx <= FP32_MAX_ABS, (call, rel, mx)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    lib = fnospec.load_library()
    B, Cin, Cout, H, W, m1, m2 = 16, 64, 64, 128, 128, 32, 32   # ~67 MB of scratch
    x = torch.zeros((B, Cin, H, W), device="cuda")
    w = torch.zeros((Cin, Cout, 2 * m1, m2, 2), device="cuda")
    y = torch.zeros((B, Cout, H, W), device="cuda")
    rc = lib.fno_spectral_conv2d_noalloc(x.data_ptr(), w.data_ptr(), y.data_ptr(), B, Cin, Cout,
                                         H, W, m1, m2, torch.cuda.current_stream().cuda_stream)
    assert rc == fnospec.FNO_ERR_UNSUPPORTED
