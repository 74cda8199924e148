"""Backward of the layer (fno_plan_backward) against the oracle's backward.

The oracle's backward is pinned on the CPU (tests/test_oracle.py: adjoint
identity, weight identity, finite differences); here the CUDA gradients dL/dx
and dL/dw match it element by element within the fp32 bars, on shapes that
exercise every path the backward takes: the fused short- and long-row
transforms (row groups, staged Z), the shape-generic transforms, the 32-mode
adjoint contraction and its shape-generic fallback, and the weight gradient
with the k2 = 0 / Nyquist column weights.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_fp32_close, f32pairs_to_cplx, rand_layer_inputs, to_dev

pytestmark = pytest.mark.gpu

BACKWARD_SHAPES = [
    # B, Cin, Cout, H, W, m1, m2
    (2, 4, 4, 16, 16, 4, 4),        # tiny: shape-generic transforms, 2*m1*m2 < 32
    (2, 3, 2, 8, 8, 2, 3),          # adjoint contraction on the generic fallback
    (3, 5, 7, 16, 64, 8, 33),       # Nyquist column kept, odd channel counts
    (2, 8, 6, 64, 64, 16, 16),      # fused 64-point rows, 32-mode adjoint blocks
    (2, 16, 16, 128, 128, 32, 32),  # fused 128-point rows with (m1, m2) compiled in
    (17, 5, 6, 32, 32, 4, 8),       # B > 16: two batch tiles
    (1, 4, 4, 256, 256, 64, 64),    # 256-point rows
    (1, 2, 3, 512, 2048, 64, 16),   # long rows, row groups (P > 1), staged Z
    (2, 3, 2, 1024, 64, 100, 7),    # m1 > R: several frequencies per residue
    (2, 3, 4, 24, 20, 5, 6),        # not powers of two: direct-DFT transforms
]


def run_backward(x, w, gy, m1, m2, want_x=True, want_w=True):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2)
    xt, wt, gyt = to_dev(x), to_dev(w), to_dev(gy)
    gx = torch.empty_like(xt) if want_x else None
    gw = torch.empty_like(wt) if want_w else None
    plan.fno_plan_backward(xt if want_w else None, wt if want_x else None, gyt, gx, gw)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    return (None if gx is None else gx.cpu().numpy(),
            None if gw is None else f32pairs_to_cplx(gw.cpu().numpy()))


@pytest.mark.parametrize("shape", BACKWARD_SHAPES)
def test_backward_matches_oracle(cuda_lib, shape):
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 7)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    gy = rng.standard_normal((B, Cout, H, W)).astype(np.float32)
    gx, gw = run_backward(x, w, gy, m1, m2)
    ref_gx, ref_gw = oracle.spectral_conv2d_backward(x, f32pairs_to_cplx(w), gy, m1, m2)
    assert_fp32_close(gx, ref_gx, f"dL/dx {shape}")
    assert_fp32_close(gw, ref_gw, f"dL/dw {shape}")


def test_backward_single_gradients(cuda_lib):
    # gx alone (x may be NULL) and gw alone (w may be NULL) give the same results
    B, Cin, Cout, H, W, m1, m2 = 2, 8, 8, 64, 64, 16, 16
    rng = np.random.default_rng(3)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    gy = rng.standard_normal((B, Cout, H, W)).astype(np.float32)
    gx_both, gw_both = run_backward(x, w, gy, m1, m2)
    gx_only, none_w = run_backward(x, w, gy, m1, m2, want_w=False)
    none_x, gw_only = run_backward(x, w, gy, m1, m2, want_x=False)
    assert none_w is None and none_x is None
    assert np.array_equal(gx_only, gx_both)
    assert np.array_equal(gw_only, gw_both)


def test_backward_rejects_bad_arguments(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, H, W, m1, m2 = 1, 2, 2, 32, 32, 4, 4
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2)
    x = torch.zeros((B, Cin, H, W), device="cuda")
    w = torch.zeros((Cin, Cout, 2 * m1, m2, 2), device="cuda")
    gy = torch.zeros((B, Cout, H, W), device="cuda")
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_plan_backward(x, w, gy, None, None)  # nothing to compute
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_plan_backward(x, w, gy, gy, None)  # dL/dx written over dL/dy
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_plan_backward(None, w, gy, None, torch.empty_like(w))  # dL/dw needs x
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG


def test_autograd_function_matches_oracle(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, H, W, m1, m2 = 2, 4, 6, 32, 32, 8, 8
    rng = np.random.default_rng(11)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    gy = rng.standard_normal((B, Cout, H, W)).astype(np.float32)
    xt = to_dev(x).requires_grad_(True)
    wt = torch.view_as_complex(to_dev(w)).detach().requires_grad_(True)
    y = fnospec.spectral_conv2d_autograd(xt, wt, m1, m2)
    (y * to_dev(gy)).sum().backward()
    ref_y = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    ref_gx, ref_gw = oracle.spectral_conv2d_backward(x, f32pairs_to_cplx(w), gy, m1, m2)
    assert_fp32_close(y.detach().cpu().numpy(), ref_y, "autograd y")
    assert_fp32_close(xt.grad.cpu().numpy(), ref_gx, "autograd dL/dx")
    assert_fp32_close(wt.grad.cpu().numpy(), ref_gw, "autograd dL/dw")
