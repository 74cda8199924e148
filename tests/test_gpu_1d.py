"""The 1D layer (fno_plan_create_1d) against the oracle's 1D layer.

The oracle's 1D layer and its backward are pinned on the CPU (tests/test_oracle.py:
numpy's rfft/irfft, the circular-convolution theorem, the adjoint and weight
identities).  Here the CUDA path -- the row transforms (pruned FFTs for
L = 512 .. 4096 with m <= 64, direct DFTs otherwise) with the orthonormal scale
on each side, and the plan's contraction -- matches it element by element
within the fp32 bars, on lengths that are and are not powers of two,
the Nyquist mode kept or not, the 32-mode contraction blocks and the
shape-generic contraction, the longest supported sequence, and L = 2.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import (TF32_REL_L2, assert_fp32_close, errors, f32pairs_to_cplx, to_dev)

pytestmark = pytest.mark.gpu

SHAPES_1D = [
    # B, Cin, Cout, L, m
    (2, 3, 2, 16, 5),         # tiny, shape-generic contraction (m < 32)
    (4, 32, 32, 1024, 64),    # 32-mode contraction blocks
    (2, 4, 6, 100, 12),       # L not a power of two
    (1, 2, 2, 15, 8),         # odd L, every mode kept (no Nyquist bin)
    (2, 3, 3, 64, 33),        # Nyquist mode kept (c = 1 at k = L/2)
    (3, 5, 7, 4096, 9),       # longest sequence
    (1, 1, 1, 2, 2),          # L = 2: only the k = 0 and Nyquist bins
    (17, 6, 5, 256, 40),      # B > 16, 40 modes (ragged 32-mode block)
    (3, 5, 7, 512, 40),       # FFT rows (L >= 512, m <= 64), odd sequence counts 15 / 21
    (1, 3, 2, 2048, 64),      # FFT rows, 64 modes, 3 / 2 sequences
    (1, 2, 3, 256, 100),      # direct DFTs with K split over CTAs both ways (2m = 200)
    (48, 832, 2, 1000, 12),   # 39,936 sequences: residue-class forward rows, streamed tiles
]


def rand_1d(rng, B, Cin, Cout, L, m):
    x = rng.standard_normal((B, Cin, L)).astype(np.float32)
    w = (rng.random((Cin, Cout, m, 2)) / (Cin * Cout)).astype(np.float32)
    return x, w


def plan_1d(B, Cin, Cout, L, m, precision="fp32"):
    from fourier_neural_spectral_gb300 import fnospec
    return fnospec.Plan1d(B, Cin, Cout, L, m, precision)


@pytest.mark.parametrize("shape", SHAPES_1D)
def test_layer_1d_matches_oracle(cuda_lib, shape):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, L, m = shape
    rng = np.random.default_rng(sum(shape) + 101)
    x, w = rand_1d(rng, B, Cin, Cout, L, m)
    plan = plan_1d(*shape)
    y = torch.empty((B, Cout, L), dtype=torch.float32, device="cuda")
    plan.fno_plan_execute(to_dev(x), to_dev(w), y)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    ref = oracle.spectral_conv1d(x, f32pairs_to_cplx(w), m)
    assert_fp32_close(y.cpu().numpy(), ref, f"1d layer {shape} [{plan.description}]")


def test_forward_modes_1d_match_truncated_rfft(cuda_lib):
    # the forward stage alone is the truncated orthonormal rfft (numpy, double)
    import torch
    B, Cin, Cout, L, m = 3, 4, 2, 100, 17
    rng = np.random.default_rng(7)
    x, _ = rand_1d(rng, B, Cin, Cout, L, m)
    plan = plan_1d(B, Cin, Cout, L, m)
    X = torch.empty((B, Cin, m, 2), dtype=torch.float32, device="cuda")
    plan.fno_forward_modes(to_dev(x), X)
    torch.cuda.synchronize()
    ref = np.fft.rfft(x.astype(np.float64), norm="ortho")[..., :m]
    assert_fp32_close(f32pairs_to_cplx(X.cpu().numpy()), ref, "1d forward modes")


def test_layer_1d_tf32(cuda_lib):
    import torch
    B, Cin, Cout, L, m = 4, 32, 32, 1024, 64
    rng = np.random.default_rng(19)
    x, w = rand_1d(rng, B, Cin, Cout, L, m)
    plan = plan_1d(B, Cin, Cout, L, m, "tf32")
    y = torch.empty((B, Cout, L), dtype=torch.float32, device="cuda")
    plan.fno_plan_execute(to_dev(x), to_dev(w), y)
    torch.cuda.synchronize()
    rel, _ = errors(y.cpu().numpy(), oracle.spectral_conv1d(x, f32pairs_to_cplx(w), m))
    assert rel <= TF32_REL_L2, f"tf32 1d rel-L2 {rel:.3e} [{plan.description}]"


@pytest.mark.parametrize("shape", [(2, 3, 2, 16, 5), (4, 32, 32, 1024, 64), (2, 4, 6, 100, 12),
                                   (2, 3, 3, 64, 33), (1, 1, 1, 2, 2), (3, 5, 7, 512, 40)])
def test_backward_1d_matches_oracle(cuda_lib, shape):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, L, m = shape
    rng = np.random.default_rng(sum(shape) + 202)
    x, w = rand_1d(rng, B, Cin, Cout, L, m)
    gy = rng.standard_normal((B, Cout, L)).astype(np.float32)
    plan = plan_1d(*shape)
    xt, wt = to_dev(x), to_dev(w)
    gx, gw = torch.empty_like(xt), torch.empty_like(wt)
    plan.fno_plan_backward(xt, wt, to_dev(gy), gx, gw)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    ref_gx, ref_gw = oracle.spectral_conv1d_backward(x, f32pairs_to_cplx(w), gy, m)
    assert_fp32_close(gx.cpu().numpy(), ref_gx, f"1d dL/dx {shape}")
    assert_fp32_close(f32pairs_to_cplx(gw.cpu().numpy()), ref_gw, f"1d dL/dw {shape}")


def test_block_1d_matches_oracle(cuda_lib):
    import torch
    B, Cin, Cout, L, m = 2, 12, 10, 200, 24
    rng = np.random.default_rng(23)
    x, w = rand_1d(rng, B, Cin, Cout, L, m)
    wpw = (rng.standard_normal((Cout, Cin)) / np.sqrt(Cin)).astype(np.float32)
    bias = rng.standard_normal(Cout).astype(np.float32)
    plan = plan_1d(B, Cin, Cout, L, m)
    y = torch.empty((B, Cout, L), dtype=torch.float32, device="cuda")
    plan.fno_block_execute(to_dev(x), to_dev(w), to_dev(wpw), to_dev(bias), y, "gelu")
    torch.cuda.synchronize()
    ref = oracle.block1d(x, f32pairs_to_cplx(w), wpw, bias, m, "gelu")
    assert_fp32_close(y.cpu().numpy(), ref, "1d block")


def test_autograd_1d_matches_oracle(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, L, m = 2, 4, 6, 96, 20
    rng = np.random.default_rng(29)
    x, w = rand_1d(rng, B, Cin, Cout, L, m)
    gy = rng.standard_normal((B, Cout, L)).astype(np.float32)
    xt = to_dev(x).requires_grad_(True)
    wt = torch.view_as_complex(to_dev(w)).detach().requires_grad_(True)
    y = fnospec.spectral_conv1d_autograd(xt, wt, m)
    (y * to_dev(gy)).sum().backward()
    wc = f32pairs_to_cplx(w)
    ref_gx, ref_gw = oracle.spectral_conv1d_backward(x, wc, gy, m)
    assert_fp32_close(y.detach().cpu().numpy(), oracle.spectral_conv1d(x, wc, m), "autograd 1d y")
    assert_fp32_close(xt.grad.cpu().numpy(), ref_gx, "autograd 1d dL/dx")
    assert_fp32_close(wt.grad.cpu().numpy(), ref_gw, "autograd 1d dL/dw")
