"""Edge shapes, invariants and error handling of the CUDA path."""
import ctypes

import numpy as np
import pytest

import oracle

from gpu_helpers import (assert_fp32_close, f32pairs_to_cplx, rand_layer_inputs, run_layer,
                         to_dev)

pytestmark = pytest.mark.gpu

EDGE_SHAPES = [
    # B, Cin, Cout, H, W, m1, m2
    (1, 1, 1, 2, 2, 1, 2),          # smallest grid, full modes incl. Nyquist
    (3, 5, 7, 16, 64, 8, 33),       # 2*m1 = H and m2 = W/2 + 1 (Nyquist column kept)
    (2, 3, 2, 64, 16, 1, 1),        # a single retained column / two rows
    (2, 3, 4, 8, 128, 2, 65),       # wide, non-square, Nyquist
    (1, 2, 3, 256, 4, 3, 3),        # tall, odd mode counts (ragged mode tile)
    (17, 5, 17, 16, 16, 3, 5),      # B > 16 and Cout > 16: ragged batch / channel tiles
    (1, 1, 1, 4096, 2, 1, 1),       # longest column transform
    (1, 1, 2, 2, 4096, 1, 2049),    # longest row transform, every column kept
    (2, 33, 31, 32, 32, 7, 9),      # channel counts off the tile sizes
    # fused transform path: row groups h = p + P*q with P > 1 (forward R = 64,
    # inverse R = 32..128, or 64 for long rows, once H > 256), Nyquist, non-square
    (2, 3, 4, 512, 64, 16, 9),      # fwd P = 8, inv R = 32, P = 16
    (1, 2, 2, 1024, 128, 64, 65),   # two retained frequencies per forward residue, Nyquist kept
    (2, 4, 4, 64, 256, 32, 129),    # 2*m1 = H, m2 = W/2 + 1
    (2, 3, 5, 256, 32, 128, 17),    # every row retained, narrow rows
    (3, 2, 3, 128, 64, 5, 7),       # odd mode counts inside the fused path
    (2, 4, 6, 2048, 32, 64, 16),    # tall grid: fwd P = 32, inv P = 16
    (1, 2, 3, 1024, 64, 100, 7),    # m1 off the column length: 1 or 2 frequencies per residue
    (2, 2, 2, 512, 32, 256, 5),     # 2*m1 = H with P > 1: 8 frequencies per forward residue
    # TMA-fed contraction: ragged boxes
    (3, 33, 40, 32, 32, 3, 5),      # B < batch tile, Cin % IC != 0, Cout % 32 != 0, NM % 4 == 2
    (5, 16, 96, 64, 32, 4, 4),      # B = 5 -> batch tile 8 split over two warp groups
    (20, 32, 32, 32, 32, 2, 3),     # B > 16: two batch tiles
    # 32-mode contraction blocks: ragged mode block, channel and batch tiles
    (5, 19, 13, 64, 64, 9, 11),     # nm = 198, Cout % 8 != 0, B = 5, Cin % IC != 0
    (20, 7, 9, 32, 64, 4, 9),       # B > 16: two batch tiles, nm = 72
    (1, 3, 2, 64, 32, 8, 2),        # B = 1, nm = 32 exactly
    # sizes that are not powers of two: direct-DFT transforms
    (2, 3, 4, 24, 16, 4, 4),        # H = 24
    (1, 2, 2, 421, 421, 12, 12),    # 421 x 421 (the Darcy-flow grid of the FNO literature)
    (3, 5, 7, 85, 85, 16, 16),      # odd sizes, 2*m1*m2 = 512 modes
    (2, 2, 3, 30, 50, 15, 26),      # 2*m1 = H, Nyquist column kept
    (1, 1, 1, 3, 5, 1, 3),          # smallest odd grid
    (1, 2, 2, 100, 4096, 10, 20),   # long power-of-two rows with H = 100
    # long rows (three-level row transform, shuffle reduce-scatter)
    (2, 3, 4, 64, 512, 16, 33),     # W = 512
    (1, 2, 2, 32, 1024, 8, 64),     # W = 1024, the largest supported m2
    (1, 1, 2, 256, 4096, 32, 17),   # W = 4096, one row group per CTA
    (2, 2, 3, 512, 2048, 128, 5),   # 2*m1 = 256 > both column lengths
    (1, 3, 3, 1024, 2048, 64, 1),   # a single kept column
    (1, 2, 2, 1024, 512, 64, 64),   # R = 64 = m1: both sides of every residue, Z staged in shared memory
]


@pytest.mark.parametrize("shape", EDGE_SHAPES)
def test_edge_shapes_match_oracle(cuda_lib, shape):
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape))
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    y, _ = run_layer(x, w, m1, m2)
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    assert_fp32_close(y, ref, str(shape))


# Direct-DFT grids whose rows (W >= ~200) take the pass kernels with streamed
# twiddle tiles, with enough rows (B * Cin * H >= 38,912) for the residue-class
# forward kernel: 32, 8 (W = 3 mod 4: all four row alignments) and 24 outputs
# per row.
MANY_ROW_SHAPES = [
    (8, 16, 4, 333, 333, 8, 16),
    (4, 32, 2, 305, 307, 6, 3),
    (4, 24, 4, 421, 421, 12, 12),
    (8, 32, 2, 160, 300, 4, 1),     # one kept column (2 outputs per row), W = 0 mod 4
    (1, 2, 2, 10, 4000, 2, 30),     # long rows (63 passes), K = 60 of the 64 the pass kernel takes
]


@pytest.mark.parametrize("shape", MANY_ROW_SHAPES)
def test_direct_dft_many_rows_match_oracle(cuda_lib, shape):
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 5)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    y, plan = run_layer(x, w, m1, m2)
    assert "direct-dft" in plan.description
    ref = oracle.spectral_conv2d(x, f32pairs_to_cplx(w), m1, m2)
    assert_fp32_close(y, ref, str(shape))


@pytest.mark.parametrize("H,W", [(16, 16), (8, 64), (128, 32)])
def test_identity_weights_full_modes_return_input(cuda_lib, H, W):
    C, m1, m2 = 3, H // 2, W // 2 + 1
    w = np.zeros((C, C, 2 * m1, m2, 2), np.float32)
    for i in range(C):
        w[i, i, :, :, 0] = 1.0
    x = np.random.default_rng(1).standard_normal((2, C, H, W)).astype(np.float32)
    y, _ = run_layer(x, w, m1, m2)
    assert_fp32_close(y, x, "identity")


def test_zero_input_gives_zero(cuda_lib):
    x = np.zeros((2, 4, 32, 32), np.float32)
    w = np.random.default_rng(2).random((4, 4, 8, 4, 2)).astype(np.float32)
    y, _ = run_layer(x, w, 4, 4)
    assert np.abs(y).max() == 0


def test_linearity_and_shift_equivariance(cuda_lib):
    rng = np.random.default_rng(3)
    B, C, H, W, m1, m2 = 2, 8, 64, 32, 5, 6
    x1, w = rand_layer_inputs(rng, B, C, C, H, W, m1, m2)
    x2 = rng.standard_normal(x1.shape).astype(np.float32)
    y1, plan = run_layer(x1, w, m1, m2)
    y2, _ = run_layer(x2, w, m1, m2, plan=plan)
    y12, _ = run_layer((x1 + 2 * x2).astype(np.float32), w, m1, m2, plan=plan)
    assert_fp32_close(y12, y1.astype(np.float64) + 2 * y2, "linearity")
    ys, _ = run_layer(np.roll(x1, (7, 3), axis=(2, 3)), w, m1, m2, plan=plan)
    assert_fp32_close(ys, np.roll(y1, (7, 3), axis=(2, 3)), "shift")


# ------------------------------------------------------------ error paths ---

@pytest.fixture()
def small_plan(cuda_lib):
    from fourier_neural_spectral_gb300 import fnospec
    return fnospec.Plan(2, 4, 4, 16, 16, 4, 4)


def _tensors(plan):
    import torch
    x = torch.randn(2, 4, 16, 16, device="cuda")
    w = torch.rand(4, 4, 8, 4, 2, device="cuda")
    y = torch.empty(2, 4, 16, 16, device="cuda")
    return x, w, y


def test_misaligned_pointer_rejected(small_plan):
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    with pytest.raises(fnospec.FnoError) as e:
        small_plan.fno_plan_execute(x.data_ptr() + 4, w, y)
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG


def test_host_pointer_rejected(small_plan):
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    host = np.zeros(2 * 4 * 16 * 16 + 64, np.float32)
    addr = (host.ctypes.data + 15) // 16 * 16
    with pytest.raises(fnospec.FnoError) as e:
        small_plan.fno_plan_execute(addr, w, y)
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG


def test_aliasing_rejected(small_plan):
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    with pytest.raises(fnospec.FnoError) as e:
        small_plan.fno_plan_execute(x, w, x)
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG


def test_small_workspace_rejected(small_plan):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    ws = torch.empty(small_plan.workspace_bytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fnospec.FnoError) as e:
        small_plan.fno_plan_execute(x, w, y, workspace=ws)
    assert e.value.status == fnospec.FNO_ERR_WORKSPACE


def test_null_pointer_rejected(small_plan):
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    with pytest.raises(fnospec.FnoError) as e:
        small_plan.fno_plan_execute(x, None, y)
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG


def test_device_status_clean_after_runs(small_plan):
    from fourier_neural_spectral_gb300 import fnospec
    x, w, y = _tensors(small_plan)
    for _ in range(3):
        small_plan.fno_plan_execute(x, w, y)
    assert small_plan.fno_get_device_status() == fnospec.FNO_OK
