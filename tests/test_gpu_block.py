"""FNO block (spectral layer + pointwise branch + bias, GELU) against the oracle.

fno_block_execute = fno_plan_execute then fno_block_epilogue (in place over y);
compared element by element with oracle.block in double, on shapes covering
ragged pixel tiles (P < 128), ragged channel chunks (Cin not a multiple of 32),
two output-channel blocks (Cout > 64, the fp32 kernel), the tensor-core pointwise
branch (Cout <= 64) with several units per CTA, no bias and no activation.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_fp32_close, f32pairs_to_cplx, rand_layer_inputs, to_dev

pytestmark = pytest.mark.gpu

BLOCK_CASES = [
    # (B, Cin, Cout, H, W, m1, m2), activation, with bias
    ((2, 4, 4, 16, 16, 4, 4), "gelu", True),      # shape-generic spectral path
    ((2, 8, 6, 64, 64, 16, 16), "gelu", True),
    ((2, 16, 16, 128, 128, 32, 32), "gelu", True),
    ((1, 3, 70, 32, 32, 8, 8), "gelu", False),    # two output blocks, one short chunk
    ((1, 100, 5, 8, 8, 2, 3), "none", True),      # four channel chunks, P = 64 < 128
    ((2, 33, 9, 16, 64, 8, 33), "none", False),   # Nyquist column, ragged channels
    # tensor-core pointwise branch (Cout <= 64): several units per CTA, so the
    # double-buffered accumulators and y tiles are reused many times
    ((4, 64, 64, 128, 128, 32, 32), "gelu", True),
    ((2, 32, 32, 256, 256, 16, 16), "none", True),
    ((3, 20, 40, 48, 80, 8, 8), "gelu", False),   # N = 64 with 40 channels: a quarter empty
    ((17, 16, 16, 8, 8, 2, 2), "gelu", True),     # P = 64 < 128 and 17 units
    ((1, 1, 1, 2, 2, 1, 2), "gelu", True),        # one channel, P = 4: boxes mostly outside
]


def run_block(x, w, wpw, bias, m1, m2, activation):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2)
    y = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
    plan.fno_block_execute(to_dev(x), to_dev(w), to_dev(wpw),
                           None if bias is None else to_dev(bias), y, activation)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    return y.cpu().numpy(), plan


@pytest.mark.parametrize("shape,activation,with_bias", BLOCK_CASES)
def test_block_matches_oracle(cuda_lib, shape, activation, with_bias):
    B, Cin, Cout, H, W, m1, m2 = shape
    rng = np.random.default_rng(sum(shape) + 31)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    wpw = (rng.standard_normal((Cout, Cin)) / np.sqrt(Cin)).astype(np.float32)
    bias = rng.standard_normal(Cout).astype(np.float32) if with_bias else None
    y, _ = run_block(x, w, wpw, bias, m1, m2, activation)
    ref = oracle.block(x, f32pairs_to_cplx(w), wpw, np.zeros(Cout) if bias is None else bias,
                       m1, m2, activation)
    assert_fp32_close(y, ref, f"block {shape} {activation}")


def test_epilogue_alone_matches_block(cuda_lib):
    # fno_plan_execute then fno_block_epilogue gives the same bits as fno_block_execute
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, Cout, H, W, m1, m2 = 2, 8, 8, 64, 64, 16, 16
    rng = np.random.default_rng(5)
    x, w = rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2)
    wpw = rng.standard_normal((Cout, Cin)).astype(np.float32)
    bias = rng.standard_normal(Cout).astype(np.float32)
    y_block, plan = run_block(x, w, wpw, bias, m1, m2, "gelu")
    y = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
    xt = to_dev(x)
    plan.fno_plan_execute(xt, to_dev(w), y)
    plan.fno_block_epilogue(xt, to_dev(wpw), to_dev(bias), y, "gelu")
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_block)


def test_block_rejects_bad_arguments(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    plan = fnospec.Plan(1, 300, 2, 16, 16, 2, 2)  # Cin above the epilogue's limit
    x = torch.zeros((1, 300, 16, 16), device="cuda")
    y = torch.zeros((1, 2, 16, 16), device="cuda")
    wpw = torch.zeros((2, 300), device="cuda")
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_block_epilogue(x, wpw, None, y, "gelu")
    assert e.value.status == fnospec.FNO_ERR_UNSUPPORTED
    plan = fnospec.Plan(1, 2, 2, 16, 16, 2, 2)
    x = torch.zeros((1, 2, 16, 16), device="cuda")
    wpw = torch.zeros((2, 2), device="cuda")
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_block_epilogue(x, wpw, None, y, 7)  # no such activation
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG
    with pytest.raises(fnospec.FnoError) as e:
        plan.fno_block_epilogue(x, wpw, None, x, "gelu")  # y over x
    assert e.value.status == fnospec.FNO_ERR_INVALID_ARG
