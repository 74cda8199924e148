"""The tcgen05 tensor-core contraction (precision "tf32" and "3xtf32") against
the oracle: stage a3 alone on seeded spectra, and the whole layer."""
import numpy as np
import pytest

import oracle
from fourier_neural_spectral_gb300 import synth

from gpu_helpers import FP32_MAX_ABS, TF32_REL_L2, errors, f32pairs_to_cplx, run_layer, to_dev

pytestmark = pytest.mark.gpu

# tolerance of the split-TF32 path: fp32-level (both bounds of the fp32 path:
# relative L2 and max-abs relative to the largest reference magnitude)
SPLIT_REL_L2 = 1e-5
SPLIT_MAX_ABS = FP32_MAX_ABS

MIX_SHAPES = [
    # B, Cin, Cout, m1, m2, kernel: the weight-in-TMEM kernel (mix_tcm) serves
    # batches up to 16, the shared-memory-operand kernel (mix_tc) larger ones
    (1, 32, 32, 1, 2, "mix_tcm"),      # one CTA, 4 of its 8 modes, batch padded 1 -> 8
    (16, 64, 64, 4, 4, "mix_tcm"),     # the 128x128 workload's channel/batch shape
    (4, 128, 128, 2, 4, "mix_tcm"),    # two channel blocks, batch padded 4 -> 8
    (3, 40, 100, 3, 2, "mix_tcm"),     # ragged Cin (last chunk partial) and Cout (partial block)
    (9, 48, 72, 3, 3, "mix_tcm"),      # batch padded 9 -> 16, 18 modes (partial mode block)
    (16, 64, 64, 32, 32, "mix_tcm"),   # the whole 128x128 contraction (2048 modes)
    (32, 64, 64, 1, 2, "mix_tc"),      # largest batch handled (shared-memory operands)
]


def mix_case(B, Cin, Cout, m1, m2, precision):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    H = 2
    while H < 2 * m1:
        H *= 2
    W = 2
    while W // 2 + 1 < m2:
        W *= 2
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, precision)
    X = synth.normal_f32((B, Cin, 2 * m1, m2, 2), seed=21, stream=7)
    w = synth.uniform_f32((Cin, Cout, 2 * m1, m2, 2), scale=1.0 / (Cin * Cout), seed=21, stream=8)
    Zt = torch.empty((B, Cout, 2 * m1, m2, 2), dtype=torch.float32, device="cuda")
    plan.fno_mix_modes(to_dev(X), to_dev(w), Zt)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    ref = oracle.mix_modes(f32pairs_to_cplx(X), f32pairs_to_cplx(w))
    return errors(f32pairs_to_cplx(Zt.cpu().numpy()), ref), plan


@pytest.mark.parametrize("shape", MIX_SHAPES)
def test_tc_mix_stage_tf32(cuda_lib, shape):
    (rel, mx), plan = mix_case(*shape[:5], "tf32")
    assert f"{shape[5]}_tf32" in plan.description, plan.description
    assert rel <= TF32_REL_L2, rel


@pytest.mark.parametrize("shape", MIX_SHAPES)
def test_tc_mix_stage_split_tf32(cuda_lib, shape):
    (rel, mx), plan = mix_case(*shape[:5], "3xtf32")
    assert f"{shape[5]}_3xtf32" in plan.description, plan.description
    assert rel <= SPLIT_REL_L2 and mx <= SPLIT_MAX_ABS, (rel, mx)


@pytest.mark.parametrize("name", ["B8_C32_64x64_m16_smooth", "B16_C64_128x128_m32",
                                  "B4_C128_256x256_m64"])
@pytest.mark.parametrize("precision", ["tf32", "3xtf32"])
def test_tc_layer_matches_oracle(cuda_lib, name, precision):
    from test_gpu_parity import oracle_layer_threaded
    cfg = synth.CONFIGS[name]
    x, w = synth.make_inputs(cfg)
    y, plan = run_layer(x, w, cfg.m1, cfg.m2, precision)
    assert "mix_tc" in plan.description
    ref = oracle_layer_threaded(cfg, x, w)
    rel, mx = errors(y, ref)
    print(f"{name} {precision}: rel-L2 {rel:.2e} max-abs {mx:.2e}")
    if precision == "tf32":
        assert rel <= TF32_REL_L2, rel
    else:
        assert rel <= SPLIT_REL_L2 and mx <= SPLIT_MAX_ABS, (rel, mx)


def test_small_channels_use_fma_even_in_tc_mode(cuda_lib):
    from fourier_neural_spectral_gb300 import fnospec
    plan = fnospec.Plan(2, 4, 4, 16, 16, 4, 4, "tf32")
    assert "mix_tc" not in plan.description
