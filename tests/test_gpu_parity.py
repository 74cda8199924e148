"""Parity of the CUDA path (through the C ABI) with the double-precision oracle
on the five seeded workloads, stage by stage and end to end."""
import numpy as np
import pytest

import oracle
from fourier_neural_spectral_gb300 import synth

from gpu_helpers import (assert_fp32_close, cplx_to_f32pairs, errors, f32pairs_to_cplx,
                         run_layer, to_dev)

pytestmark = pytest.mark.gpu

SMALL = ["B2_C4_16x16_m4", "B8_C32_64x64_m16_smooth", "B16_C64_128x128_m32"]


def oracle_layer_threaded(cfg, x, w):
    X = oracle.forward_modes_parallel(x, cfg.m1, cfg.m2)
    Z = oracle.mix_modes(X, f32pairs_to_cplx(w))
    return oracle.inverse_modes_parallel(Z, cfg.H, cfg.W)


@pytest.mark.parametrize("name", SMALL + ["B4_C128_256x256_m64"])
def test_layer_matches_oracle_elementwise(cuda_lib, name):
    cfg = synth.CONFIGS[name]
    x, w = synth.make_inputs(cfg)
    y, plan = run_layer(x, w, cfg.m1, cfg.m2)
    ref = oracle_layer_threaded(cfg, x, w)
    rel, mx = assert_fp32_close(y, ref, name)
    print(f"{name}: {plan.description} rel-L2 {rel:.2e} max-abs {mx:.2e}")


def test_2048_grid_full_layer_and_forward_stage(cuda_lib):
    """Full 2048x2048 workload: the forward stage and the whole layer output are
    compared with the oracle element by element over the full tensors (the
    oracle's planes run on host threads), plus corner and edge points of y
    against the oracle's pointwise inverse."""
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    cfg = synth.CONFIGS["B2_C32_2048x2048_m64"]
    x, w = synth.make_inputs(cfg)
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2, "fp32")
    xt, wt = to_dev(x), to_dev(w)
    Xt = torch.empty((cfg.B, cfg.Cin, 2 * cfg.m1, cfg.m2, 2), dtype=torch.float32, device="cuda")
    plan.fno_forward_modes(xt, Xt)
    yt = torch.empty((cfg.B, cfg.Cout, cfg.H, cfg.W), dtype=torch.float32, device="cuda")
    plan.fno_plan_execute(xt, wt, yt)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    X_ref = oracle.forward_modes_parallel(x, cfg.m1, cfg.m2)
    assert_fp32_close(f32pairs_to_cplx(Xt.cpu().numpy()), X_ref, "forward stage")
    Z_ref = oracle.mix_modes(X_ref, f32pairs_to_cplx(w))
    del X_ref
    y = yt.cpu().numpy()
    # whole output: the same two bounds as every fp32 case, accumulated over
    # the batch rows so that only one row's double copies are alive at a time
    num = den = 0.0
    dmax = rmax = 0.0
    for b in range(cfg.B):
        ref_b = oracle.inverse_modes_parallel(Z_ref[b:b + 1], cfg.H, cfg.W)[0]
        d = y[b].astype(np.float64) - ref_b
        num += float(np.vdot(d, d).real)
        den += float(np.vdot(ref_b, ref_b).real)
        dmax = max(dmax, float(np.abs(d).max()))
        rmax = max(rmax, float(np.abs(ref_b).max()))
        del d, ref_b
    rel, mx = (num / den) ** 0.5, dmax / rmax
    print(f"2048x2048 layer: rel-L2 {rel:.2e} max-abs {mx:.2e}")
    assert rel <= 1e-5 and mx <= 1e-4, (rel, mx)
    # corners and edges once more through the oracle's pointwise inverse (an
    # independent evaluation of the same sums)
    idx = np.array([[0, 0, 0, 0], [0, 1, 0, cfg.W - 1], [1, 2, cfg.H - 1, 0],
                    [1, cfg.Cout - 1, cfg.H - 1, cfg.W - 1], [0, 5, cfg.H // 2, cfg.W // 2],
                    [1, 7, 1, 1], [0, 9, cfg.H - 2, 3], [1, 11, 7, cfg.W - 5]])
    ref = oracle.inverse_modes_at(Z_ref, cfg.H, cfg.W, idx)
    got = y[tuple(idx.T)]
    assert np.abs(got - ref).max() <= 1e-4 * rmax


@pytest.mark.parametrize("name", SMALL)
def test_forward_stage_matches_oracle(cuda_lib, name):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    cfg = synth.CONFIGS[name]
    x = synth.make_x(cfg)
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
    Xt = torch.empty((cfg.B, cfg.Cin, 2 * cfg.m1, cfg.m2, 2), dtype=torch.float32, device="cuda")
    plan.fno_forward_modes(to_dev(x), Xt)
    torch.cuda.synchronize()
    assert_fp32_close(f32pairs_to_cplx(Xt.cpu().numpy()), oracle.forward_modes(x, cfg.m1, cfg.m2),
                      name)


@pytest.mark.parametrize("name", SMALL + ["B4_C128_256x256_m64"])
def test_mix_stage_matches_oracle(cuda_lib, name):
    """Same seeded spectrum X fed to both sides (drawn from the generator)."""
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    cfg = synth.CONFIGS[name]
    Xf = synth.normal_f32((cfg.B, cfg.Cin, 2 * cfg.m1, cfg.m2, 2), seed=11, stream=5)
    w = synth.make_w(cfg)
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
    Zt = torch.empty((cfg.B, cfg.Cout, 2 * cfg.m1, cfg.m2, 2), dtype=torch.float32, device="cuda")
    plan.fno_mix_modes(to_dev(Xf), to_dev(w), Zt)
    torch.cuda.synchronize()
    ref = oracle.mix_modes(f32pairs_to_cplx(Xf), f32pairs_to_cplx(w))
    assert_fp32_close(f32pairs_to_cplx(Zt.cpu().numpy()), ref, name)


@pytest.mark.parametrize("name", SMALL)
def test_inverse_stage_matches_oracle(cuda_lib, name):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    cfg = synth.CONFIGS[name]
    Zf = synth.normal_f32((cfg.B, cfg.Cout, 2 * cfg.m1, cfg.m2, 2), seed=12, stream=6)
    plan = fnospec.Plan(cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1, cfg.m2)
    yt = torch.empty((cfg.B, cfg.Cout, cfg.H, cfg.W), dtype=torch.float32, device="cuda")
    plan.fno_inverse_modes(to_dev(Zf), yt)
    torch.cuda.synchronize()
    ref = oracle.inverse_modes(f32pairs_to_cplx(Zf), cfg.H, cfg.W)
    assert_fp32_close(yt.cpu().numpy(), ref, name)


def test_one_shot_equals_plan_and_is_deterministic(cuda_lib):
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    cfg = synth.CONFIGS["B8_C32_64x64_m16_smooth"]
    x, w = synth.make_inputs(cfg)
    y1, plan = run_layer(x, w, cfg.m1, cfg.m2)
    y2, _ = run_layer(x, w, cfg.m1, cfg.m2, plan=plan)
    xt, wt = to_dev(x), to_dev(w)
    y3 = torch.empty_like(torch.from_numpy(y1)).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fnospec.fno_spectral_conv2d(xt, wt, y3, cfg.B, cfg.Cin, cfg.Cout, cfg.H, cfg.W, cfg.m1,
                                    cfg.m2)
    s.synchronize()
    assert np.array_equal(y1, y2)
    assert np.array_equal(y1, y3.cpu().numpy())
