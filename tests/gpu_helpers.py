"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle in double on the host."""
from __future__ import annotations

import numpy as np

# Tolerances of the fp32 path (relative L2 over the whole tensor, and max-abs
# relative to the largest reference magnitude) and of the TF32 tensor path.
FP32_REL_L2 = 1e-5
FP32_MAX_ABS = 1e-4
TF32_REL_L2 = 3e-3


def errors(got, ref):
    if np.iscomplexobj(ref) or np.iscomplexobj(got):
        got = np.asarray(got, dtype=np.complex128)
        ref = np.asarray(ref, dtype=np.complex128)
    else:
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    nref = np.linalg.norm(ref.ravel())
    rel = np.linalg.norm(d.ravel()) / (nref if nref > 0 else 1.0)
    mref = np.abs(ref).max() if ref.size else 0.0
    mx = np.abs(d).max() / (mref if mref > 0 else 1.0) if ref.size else 0.0
    return float(rel), float(mx)


def assert_fp32_close(got, ref, what=""):
    rel, mx = errors(got, ref)
    assert rel <= FP32_REL_L2 and mx <= FP32_MAX_ABS, f"{what}: rel-L2 {rel:.3e}, max-abs {mx:.3e}"
    return rel, mx


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def cplx_to_f32pairs(a):
    a = np.asarray(a, dtype=np.complex64)
    return np.ascontiguousarray(a).view(np.float32).reshape(a.shape + (2,))


def f32pairs_to_cplx(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a.view(np.complex64)[..., 0]


def run_layer(x, w, m1, m2, precision="fp32", plan=None):
    """y = layer(x, w) through fno_plan_execute; x float32 [B,Cin,H,W], w float32
    [Cin,Cout,2m1,m2,2].  Returns (y numpy float32, plan)."""
    import torch
    from fourier_neural_spectral_gb300 import fnospec
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    if plan is None:
        plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, precision)
    xt, wt = to_dev(x), to_dev(w)
    yt = torch.empty((B, Cout, H, W), dtype=torch.float32, device="cuda")
    plan.fno_plan_execute(xt, wt, yt)
    torch.cuda.synchronize()
    assert plan.fno_get_device_status() == fnospec.FNO_OK
    return yt.cpu().numpy(), plan


def rand_layer_inputs(rng, B, Cin, Cout, H, W, m1, m2):
    x = rng.standard_normal((B, Cin, H, W)).astype(np.float32)
    w = (rng.random((Cin, Cout, 2 * m1, m2, 2)) / (Cin * Cout)).astype(np.float32)
    return x, w
