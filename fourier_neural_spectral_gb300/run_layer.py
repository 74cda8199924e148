"""Run the spectral-convolution layer on one shape a few times (for profilers).

    python -m fourier_neural_spectral_gb300.run_layer B Cin Cout H W m1 m2 REPS [fp32|tf32|3xtf32]

Inputs are seeded normal draws made on the device; the call goes through the
C ABI (fno_plan_execute) and the device error word is checked at the end.
"""
import sys

import torch

from . import fnospec


def main(argv):
    if len(argv) not in (8, 9):
        print(__doc__)
        return 2
    B, Cin, Cout, H, W, m1, m2, reps = map(int, argv[:8])
    prec = argv[8] if len(argv) == 9 else "fp32"
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(B, Cin, H, W, device="cuda", generator=g)
    w = torch.randn(Cin, Cout, 2 * m1, m2, 2, device="cuda", generator=g) * 0.1
    y = torch.empty(B, Cout, H, W, device="cuda")
    plan = fnospec.Plan(B, Cin, Cout, H, W, m1, m2, precision=prec)
    print(plan.description)
    for _ in range(reps):
        plan.fno_plan_execute(x, w, y)
    torch.cuda.synchronize()
    status = plan.fno_get_device_status()
    print("device status", status, "max|y|", float(y.abs().max()))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
