"""The bf16 epilogue's fast GELU / GELU' (erf from Abramowitz & Stegun 7.1.26,
|erf error| <= 1.5e-7) and the fp32 path's erff form, evaluated on the GPU
by the library, against the oracle's double-precision GELU.

Bound for the fast form: |dPhi| <= 0.75e-7 (approximation) plus a few fp32
roundings of values <= 1, so |dGELU| = |x| |dPhi| and |dGELU'| stay below
1e-6 * max(1, |x|) -- four orders of magnitude under bf16 spacing."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fast", [1, 0])
def test_gelu_against_oracle(fast):
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.linspace(-10, 10, 40001), torch.randn(20000, generator=g) * 3,
                   torch.tensor([0.0, -0.0, 1e-30, -1e-30, 5.0, -5.0])]).float()
    xd = x.cuda()
    out = torch.empty_like(xd)
    outg = torch.empty_like(xd)
    ops.moe_debug_gelu(xd, out, outg, fast)
    torch.cuda.synchronize()
    xs = x.double().numpy()
    ref = np.array([oracle.gelu(v) for v in xs])
    refg = np.array([oracle.gelu_grad(v) for v in xs])
    scale = np.maximum(1.0, np.abs(xs))
    err = np.abs(out.double().cpu().numpy() - ref) / scale
    errg = np.abs(outg.double().cpu().numpy() - refg) / scale
    assert err.max() <= 1e-6, err.max()
    assert errg.max() <= 1e-6, errg.max()
    # GELU(0) = 0 exactly, GELU'(0) = 1/2 to fp32 accuracy
    assert float(out[-6]) == 0.0
    assert abs(float(outg[-6]) - 0.5) <= 1e-7
