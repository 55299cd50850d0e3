"""GPU parity of the permute (A4), combine (A6), combine backward (A7) and
permute backward (A9) kernels against the oracle, with the positions taken
from the oracle's own dispatch of a seeded routing."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close, assert_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _routing(T, E, k, renorm, seed):
    L = synth.make_logits(T, E, seed=seed)
    idx, w = oracle.gate(L.double().numpy(), k, renorm)
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    return idx, w, offsets, pos, perm


def _tensor(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).to(DEV)


CASES = [("bf16", 1000, 768, 8, 2), ("f32", 256, 64, 4, 1), ("bf16", 777, 4096, 128, 8),
         ("bf16", 33, 256, 16, 16), ("f32", 1025, 200, 32, 3)]


@pytest.mark.parametrize("dtype,T,d,E,k", CASES)
def test_permute_combine_and_backward(dtype, T, d, E, k):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rb = dtype == "bf16"
    idx, w, offsets, pos, perm = _routing(T, E, k, 1, seed=T + d)
    g = torch.Generator().manual_seed(T)
    x = torch.randn(T, d, generator=g, dtype=torch.float32).to(tdt)
    Y = torch.randn(T * k, d, generator=g, dtype=torch.float32).to(tdt)
    dy = torch.randn(T, d, generator=g, dtype=torch.float32).to(tdt)
    s = ops.make_shape(T, d, 64, E, k, dtype, 1)
    pos_d = _tensor(pos, torch.int32)
    w32 = w.astype(np.float32)
    w_d = _tensor(w32, torch.float32)
    # A4
    xp = torch.empty(T * k, d, dtype=tdt, device=DEV)
    ops.moe_permute(s, x.to(DEV), pos_d, xp)
    assert_equal("x_perm", xp.cpu().to(torch.float32).numpy(),
                 oracle.permute(x, pos).astype(np.float32))
    # A6 (the same fp32 gate weights on both sides)
    y = torch.empty(T, d, dtype=tdt, device=DEV)
    ops.moe_combine_fwd(s, Y.to(DEV), pos_d, w_d, y)
    assert_close("y", y, oracle.combine(Y, pos, w32, rb), dtype)
    # A9 (unweighted)
    ops.moe_combine_fwd(s, Y.to(DEV), pos_d, None, y)
    assert_close("dx_perm_sum", y, oracle.combine(Y, pos, None, rb), dtype)
    # A7
    dY = torch.empty(T * k, d, dtype=tdt, device=DEV)
    dw = torch.empty(T, k, dtype=torch.float32, device=DEV)
    ops.moe_combine_bwd(s, dy.to(DEV), Y.to(DEV), pos_d, w_d, dY, dw)
    rdY, rdw = oracle.combine_bwd(dy, Y, pos, w32, rb)
    assert_close("dY_perm", dY, rdY, dtype)
    # dw is an fp32 output: exact products of the stored values, fp32 sums
    assert_close("dw", dw, rdw, "f32", rel=1e-5 if dtype == "f32" else 1e-4)
    torch.cuda.synchronize()
