"""GPU parity of the router backward (A10) against the oracle, with the
permute backward (A9) fused in (dx = sum_j dX_perm[pos] + router term) and
without it (dx += router term).  Routing, positions and the fp32 logits come
from the oracle on both sides."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [("f32", 256, 64, 4, 1, 0), ("bf16", 1000, 768, 8, 2, 1), ("bf16", 777, 256, 64, 1, 0),
         ("bf16", 513, 512, 128, 8, 1), ("f32", 300, 96, 16, 4, 0),
         ("bf16", 333, 200, 40, 3, 0), ("f32", 129, 136, 72, 2, 0)]


@pytest.mark.parametrize("dtype,T,d,E,k,renorm", CASES)
@pytest.mark.parametrize("fused", [True, False])
def test_route_bwd(dtype, T, d, E, k, renorm, fused):
    cfg = synth.MoEConfig("t", T=T, d=d, f=64, E=E, k=k, renorm=renorm, dtype=dtype)
    inp = synth.make_inputs(cfg, seed=T + E)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"])).float()
    _check(cfg, inp, L, fused)


@pytest.mark.parametrize("zipf", [None, 1.2])
def test_route_bwd_large_source(zipf):
    """x of 64 MB (T = 8192, d = 4096, bf16), beyond what L2 keeps: dWg sums
    its gathered rows in token-window pieces of every expert's segment.  With
    a Zipf logit shift the hot experts' pieces are long and some experts get
    no rows (empty pieces).  Seeded logits stand in for x Wg^T (the backward
    only needs the same logits on both sides)."""
    T, d, E, k = 8192, 4096, 128, 8
    cfg = synth.MoEConfig("t", T=T, d=d, f=64, E=E, k=k, renorm=1, dtype="bf16")
    inp = synth.make_inputs(cfg, seed=17)
    L = synth.make_logits(T, E, seed=19).float()
    if zipf:
        L = L + synth.zipf_logit_bias(E, zipf, 2.0).float()
    _check(cfg, inp, L, True)


def _check(cfg, inp, L, fused):
    dtype, T, d, E, k, renorm = cfg.dtype, cfg.T, cfg.d, cfg.E, cfg.k, cfg.renorm
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rb = dtype == "bf16"
    idx, w = oracle.gate(L.double().numpy(), k, renorm)
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    g = torch.Generator().manual_seed(T)
    dw = torch.randn(T, k, generator=g, dtype=torch.float32)
    dXp = torch.randn(T * k, d, generator=g, dtype=torch.float32).to(tdt)
    dx0 = torch.randn(T, d, generator=g, dtype=torch.float32).to(tdt)
    w32 = w.astype(np.float32)
    _, dxr, rdWg = oracle.router_bwd(dw, L.double().numpy(), idx, w32, inp["x"], inp["Wg"], renorm)
    if fused:
        ref_dx = oracle.combine(dXp, pos, None, False) + dxr
    else:
        ref_dx = dx0.double().numpy() + dxr
    if rb:
        ref_dx = oracle.round_bf16_array(ref_dx)
    s = ops.make_shape(T, d, 64, E, k, dtype, renorm)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).to(DEV)  # noqa: E731
    dx = dx0.clone().to(DEV)
    dWg = torch.full((E, d), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.moe_route_bwd(s, dw.to(DEV), L.to(DEV), t(idx, torch.int32), t(w32, torch.float32),
                      t(perm, torch.int32), t(offsets, torch.int32), inp["x"].to(DEV),
                      inp["Wg"].to(DEV), dXp.to(DEV) if fused else None,
                      t(pos, torch.int32) if fused else None, dx, dWg, 0, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("dx", dx, ref_dx, dtype)
    # dWg is an fp32 output: sums of exact products of stored values
    assert_close("dWg", dWg, rdWg, "f32", rel=1e-5 if dtype == "f32" else 1e-4)
