"""GPU parity of the routing steps (A1 router logits, A2 gate, A3 dispatch)
against the oracle.  Routing is compared bit-exactly on identical fp32
logits fed to both sides (the GPU's moe_route with compute_logits = 0)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close, assert_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_given(logits: torch.Tensor, k: int, renorm: int, E: int):
    T = logits.shape[0]
    s = ops.make_shape(T, 64, 64, E, k, "f32", renorm)
    L = logits.to(DEV).contiguous()
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    pos = torch.empty(T, k, dtype=torch.int32, device=DEV)
    perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=DEV)
    ws = torch.empty(max(ops.moe_workspace_size(s), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.moe_route(s, None, None, None, L, 0, idx, w, counts, offsets, pos, perm, ws, st)
    torch.cuda.synchronize()
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, pos=pos, perm=perm[:T * k],
                status=int(st.item()))


CASES = [  # T, E, k, renorm, ties
    (1, 4, 1, 0, False), (255, 8, 2, 1, False), (256, 8, 2, 1, True), (257, 4, 1, 0, True),
    (1000, 64, 1, 0, False), (3001, 128, 8, 1, False), (777, 16, 16, 1, True),
    (2048, 256, 8, 1, False), (513, 3, 3, 0, True), (4096, 32, 4, 0, False),
]


@pytest.mark.parametrize("T,E,k,renorm,ties", CASES)
def test_route_given_logits_bit_exact(T, E, k, renorm, ties):
    L = synth.make_logits(T, E, seed=T + E + k, ties=ties)
    g = _route_given(L, k, renorm, E)
    assert g["status"] == 0
    idx, w = oracle.gate(L.double().numpy(), k, renorm)
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    assert_equal("idx", g["idx"], idx)
    assert_equal("counts", g["counts"], counts)
    assert_equal("offsets", g["offsets"], offsets)
    assert_equal("pos", g["pos"], pos)
    assert_equal("perm", g["perm"], perm)
    assert_close("w", g["w"], w, "f32")


def test_route_empty():
    g = _route_given(torch.zeros(0, 8), 2, 1, 8)
    assert g["status"] == 0
    assert_equal("counts", g["counts"], np.zeros(8, np.int32))
    assert_equal("offsets", g["offsets"], np.zeros(9, np.int32))


def test_route_nonfinite_flags_and_stays_in_range():
    L = synth.make_logits(300, 16, seed=1)
    L[5, 3] = float("nan")
    L[7] = float("nan")
    L[9, 0] = float("inf")
    g = _route_given(L, 4, 1, 16)
    assert g["status"] == ops.MOE_ERR_NONFINITE
    idx = g["idx"].cpu().numpy()
    assert idx.min() >= 0 and idx.max() < 16
    for row in idx:
        assert len(set(row.tolist())) == 4
    assert int(g["offsets"][-1]) == 300 * 4


@pytest.mark.parametrize("dtype,T,d,E,zipf", [("f32", 256, 64, 4, None), ("bf16", 1000, 768, 8, None),
                                              ("bf16", 777, 256, 64, 1.2), ("bf16", 300, 4096, 128, 1.1),
                                              ("f32", 129, 200, 256, None),
                                              ("bf16", 333, 128, 5, None), ("bf16", 200, 192, 256, None)])
def test_router_logits(dtype, T, d, E, zipf):
    cfg = synth.MoEConfig("t", T=T, d=d, f=64, E=E, k=1, renorm=0, dtype=dtype, zipf_s=zipf)
    inp = synth.make_inputs(cfg, seed=3)
    ref = oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])
    s = ops.make_shape(T, d, 64, E, 1, dtype, 0)
    x, Wg = inp["x"].to(DEV), inp["Wg"].to(DEV)
    beta = None if inp["beta"] is None else inp["beta"].to(DEV)
    logits = torch.empty(T, E, dtype=torch.float32, device=DEV)
    idx = torch.empty(T, 1, dtype=torch.int32, device=DEV)
    w = torch.empty(T, 1, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    pos = torch.empty(T, 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T, dtype=torch.int32, device=DEV)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.moe_route(s, x, Wg, beta, logits, 1, idx, w, counts, offsets, pos, perm, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # logits are fp32 outputs in both configurations
    assert_close("logits", logits, ref, "f32")


def test_route_deterministic():
    L = synth.make_logits(5000, 64, seed=9, ties=True)
    a = _route_given(L, 4, 1, 64)
    b = _route_given(L, 4, 1, 64)
    for n in ("idx", "w", "counts", "offsets", "pos", "perm"):
        assert torch.equal(a[n], b[n]), n
