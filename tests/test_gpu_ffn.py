"""GPU parity of the grouped expert FFN, forward (A5) and backward (A8),
against the oracle: tcgen05 tensor-core path for bf16, CUDA-core path for
fp32.  Segments come from the oracle's dispatch of a seeded routing and
include empty experts, ragged segment ends and partial N / K tiles.

The bf16 cases run in three launch shapes: CTA pairs with the full grid;
CTA pairs capped at two per launch (MOE_GEMM_MAX_UNITS=2), so that each pair
walks many tiles of the static tile list and the epilogue's cross-tile state
(bias and GELU' operands streamed one tile ahead, the GELU' ring) is used
at every tile boundary; and single CTAs (MOE_GEMM_PAIR=0)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _segments(T, E, k, zipf, seed):
    L = synth.make_logits(T, E, seed=seed).double().numpy()
    if zipf:
        L = L + synth.zipf_logit_bias(E, zipf, 2.0).double().numpy()
    idx, _ = oracle.gate(L, k, 1 if k > 1 else 0)
    counts, offsets, _, _ = oracle.dispatch(idx, E)
    return counts, offsets


CASES = [  # dtype, T, d, f, E, k, zipf
    ("bf16", 1000, 256, 512, 8, 2, None),
    ("bf16", 700, 192, 320, 16, 1, 1.2),     # empty experts, partial N tiles
    ("bf16", 2048, 768, 1024, 4, 2, None),
    ("bf16", 600, 128, 64, 64, 4, 1.1),
    ("bf16", 4096, 128, 256, 8, 1, 2.0),     # one expert takes most rows: long K in wgrad
    ("f32", 256, 64, 128, 4, 1, None),
    ("f32", 333, 96, 40, 6, 2, 1.2),
]


SHAPES = {"pairs": {}, "pairs_2_units": {"MOE_GEMM_MAX_UNITS": "2"},
          "single_cta": {"MOE_GEMM_PAIR": "0"}}


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("dtype,T,d,f,E,k,zipf", CASES)
def test_expert_ffn_fwd_bwd(dtype, T, d, f, E, k, zipf, shape, monkeypatch):
    if dtype != "bf16" and shape != "pairs":
        pytest.skip("the launch shapes are those of the tensor-core path")
    for n, v in SHAPES[shape].items():
        monkeypatch.setenv(n, v)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rb = dtype == "bf16"
    counts, offsets = _segments(T, E, k, zipf, seed=T * 7 + E)
    P = T * k
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype=dtype)
    inp = synth.make_inputs(cfg, seed=E + d, random_bias=True)
    g = torch.Generator().manual_seed(P)
    X = torch.randn(P, d, generator=g, dtype=torch.float32).to(tdt)
    dY = torch.randn(P, d, generator=g, dtype=torch.float32).to(tdt)
    s = ops.make_shape(T, d, f, E, k, dtype, 1)
    dev = {n: inp[n].to(DEV) for n in ("W1", "b1", "W2", "b2")}
    offs = torch.from_numpy(offsets).to(DEV)
    Xd, dYd = X.to(DEV), dY.to(DEV)
    G = torch.empty(P, f, dtype=tdt, device=DEV)
    A = torch.empty(P, f, dtype=tdt, device=DEV)
    Y = torch.empty(P, d, dtype=tdt, device=DEV)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.moe_expert_ffn_fwd(s, Xd, offs, dev["W1"], dev["b1"], dev["W2"], dev["b2"], G, A, Y, ws, st)
    rG, rA, rY = oracle.expert_ffn_fwd(X, offsets, inp["W1"], inp["b1"], inp["W2"], inp["b2"], rb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("G", G, rG, dtype)
    assert_close("A", A, rA, dtype)
    assert_close("Y", Y, rY, dtype)

    dX = torch.empty(P, d, dtype=tdt, device=DEV)
    grads = {n: torch.full(sh, float("nan"), dtype=torch.float32, device=DEV) for n, sh in
             (("dW1", (E, f, d)), ("db1", (E, f)), ("dW2", (E, d, f)), ("db2", (E, d)))}
    ops.moe_expert_ffn_bwd(s, dYd, Xd, G, A, offs, dev["W1"], dev["W2"], dX, grads["dW1"],
                           grads["db1"], grads["dW2"], grads["db2"], 0, ws, st)
    # oracle backward from the oracle's own forward activations
    _, rdX, rdW1, rdb1, rdW2, rdb2 = oracle.expert_ffn_bwd(dY, X, rG, rA, offsets, inp["W1"],
                                                           inp["W2"], rb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close("dX_perm", dX, rdX, dtype)
    for n, r in (("dW1", rdW1), ("db1", rdb1), ("dW2", rdW2), ("db2", rdb2)):
        assert_close(n, grads[n], r, dtype)
    # experts without tokens get exact zeros
    for e in np.flatnonzero(counts == 0):
        assert float(grads["dW1"][e].abs().max()) == 0.0
        assert float(grads["db2"][e].abs().max()) == 0.0
    # accumulate: a second identical pass doubles every gradient exactly
    first = {n: t.clone() for n, t in grads.items()}
    ops.moe_expert_ffn_bwd(s, dYd, Xd, G, A, offs, dev["W1"], dev["W2"], dX, grads["dW1"],
                           grads["db1"], grads["dW2"], grads["db2"], 1, ws, st)
    torch.cuda.synchronize()
    for n in grads:
        assert torch.equal(grads[n], 2 * first[n]), n


@pytest.mark.parametrize("dtype,nchunks,T,d,f,E,k", [
    ("bf16", 3, 700, 256, 384, 8, 2),
    ("bf16", 19, 100, 128, 192, 16, 3),    # more chunks than one launch walks: two launches
    ("f32", 4, 150, 64, 96, 6, 2),
])
def test_expert_ffn_bwd_data_and_weights_over_chunks(dtype, nchunks, T, d, f, E, k):
    """moe_expert_ffn_bwd_data per chunk, then moe_expert_ffn_bwd_weights over
    all chunks in one call, against the oracle's per-chunk backward with the
    weight gradients accumulated over the chunks."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rb = dtype == "bf16"
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype=dtype)
    inp = synth.make_inputs(cfg, seed=E + nchunks, random_bias=True)
    W = {n: inp[n].to(DEV) for n in ("W1", "b1", "W2", "b2")}
    s = ops.make_shape(T, d, f, E, k, dtype, 1)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    P = T * k
    stride = (E + 1 + 3) // 4 * 4
    offs_all = torch.zeros(nchunks, stride, dtype=torch.int32)
    g = torch.Generator().manual_seed(nchunks)
    X_all, dY_all, G_all, A_all, dH_all = [], [], [], [], []
    grads = None
    db1_dev = torch.full((E, f), float("nan"), device=DEV)
    dX_dev = torch.empty(P, d, dtype=tdt, device=DEV)
    for c in range(nchunks):
        # chunk c's routing: Zipf-shifted logits, a different shift per chunk
        counts, offsets = _segments(T, E, k, 1.0 + 0.1 * c, seed=100 + c)
        offs_all[c, :E + 1] = torch.from_numpy(offsets)
        X = torch.randn(P, d, generator=g).to(tdt)
        dY = torch.randn(P, d, generator=g).to(tdt)
        rG, rA, _ = oracle.expert_ffn_fwd(X, offsets, inp["W1"], inp["b1"], inp["W2"], inp["b2"], rb)
        res = oracle.expert_ffn_bwd(dY, X, rG, rA, offsets, inp["W1"], inp["W2"], rb, grads)
        grads = dict(zip(("dW1", "db1", "dW2", "db2"), res[2:]))
        G = torch.from_numpy(rG).to(tdt).to(DEV)
        dH = torch.empty(P, f, dtype=tdt, device=DEV)
        ops.moe_expert_ffn_bwd_data(s, dY.to(DEV), G, offs_all[c, :E + 1].to(DEV), W["W1"],
                                    W["W2"], dH, dX_dev, db1_dev, int(c > 0), ws, st)
        torch.cuda.synchronize()
        assert_close(f"dX_perm[{c}]", dX_dev, res[1], dtype)
        X_all.append(X)
        dY_all.append(dY)
        A_all.append(torch.from_numpy(rA).to(tdt))
        dH_all.append(dH)
    dW1 = torch.full((E, f, d), float("nan"), device=DEV)
    dW2 = torch.full((E, d, f), float("nan"), device=DEV)
    db2 = torch.full((E, d), float("nan"), device=DEV)
    ops.moe_expert_ffn_bwd_weights(s, [T] * nchunks, offs_all.to(DEV), torch.cat(dY_all).to(DEV),
                                   torch.cat(X_all).to(DEV), torch.cat(dH_all),
                                   torch.cat(A_all).to(DEV), dW1, dW2, db2, 0, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for n, t in (("dW1", dW1), ("db1", db1_dev), ("dW2", dW2), ("db2", db2)):
        assert_close(n, t, grads[n], dtype)


_WIDE_CACHE = {}


def _wide_case(nchunks, T, E, k):
    """Inputs of test_weights_wide_tiles and the oracle's weight gradients,
    computed once per routing case (the oracle's backward of d = f = 1024 is
    the slow part)."""
    key = (nchunks, T, E, k)
    if key in _WIDE_CACHE:
        return _WIDE_CACHE[key]
    d = f = 1024
    tdt = torch.bfloat16
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype="bf16")
    inp = synth.make_inputs(cfg, seed=E + nchunks + T, random_bias=True)
    P = T * k
    stride = (E + 1 + 3) // 4 * 4
    offs_all = torch.zeros(nchunks, stride, dtype=torch.int32)
    g = torch.Generator().manual_seed(T + nchunks)
    Xs, dYs, dHs, As = [], [], [], []
    grads = None
    for c in range(nchunks):
        _, offsets = _segments(T, E, k, 1.0 + 0.2 * c, seed=300 + c)
        offs_all[c, :E + 1] = torch.from_numpy(offsets)
        X = torch.randn(P, d, generator=g).to(tdt)
        dY = torch.randn(P, d, generator=g).to(tdt)
        G = torch.rand(P, f, generator=g).to(tdt)
        A = torch.randn(P, f, generator=g).to(tdt)
        # the oracle's backward of this chunk (dH = (dY W2) * G, stored in
        # bf16), its weight gradients accumulated over the chunks; the GPU's
        # weight pass gets the oracle's dH
        res = oracle.expert_ffn_bwd(dY, X, G, A, offsets, inp["W1"], inp["W2"], True, grads)
        grads = dict(zip(("dW1", "db1", "dW2", "db2"), res[2:]))
        Xs.append(X); dYs.append(dY); As.append(A)
        dHs.append(torch.from_numpy(res[0]).to(tdt))
    case = (offs_all, [torch.cat(t) for t in (dYs, Xs, dHs, As)], grads)
    _WIDE_CACHE[key] = case
    return case


@pytest.mark.parametrize("units", [None, "20", "17"])
@pytest.mark.parametrize("nchunks,T,E,k", [(2, 600, 4, 2), (2, 9000, 1, 1)])
def test_weights_wide_tiles(nchunks, T, E, k, units, monkeypatch):
    """Weight gradients of d = f = 1024 (4 x 4 tiles of 256 x 256 per expert)
    over two chunks, on all pairs and with the pairs capped at 20 and 17,
    against the oracle.  The second case has one expert of 18000 rows over
    the chunks: 282 K blocks, split into two parts."""
    if units:
        monkeypatch.setenv("MOE_GEMM_MAX_UNITS", units)
    d = f = 1024
    offs_all, data, grads = _wide_case(nchunks, T, E, k)
    s = ops.make_shape(T, d, f, E, k, "bf16", 1)
    chunk_T = [T] * nchunks
    wn = ops.moe_expert_ffn_bwd_weights_workspace_size(s, chunk_T)
    wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = [torch.full(sh, float("nan"), device=DEV) for sh in ((E, f, d), (E, d, f), (E, d))]
    ops.moe_expert_ffn_bwd_weights(s, chunk_T, offs_all.to(DEV), *[t.to(DEV) for t in data],
                                   *out, 0, wws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for n, t in zip(("dW1", "dW2", "db2"), out):
        assert_close(n, t, grads[n], "bf16")
