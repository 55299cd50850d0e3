"""GPU parity of the permute fused into the expert GEMMs' operand loads
(moe_expert_ffn_fwd_gather, moe_expert_ffn_bwd_weights_gather).

The fused calls read row r of X_perm as x[perm[r] / k] instead of a stored
X_perm (TMA tile::gather4 loads on the tensor-core path).  They run the same
GEMMs on the same values, so they must equal the unfused calls bit for bit;
the unfused calls are checked against the oracle elsewhere, and the forward
here is also compared with the oracle (permute, then expert forward) directly.
Launch shapes as in test_gpu_ffn: CTA pairs, pairs capped at two per launch,
single CTAs."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = {"pairs": {}, "pairs_2_units": {"MOE_GEMM_MAX_UNITS": "2"},
          "single_cta": {"MOE_GEMM_PAIR": "0"}}

CASES = [  # dtype, T, d, f, E, k, zipf
    ("bf16", 1000, 256, 512, 8, 2, None),
    ("bf16", 700, 192, 320, 16, 1, 1.2),     # empty experts, partial N tiles (d = 192)
    ("bf16", 600, 128, 64, 64, 4, 1.1),
    ("bf16", 4096, 128, 256, 8, 1, 2.0),     # long K in the weight gradients
    ("f32", 333, 96, 40, 6, 2, 1.2),
]


def _routing(T, E, k, zipf, seed):
    L = synth.make_logits(T, E, seed=seed).double().numpy()
    if zipf:
        L = L + synth.zipf_logit_bias(E, zipf, 2.0).double().numpy()
    idx, _ = oracle.gate(L, k, 1 if k > 1 else 0)
    return oracle.dispatch(idx, E)   # counts, offsets, pos, perm


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("dtype,T,d,f,E,k,zipf", CASES)
def test_ffn_gather_equals_unfused(dtype, T, d, f, E, k, zipf, shape, monkeypatch):
    if dtype != "bf16" and shape != "pairs":
        pytest.skip("the launch shapes are those of the tensor-core path")
    for n, v in SHAPES[shape].items():
        monkeypatch.setenv(n, v)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rb = dtype == "bf16"
    counts, offsets, pos, perm = _routing(T, E, k, zipf, seed=T + 3 * E)
    P = T * k
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype=dtype)
    inp = synth.make_inputs(cfg, seed=E + d + 1, random_bias=True)
    g = torch.Generator().manual_seed(P + 5)
    x = torch.randn(T, d, generator=g).to(tdt)
    dY = torch.randn(P, d, generator=g).to(tdt)
    perm_t = torch.from_numpy(perm.astype(np.int64))
    X_perm = x[perm_t // k]                  # row r of X_perm = x[perm[r] / k]
    s = ops.make_shape(T, d, f, E, k, dtype, 1)
    W = {n: inp[n].to(DEV) for n in ("W1", "b1", "W2", "b2")}
    offs = torch.from_numpy(offsets).to(DEV)
    perm_d = torch.from_numpy(perm).to(DEV)
    xd, Xd, dYd = x.to(DEV), X_perm.to(DEV), dY.to(DEV)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = {}
    for name in ("unfused", "gather"):
        G = torch.empty(P, f, dtype=tdt, device=DEV)
        A = torch.empty(P, f, dtype=tdt, device=DEV)
        Y = torch.empty(P, d, dtype=tdt, device=DEV)
        if name == "gather":
            ops.moe_expert_ffn_fwd_gather(s, xd, perm_d, offs, W["W1"], W["b1"], W["W2"],
                                          W["b2"], G, A, Y, ws, st)
        else:
            ops.moe_expert_ffn_fwd(s, Xd, offs, W["W1"], W["b1"], W["W2"], W["b2"], G, A, Y,
                                   ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        out[name] = (G, A, Y)
    for n, a, b in zip("GAY", out["unfused"], out["gather"]):
        assert torch.equal(a, b), n
    # and the oracle's own permute + forward
    rX = oracle.permute(x, pos)
    rG, rA, rY = oracle.expert_ffn_fwd(rX, offsets, inp["W1"], inp["b1"], inp["W2"], inp["b2"], rb)
    for n, a, r in zip("GAY", out["gather"], (rG, rA, rY)):
        assert_close(n, a, r, dtype)

    # weight gradients over one chunk: X through perm vs X_perm
    G, A, _ = out["unfused"]
    dH = torch.empty(P, f, dtype=tdt, device=DEV)
    dX = torch.empty(P, d, dtype=tdt, device=DEV)
    db1 = torch.empty(E, f, device=DEV)
    ops.moe_expert_ffn_bwd_data(s, dYd, G, offs, W["W1"], W["W2"], dH, dX, db1, 0, ws, st)
    wn = ops.moe_expert_ffn_bwd_weights_workspace_size(s, [T])
    wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=DEV)
    res = {}
    for name in ("unfused", "gather"):
        gr = [torch.full(sh, float("nan"), device=DEV) for sh in ((E, f, d), (E, d, f), (E, d))]
        if name == "gather":
            ops.moe_expert_ffn_bwd_weights_gather(s, [T], offs[None], dYd, xd, perm_d, P, dH, A,
                                                  *gr, 0, wws, st)
        else:
            ops.moe_expert_ffn_bwd_weights(s, [T], offs[None], dYd, Xd, dH, A, *gr, 0, wws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[name] = gr
    for n, a, b in zip(("dW1", "dW2", "db2"), res["unfused"], res["gather"]):
        assert torch.equal(a, b), n


@pytest.mark.parametrize("dtype,nchunks,T,d,f,E,k", [
    ("bf16", 3, 700, 256, 384, 8, 2),
    ("bf16", 17, 90, 128, 192, 16, 3),     # 16 + 1 chunks: the second launch has one chunk
    ("bf16", 2, 40000, 128, 128, 2, 1),    # > 256 K blocks per expert: split parts
    ("f32", 4, 150, 64, 96, 6, 2),
])
def test_bwd_weights_gather_over_chunks(dtype, nchunks, T, d, f, E, k):
    """moe_expert_ffn_bwd_weights_gather over several chunks (x of all chunks
    one after the other, each chunk's perm at its stride) equals
    moe_expert_ffn_bwd_weights over the chunks' X_perm rows, bit for bit."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    s = ops.make_shape(T, d, f, E, k, dtype, 1)
    stride = (E + 1 + 3) // 4 * 4
    P = T * k
    pstride = (P + 3) // 4 * 4 + 4          # a stride wider than one chunk's perm
    offs_all = torch.zeros(nchunks, stride, dtype=torch.int32)
    perm_all = torch.full((nchunks, pstride), -1, dtype=torch.int32)
    g = torch.Generator().manual_seed(31 * nchunks + T)
    x = torch.randn(nchunks * T, d, generator=g).to(tdt)
    Xp = []
    for c in range(nchunks):
        _, offsets, _, perm = _routing(T, E, k, 1.0 + 0.1 * c, seed=200 + c)
        offs_all[c, :E + 1] = torch.from_numpy(offsets)
        perm_all[c, :P] = torch.from_numpy(perm)
        Xp.append(x[c * T + torch.from_numpy(perm.astype(np.int64)) // k])
    dY = torch.randn(nchunks * P, d, generator=g).to(tdt).to(DEV)
    dH = torch.randn(nchunks * P, f, generator=g).to(tdt).to(DEV)
    A = torch.randn(nchunks * P, f, generator=g).to(tdt).to(DEV)
    chunk_T = [T] * nchunks
    wn = ops.moe_expert_ffn_bwd_weights_workspace_size(s, chunk_T)
    wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    offs_d = offs_all.to(DEV)
    res = {}
    for name in ("unfused", "gather"):
        gr = [torch.full(sh, float("nan"), device=DEV) for sh in ((E, f, d), (E, d, f), (E, d))]
        if name == "gather":
            ops.moe_expert_ffn_bwd_weights_gather(s, chunk_T, offs_d, dY, x.to(DEV),
                                                  perm_all.to(DEV), pstride, dH, A, *gr, 0,
                                                  wws, st)
        else:
            ops.moe_expert_ffn_bwd_weights(s, chunk_T, offs_d, dY, torch.cat(Xp).to(DEV), dH, A,
                                           *gr, 0, wws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[name] = gr
    for n, a, b in zip(("dW1", "dW2", "db2"), res["unfused"], res["gather"]):
        assert torch.equal(a, b), n


@pytest.mark.parametrize("mode", ["one_chunk", "chunks_deferred", "chunks_per_chunk_wgrad",
                                  "chunks_serial", "recompute"])
def test_layer_gather_equals_unfused(mode):
    """The whole layer (forward + backward) with the permute fused into the
    GEMM loads equals the layer with moe_permute, bit for bit, in every chunking
    and weight-gradient mode (the unfused layer is checked against the oracle
    in test_gpu_layer)."""
    from mixture_experts_layer_11_gb300.layer import LayerPass
    T, d, f, E, k = 1000, 256, 384, 16, 2
    chunk = None if mode == "one_chunk" else 248
    kw = {"chunk": chunk, "device": DEV}
    if mode == "chunks_per_chunk_wgrad":
        kw["defer_wgrad"] = False
    if mode == "chunks_serial":
        kw["pipeline"] = False
    if mode == "recompute":
        kw["recompute"] = True
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype="bf16", zipf_s=1.2)
    inp = synth.make_inputs(cfg, seed=7, device=DEV)
    outs = {}
    for gather in (False, True):
        lp = LayerPass(T, d, f, E, k, torch.bfloat16, 1, gather=gather, **kw)
        y = lp.forward(inp["x"], inp["Wg"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                       inp["beta"]).clone()
        lp.backward(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W2"])
        lp.check_status()
        outs[gather] = [y] + [t.clone() for t in (lp.dx, lp.dw, lp.dW1, lp.db1, lp.dW2, lp.db2,
                                                  lp.dWg)]
    for n, a, b in zip(("y", "dx", "dw", "dW1", "db1", "dW2", "db2", "dWg"), outs[False],
                       outs[True]):
        assert torch.equal(a, b), n
