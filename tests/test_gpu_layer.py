"""Whole-layer GPU parity (A1-A10 through the C ABI, as the benchmark runs
it) against the oracle, on each workload family at sizes the oracle
finishes in seconds (several tiles, ragged tails, dispatch chunks).

Two modes:
  * identical logits (compute_logits = 0, the oracle's logits rounded to
    fp32 given to both sides): every output, bit-exact routing;
  * own logits (compute_logits = 1): logits within fp32 tolerance, routing
    identical on every token whose top-k margin exceeds the logit error,
    and per-token y and dx within tolerance on those tokens."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import synth
from mixture_experts_layer_11_gb300.layer import LayerPass
from parity_util import assert_close, assert_equal, to_dev, topk_margin

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = {
    "tiny_f32": dict(),
    "moe_s_bf16": dict(T=1000, d=256, f=512),
    "skewed64_bf16": dict(T=1500, d=256, f=384),
    "moe_l_bf16": dict(T=600, d=512, f=1024),
    "longctx128_bf16": dict(T=1200, d=512, f=256, chunk=512),
}


def _run(cfg, inp, logits=None, pipeline=True, defer_wgrad=None):
    g = to_dev(inp, DEV)
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV, pipeline=pipeline, defer_wgrad=defer_wgrad)
    lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"],
               compute_logits=logits is None,
               logits=None if logits is None else logits.to(DEV))
    lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    lp.check_status()
    return lp


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_identical_logits(name):
    cfg = synth.CONFIGS[name].scaled(**SMALL[name])
    inp = synth.make_inputs(cfg, seed=1, random_bias=True)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])).float()
    rb = cfg.dtype == "bf16"
    ref = oracle.layer(inp, cfg.k, cfg.renorm, rb, chunk=cfg.chunk, logits=L.double().numpy())
    lp = _run(cfg, inp, logits=L)
    assert_equal("idx", lp.idx, ref["idx"])
    nch = len(lp.chunks)
    for ci in range(nch):
        r_off = ref["offsets"][ci] if cfg.chunk else ref["offsets"]
        r_perm = ref["perm"][ci] if cfg.chunk else ref["perm"]
        r_pos = ref["pos"][ci] if cfg.chunk else ref["pos"]
        c0, c1 = lp.chunks[ci]
        assert_equal(f"offsets[{ci}]", lp.offsets_of(ci), r_off)
        assert_equal(f"perm[{ci}]", lp.perm[c0 * cfg.k:c1 * cfg.k], r_perm)
        assert_equal(f"pos[{ci}]", lp.pos[c0:c1], r_pos)
    dt = cfg.dtype
    assert_close("w", lp.w, ref["w"], "f32")
    for n in ("y", "dx", "dW1", "db1", "dW2", "db2", "dWg", "dw"):
        assert_close(n, getattr(lp, n), ref[n], dt)


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_own_logits(name):
    cfg = synth.CONFIGS[name].scaled(**SMALL[name])
    inp = synth.make_inputs(cfg, seed=2, random_bias=True)
    rb = cfg.dtype == "bf16"
    ref = oracle.layer(inp, cfg.k, cfg.renorm, rb, chunk=cfg.chunk)
    lp = _run(cfg, inp)
    assert_close("logits", lp.logits, ref["logits"], "f32")
    # the GPU's fp32 logits differ from the oracle's by far less than delta
    delta = 1e-4 * max(1.0, float(np.abs(ref["logits"]).max()))
    margin = topk_margin(ref["logits"], cfg.k)
    sure = margin > delta
    gidx = lp.idx.cpu().numpy()
    assert (gidx[sure] == ref["idx"][sure]).all()
    # near-ties: the GPU's choice must still be a top-k set within delta
    for t in np.flatnonzero(~sure):
        Lr = ref["logits"][t]
        kth = np.sort(Lr)[::-1][cfg.k - 1]
        assert (Lr[gidx[t]] >= kth - delta).all()
    same = (gidx == ref["idx"]).all(axis=1)
    assert same.mean() > 0.99
    assert_close("y", lp.y[torch.from_numpy(same).to(DEV)], ref["y"][same], cfg.dtype)
    assert_close("dx", lp.dx[torch.from_numpy(same).to(DEV)], ref["dx"][same], cfg.dtype)


def test_layer_deterministic():
    cfg = synth.CONFIGS["moe_s_bf16"].scaled(T=700, d=256, f=512)
    inp = synth.make_inputs(cfg, seed=5, random_bias=True)
    a, b = _run(cfg, inp), _run(cfg, inp)
    for n in ("idx", "pos", "perm", "y", "dx", "dW1", "db1", "dW2", "db2", "dWg", "dw"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n


OUTPUTS = ("idx", "w", "pos", "perm", "y", "dx", "dw", "dW1", "db1", "dW2", "db2", "dWg")


def test_layer_pipelined_equals_serial():
    """Two-stream chunk pipelining (5 chunks, the last one ragged) gives the
    one-stream loop's results bit for bit, eagerly and replayed from a CUDA
    graph captured with its side stream."""
    cfg = synth.CONFIGS["longctx128_bf16"].scaled(T=2300, d=512, f=256, chunk=512)
    inp = synth.make_inputs(cfg, seed=9, random_bias=True)
    ser = _run(cfg, inp, pipeline=False)
    pip = _run(cfg, inp, pipeline=True)
    assert not ser.pipeline and pip.pipeline and len(pip.chunks) == 5
    for n in OUTPUTS:
        assert torch.equal(getattr(ser, n), getattr(pip, n)), n
    # the same pass captured in a CUDA graph (as the benchmark runs it)
    g = to_dev(inp, DEV)
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV)

    def step():
        lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"])
        lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])

    step()   # eager warm-up on the side stream's first use
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for n in ("y", "dx", "dW1", "dWg"):
        getattr(lp, n).zero_()
    graph.replay()
    torch.cuda.synchronize()
    lp.check_status()
    for n in OUTPUTS:
        assert torch.equal(getattr(ser, n), getattr(lp, n)), n


@pytest.mark.parametrize("name,kw", [
    ("longctx128_bf16", dict(T=2300, d=512, f=256, chunk=512)),
    ("moe_s_bf16", dict(T=700, d=256, f=512)),
])
def test_layer_recompute_equals_saved(name, kw):
    """Recomputing the permute and expert forward in the backward (only the
    routing kept) gives the saved-activation pass's results bit for bit (both
    accumulate the weight gradients chunk by chunk)."""
    cfg = synth.CONFIGS[name].scaled(**kw)
    inp = synth.make_inputs(cfg, seed=11, random_bias=True)
    saved = _run(cfg, inp, pipeline=False, defer_wgrad=False)
    g = to_dev(inp, DEV)
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV, recompute=True)
    assert lp.recompute and not lp.pipeline
    assert lp.G.shape[0] == (cfg.chunk or cfg.T) * cfg.k   # one chunk's activations
    lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"])
    lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    lp.check_status()
    for n in OUTPUTS:
        assert torch.equal(getattr(saved, n), getattr(lp, n)), n


@pytest.mark.parametrize("name", [n for n in SMALL if n != "tiny_f32"])
def test_layer_identical_logits_many_tiles_per_pair(name, monkeypatch):
    """The small workloads with every expert GEMM launch capped at three CTA
    pairs, so that each pair walks several tiles (the full-size launch paths
    at sizes the oracle finishes in seconds)."""
    monkeypatch.setenv("MOE_GEMM_MAX_UNITS", "3")
    test_layer_identical_logits(name)


def test_layer_recompute_identical_logits():
    """Recompute mode (only the routing kept; the backward re-runs each chunk's
    permute and expert forward) against the oracle, on five dispatch chunks."""
    cfg = synth.CONFIGS["longctx128_bf16"].scaled(T=2300, d=512, f=256, chunk=512)
    inp = synth.make_inputs(cfg, seed=12, random_bias=True)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])).float()
    ref = oracle.layer(inp, cfg.k, cfg.renorm, True, chunk=cfg.chunk, logits=L.double().numpy())
    g = to_dev(inp, DEV)
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV, recompute=True)
    assert lp.recompute and len(lp.chunks) == 5
    lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"],
               compute_logits=False, logits=L.to(DEV))
    lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    lp.check_status()
    assert_equal("idx", lp.idx, ref["idx"])
    for ci, (c0, c1) in enumerate(lp.chunks):
        assert_equal(f"perm[{ci}]", lp.perm[c0 * cfg.k:c1 * cfg.k], ref["perm"][ci])
    for n in ("y", "dx", "dw", "dW1", "db1", "dW2", "db2", "dWg"):
        assert_close(n, getattr(lp, n), ref[n], cfg.dtype)


@pytest.mark.parametrize("name", ["moe_s_bf16", "longctx128_bf16"])
def test_layer_meets_the_h_storage_reading(name):
    """The kernels store G = GELU'(h) in bf16.  The other plain reading of the
    bf16 configurations stores h itself and takes GELU' of it in the backward;
    the GPU's results must meet the same tolerance against that oracle too."""
    cfg = synth.CONFIGS[name].scaled(**SMALL[name])
    inp = synth.make_inputs(cfg, seed=4, random_bias=True)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])).float()
    ref = oracle.layer(inp, cfg.k, cfg.renorm, True, chunk=cfg.chunk, logits=L.double().numpy(),
                       store_h=True)
    lp = _run(cfg, inp, logits=L)
    for n in ("y", "dx", "dw", "dW1", "db1", "dW2", "db2", "dWg"):
        assert_close(n, getattr(lp, n), ref[n], cfg.dtype)


@pytest.mark.parametrize("defer", [True, False])
def test_layer_weight_gradient_modes_identical_logits(defer):
    """The one weight-gradient pass over all chunks (default with several
    chunks) and the chunk-by-chunk accumulation, each against the oracle, on
    five dispatch chunks with a ragged last one, pipelined."""
    cfg = synth.CONFIGS["longctx128_bf16"].scaled(T=2300, d=512, f=256, chunk=512)
    inp = synth.make_inputs(cfg, seed=15, random_bias=True)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])).float()
    ref = oracle.layer(inp, cfg.k, cfg.renorm, True, chunk=cfg.chunk, logits=L.double().numpy())
    lp = _run(cfg, inp, logits=L, defer_wgrad=defer)
    assert lp.defer_wgrad == defer and lp.pipeline
    for n in ("y", "dx", "dw", "dW1", "db1", "dW2", "db2", "dWg"):
        assert_close(n, getattr(lp, n), ref[n], cfg.dtype)
