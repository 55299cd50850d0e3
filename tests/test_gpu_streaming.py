"""The layer pass with expert weights in pinned host memory, streamed to the
GPU one group of experts at a time (ExpertStreamingPass), against the pass
with device-resident weights (LayerPass) and against the oracle.

Per expert the kernels see the same rows and weights in both passes, so y,
dx, dw, dWg and db1 must be bit-identical; the weight gradients' reductions
are cut into parts per launch, and a launch here holds one group's experts
instead of all of them, so dW1, dW2 and db2 are compared with the oracle at
the bf16 tolerance."""
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import synth
from mixture_experts_layer_11_gb300.layer import LayerPass
from mixture_experts_layer_11_gb300.streaming import ExpertStreamingPass
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [  # name, sizes, experts per streamed group
    ("longctx128_bf16", dict(T=1200, d=512, f=256, chunk=512), 16),   # 8 groups, 3 chunks
    ("skewed64_bf16", dict(T=900, d=256, f=384), 24),                  # groups of 24, 24, 16
]


@pytest.mark.parametrize("name,kw,group", CASES)
def test_streamed_weights_match_resident_and_oracle(name, kw, group):
    cfg = synth.CONFIGS[name].scaled(**kw)
    inp = synth.make_inputs(cfg, seed=6, random_bias=True)
    g = to_dev(inp, DEV)
    host = {n: inp[n].pin_memory() for n in ("W1", "b1", "W2", "b2")}
    sp = ExpertStreamingPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                             chunk=cfg.chunk, group=group, device=DEV)
    assert len(sp.groups) == -(-cfg.E // group)
    sp.forward(g["x"], g["Wg"], host["W1"], host["b1"], host["W2"], host["b2"], g["beta"])
    sp.backward(g["dy"], g["x"], g["Wg"], host["W1"], host["W2"])
    torch.cuda.synchronize()
    sp.check_status()
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV, pipeline=False)
    lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"])
    lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    lp.check_status()
    for n in ("logits", "idx", "pos", "y", "dx", "dw", "dWg", "db1"):
        assert torch.equal(getattr(sp, n), getattr(lp, n)), n
    # the oracle on the GPU's logits (identical routing decisions)
    ref = oracle.layer(inp, cfg.k, cfg.renorm, True, chunk=cfg.chunk,
                       logits=sp.logits.cpu().double().numpy())
    for n, got in (("y", sp.y), ("dx", sp.dx), ("dW1", sp.dW1_host), ("dW2", sp.dW2_host),
                   ("db1", sp.db1), ("db2", sp.db2), ("dWg", sp.dWg)):
        assert_close(n, got, ref[n], cfg.dtype)
