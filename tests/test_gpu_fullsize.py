"""GPU parity at the workloads' own sizes, where every launch of the grouped
expert GEMM walks many tiles per CTA pair: the static persistent tile order,
the bias and GELU' operands streamed one tile ahead, the GELU' ring kept two
chunks ahead across tiles, and the weight-gradient add-reductions over
dispatch chunks all take the paths they take in the benchmark.

* moe_s_bf16 and skewed64_bf16 at full size, and moe_l_bf16 /
  longctx128_bf16 at reduced T (same d, f, E, k; several dispatch chunks for
  the long-context family), sized so that every bias+GELU and GELU'-scaling
  launch has at least three times as many work units as there are
  co-resident CTA pairs: every output against the complete oracle run, on
  identical fp32 logits.
* moe_l_bf16 and longctx128_bf16 at full size (T = 16384 and T = 262144 in 8
  dispatch chunks), where the complete oracle would run for hours on the host.
  The GPU computes its own logits; they must match the oracle's on a token
  sample, and the oracle takes its routing decisions on the GPU's fp32 logits
  (both sides decide on identical values).  Then:
    - idx, w, and per chunk counts, offsets, pos, perm over every token;
    - y, dx and dw on a seeded token sample: each depends only on its own
      token's routing, so the oracle computes them from the sampled tokens
      alone;
    - dW1, db1, dW2, db2 of selected experts, from the oracle's steps over
      exactly the rows routed to that expert (all chunks together);
    - dWg of experts with few tokens, from the oracle's layer on exactly the
      tokens routed there (with renormalised gates no other token reaches
      those rows of dWg)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_11_gb300 import synth
from mixture_experts_layer_11_gb300.layer import LayerPass
from parity_util import assert_close, assert_equal, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRAD = ("dW1", "db1", "dW2", "db2")


def _units(offsets, N, tile_m=256, tile_n=256):
    """Work units of one VarM launch (m-tiles of each expert x n-tiles)."""
    n = np.diff(np.asarray(offsets, dtype=np.int64))
    return int(sum(-(-int(c) // tile_m) * -(-N // tile_n) for c in n if c > 0))


def _pairs():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def _layer(cfg, g, logits=None):
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=DEV)
    lp.forward(g["x"], g["Wg"], g["W1"], g["b1"], g["W2"], g["b2"], g["beta"],
               compute_logits=logits is None,
               logits=None if logits is None else logits.to(DEV))
    lp.backward(g["dy"], g["x"], g["Wg"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    lp.check_status()
    return lp


COMPLETE = {
    "moe_s_bf16": dict(),
    "skewed64_bf16": dict(),
    "moe_l_bf16": dict(T=2048),
    "longctx128_bf16": dict(T=4096, chunk=2048),
}


@pytest.mark.parametrize("name", list(COMPLETE))
def test_complete_parity_many_tiles_per_pair(name):
    cfg = synth.CONFIGS[name].scaled(**COMPLETE[name])
    inp = synth.make_inputs(cfg, seed=3, random_bias=True)
    L = torch.from_numpy(oracle.router_logits(inp["x"], inp["Wg"], inp["beta"])).float()
    ref = oracle.layer(inp, cfg.k, cfg.renorm, True, chunk=cfg.chunk, logits=L.double().numpy())
    offs = ref["offsets"] if cfg.chunk else [ref["offsets"]]
    # every bias+GELU / GELU'-scaling launch (N = d_ffn) gives each pair >= 3 tiles
    assert min(_units(o, cfg.f) for o in offs) >= 3 * _pairs()
    lp = _layer(cfg, to_dev(inp, DEV), logits=L)
    assert_equal("idx", lp.idx, ref["idx"])
    for ci, (c0, c1) in enumerate(lp.chunks):
        pick = (lambda v: v[ci]) if cfg.chunk else (lambda v: v)
        assert_equal(f"offsets[{ci}]", lp.offsets_of(ci), pick(ref["offsets"]))
        assert_equal(f"perm[{ci}]", lp.perm[c0 * cfg.k:c1 * cfg.k], pick(ref["perm"]))
        assert_equal(f"pos[{ci}]", lp.pos[c0:c1], pick(ref["pos"]))
    assert_close("w", lp.w, ref["w"], "f32")
    for n in ("y", "dx", "dw", "dWg") + GRAD:
        assert_close(n, getattr(lp, n), ref[n], cfg.dtype)


# ---- full size, sampled -----------------------------------------------------------

def _expert_grads(e, idx, w, x, dy, W1, b1, W2, b2):
    """Oracle weight / bias gradients of expert e: its steps (permute, expert
    FFN forward, combine backward, expert FFN backward) over exactly the rows
    routed to e, in token order, as one segment."""
    rows = np.flatnonzero((idx == e).any(axis=1))
    j = np.argmax(idx[rows] == e, axis=1)
    n = len(rows)
    pos = np.arange(n, dtype=np.int32)[:, None]
    offs = np.array([0, n], np.int32)
    X = oracle.permute(x[rows], pos)
    sl = slice(e, e + 1)
    G, A, Y = oracle.expert_ffn_fwd(X, offs, W1[sl], b1[sl], W2[sl], b2[sl], True)
    dY, _ = oracle.combine_bwd(dy[rows], Y, pos, w[rows, j][:, None], True)
    res = oracle.expert_ffn_bwd(dY, X, G, A, offs, W1[sl], W2[sl], True)
    return dict(zip(GRAD, (r[0] for r in res[2:])))


def _sampled_full_size(name, n_first, n_per_chunk, grad_experts, dwg_experts):
    cfg = synth.CONFIGS[name]
    g = synth.make_inputs(cfg, seed=0, device=DEV)
    lp = _layer(cfg, g)
    C = cfg.chunk_tokens
    rng = np.random.default_rng(7)
    sample = [np.arange(n_first)]
    for c0 in range(0, cfg.T, C):
        sample.append(rng.choice(np.arange(c0, min(cfg.T, c0 + C)), n_per_chunk, replace=False))
    sub = np.unique(np.concatenate(sample))
    cpu = {n: (None if v is None else v.cpu()) for n, v in g.items()}
    # host copies in the oracle's float64 (converted once, not per call)
    W = {n: oracle._f64(cpu[n]) for n in ("Wg", "W1", "b1", "W2", "b2")}
    Lg = lp.logits.cpu().double().numpy()
    # the GPU's own logits against the oracle's on the sample
    Lr = oracle.router_logits(cpu["x"][sub], W["Wg"], cpu["beta"])
    assert_close("logits[sample]", Lg[sub], Lr, "f32")
    # routing over every token and chunk, decided on the GPU's fp32 logits
    idx, w = oracle.gate(Lg, cfg.k, cfg.renorm)
    assert_equal("idx", lp.idx, idx)
    assert_close("w", lp.w, w, "f32")
    for ci, (c0, c1) in enumerate(lp.chunks):
        counts, offsets, pos, perm = oracle.dispatch(idx[c0:c1], cfg.E)
        assert_equal(f"counts[{ci}]", lp.counts_of(ci), counts)
        assert_equal(f"offsets[{ci}]", lp.offsets_of(ci), offsets)
        assert_equal(f"pos[{ci}]", lp.pos[c0:c1], pos)
        assert_equal(f"perm[{ci}]", lp.perm[c0 * cfg.k:c1 * cfg.k], perm)
        assert _units(offsets, cfg.f) >= 3 * _pairs()
    # per-token outputs on the sample
    si = torch.from_numpy(sub)

    def sub_inputs(rows):
        r = torch.from_numpy(rows)
        return dict(x=cpu["x"][r], dy=cpu["dy"][r], beta=cpu["beta"], **W)

    ref = oracle.layer(sub_inputs(sub), cfg.k, cfg.renorm, True, logits=Lg[sub])
    for n in ("y", "dx", "dw"):
        assert_close(f"{n}[sample]", getattr(lp, n).cpu()[si], ref[n], cfg.dtype)
    # weight and bias gradients of selected experts (every chunk's rows)
    total = np.bincount(idx.reshape(-1), minlength=cfg.E)
    for e in grad_experts(total):
        r = _expert_grads(e, idx, w, cpu["x"], cpu["dy"], W["W1"], W["b1"], W["W2"], W["b2"])
        for n in GRAD:
            assert_close(f"{n}[{e}] ({total[e]} rows)", getattr(lp, n)[e].cpu(), r[n], cfg.dtype)
    for e in dwg_experts(total):
        rows = np.flatnonzero((idx == e).any(axis=1))
        r = oracle.layer(sub_inputs(rows), cfg.k, cfg.renorm, True, logits=Lg[rows])
        assert_close(f"dWg[{e}] ({total[e]} tokens)", lp.dWg[e].cpu(), r["dWg"][e], cfg.dtype)
    del lp
    torch.cuda.empty_cache()


def _smallest(total, m, lo=1, hi=None):
    cand = [e for e in np.argsort(total, kind="stable")
            if total[e] >= lo and (hi is None or total[e] <= hi)]
    return [int(e) for e in cand[:m]]


def test_moe_l_full_size_sampled():
    # the expert with the fewest rows (about 1900 of 32768): its gradients
    _sampled_full_size("moe_l_bf16", n_first=256, n_per_chunk=256,
                       grad_experts=lambda t: _smallest(t, 1),
                       dwg_experts=lambda t: [])


def test_longctx128_full_size_sampled():
    # 262144 tokens in 8 dispatch chunks; gradients of two experts with few
    # rows and of one with a few hundred, dWg of the two small ones
    _sampled_full_size(
        "longctx128_bf16", n_first=192, n_per_chunk=48,
        grad_experts=lambda t: _smallest(t, 2, lo=8) + _smallest(t, 1, lo=200, hi=1000),
        dwg_experts=lambda t: _smallest(t, 2, lo=8))
