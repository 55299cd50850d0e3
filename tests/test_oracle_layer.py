"""Pins for the oracle's arithmetic (A1, A5-A10 and the whole layer) against
things other than itself: library routines (torch float64 linear / GELU /
autograd, scipy softmax), closed forms, a different formulation of the same
layer (the dense dispatch mask that the expert-wise design replaces), and
central finite differences."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from mixture_experts_layer_11_gb300 import synth


# ---- scalar helpers -----------------------------------------------------------

def test_round_bf16_matches_library():
    g = torch.Generator().manual_seed(0)
    v = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(20000, generator=g, dtype=torch.float32) * 8)
    # values exactly representable in fp32, so torch's fp32 -> bf16 rounding
    # (round to nearest even) is a single rounding of the same value
    ref = v.to(torch.bfloat16).double().numpy()
    got = oracle.round_bf16_array(v.double().numpy())
    np.testing.assert_array_equal(got, ref)
    # ties: halfway cases go to the even neighbour
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert oracle.round_bf16(-(1 + 2 ** -8)) == -1.0


def test_gelu_special_values_and_library():
    assert oracle.gelu(0.0) == 0.0
    assert oracle.gelu_grad(0.0) == 0.5
    xs = np.linspace(-6, 6, 241)
    for v in xs:
        assert abs(oracle.gelu(v) - oracle.gelu(-v) - v) < 1e-14 * max(1, abs(v))
    t = torch.tensor(xs, dtype=torch.float64, requires_grad=True)
    y = F.gelu(t, approximate="none")
    y.sum().backward()
    np.testing.assert_allclose([oracle.gelu(v) for v in xs], y.detach().numpy(),
                               rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose([oracle.gelu_grad(v) for v in xs], t.grad.numpy(),
                               rtol=1e-13, atol=1e-15)


# ---- helpers ----------------------------------------------------------------------

def _inputs(cfg, seed=0, random_bias=True):
    inp = synth.make_inputs(cfg, seed=seed, random_bias=random_bias)
    return {k: (None if v is None else v.double()) for k, v in inp.items()}


def _ffn_torch(x, W1, b1, W2, b2):
    return F.linear(F.gelu(F.linear(x, W1, b1), approximate="none"), W2, b2)


def _dense_mask_layer(inp, k, renorm):
    """The dense dispatch-mask formulation: every expert runs on every token
    and a [T, E] gate matrix (zero outside each token's top-k) mixes the
    outputs.  This is the batched form the expert-wise design removes (ES-MoE
    review, section 1 challenge 3 and section 3 memory savings); it computes
    the same function.  Returns y and the autograd gradients."""
    leaves = {n: inp[n].clone().requires_grad_(True)
              for n in ("x", "Wg", "W1", "b1", "W2", "b2")}
    x, Wg = leaves["x"], leaves["Wg"]
    L = x @ Wg.T
    if inp["beta"] is not None:
        L = L + inp["beta"]
    # selection: stable descending sort (equal logits keep index order)
    order = torch.sort(L.detach(), dim=1, descending=True, stable=True).indices[:, :k]
    mask = torch.zeros_like(L).scatter_(1, order, 1.0)
    p = torch.softmax(L, dim=1)
    G = p * mask
    if renorm:
        G = G / G.sum(1, keepdim=True)
    E = Wg.shape[0]
    outs = torch.stack([_ffn_torch(x, leaves["W1"][e], leaves["b1"][e],
                                   leaves["W2"][e], leaves["b2"][e]) for e in range(E)], 1)
    y = (G.unsqueeze(-1) * outs).sum(1)
    y.backward(inp["dy"])
    res = {"y": y.detach().numpy(), "logits": L.detach().numpy()}
    for n, v in leaves.items():
        res["d" + n] = v.grad.numpy()
    return res


def _close(a, b, rtol):
    a, b = np.asarray(a), np.asarray(b)
    scale = max(np.abs(b).max(), 1e-300)
    assert np.abs(a - b).max() <= rtol * scale, (np.abs(a - b).max(), scale)


# ---- whole-layer pins ------------------------------------------------------------

@pytest.mark.parametrize("E,k,renorm,zipf", [(4, 1, 0, None), (6, 2, 1, None),
                                             (8, 3, 0, None), (8, 4, 1, 1.2),
                                             (5, 5, 1, None)])
def test_layer_equals_dense_mask_autograd(E, k, renorm, zipf):
    cfg = synth.MoEConfig("t", T=48, d=12, f=20, E=E, k=k, renorm=renorm,
                          dtype="f32", zipf_s=zipf)
    inp = _inputs(cfg, seed=E + k)
    ref = _dense_mask_layer(inp, k, renorm)
    got = oracle.layer(inp, k, renorm, round_bf16=False)
    _close(got["logits"], ref["logits"], 1e-13)
    for name, rname in (("y", "y"), ("dx", "dx"), ("dWg", "dWg"), ("dW1", "dW1"),
                        ("db1", "db1"), ("dW2", "dW2"), ("db2", "db2")):
        _close(got[name], ref[rname], 1e-11)


def test_single_expert_is_dense_ffn():
    cfg = synth.MoEConfig("t", T=40, d=16, f=24, E=1, k=1, renorm=0, dtype="f32")
    inp = _inputs(cfg, seed=5)
    got = oracle.layer(inp, 1, 0, round_bf16=False)
    x = inp["x"].clone().requires_grad_(True)
    W1 = inp["W1"][0].clone().requires_grad_(True)
    W2 = inp["W2"][0].clone().requires_grad_(True)
    b1 = inp["b1"][0].clone().requires_grad_(True)
    b2 = inp["b2"][0].clone().requires_grad_(True)
    y = _ffn_torch(x, W1, b1, W2, b2)
    y.backward(inp["dy"])
    np.testing.assert_array_equal(got["idx"], 0)
    np.testing.assert_allclose(got["w"], 1.0, rtol=0, atol=0)
    _close(got["y"], y.detach().numpy(), 1e-13)
    _close(got["dx"], x.grad.numpy(), 1e-12)
    _close(got["dW1"][0], W1.grad.numpy(), 1e-12)
    _close(got["dW2"][0], W2.grad.numpy(), 1e-12)
    _close(got["db1"][0], b1.grad.numpy(), 1e-12)
    _close(got["db2"][0], b2.grad.numpy(), 1e-12)
    # one expert: p = 1 exactly, so the router receives no gradient
    assert np.abs(got["dWg"]).max() == 0.0


def test_identical_experts_closed_form():
    cfg = synth.MoEConfig("t", T=30, d=10, f=14, E=5, k=3, renorm=1, dtype="f32")
    inp = _inputs(cfg, seed=9)
    for n in ("W1", "b1", "W2", "b2"):
        inp[n] = inp[n][:1].expand_as(inp[n]).contiguous()
    got = oracle.layer(inp, 3, 1, round_bf16=False)
    y_ref = _ffn_torch(inp["x"], inp["W1"][0], inp["b1"][0], inp["W2"][0], inp["b2"][0])
    _close(got["y"], y_ref.numpy(), 1e-13)
    # renormalised weights sum to one and every expert gives the same output,
    # so the gate weights receive equal gradients and the logits none
    assert np.abs(got["dL"]).max() < 1e-14
    assert np.abs(got["dWg"]).max() < 1e-13


def test_k_equals_E_is_softmax_mixture():
    cfg = synth.MoEConfig("t", T=25, d=8, f=12, E=4, k=4, renorm=1, dtype="f32")
    inp = _inputs(cfg, seed=11)
    got = oracle.layer(inp, 4, 1, round_bf16=False, backward=False)
    p = torch.softmax(inp["x"] @ inp["Wg"].T, 1)
    outs = torch.stack([_ffn_torch(inp["x"], inp["W1"][e], inp["b1"][e], inp["W2"][e],
                                   inp["b2"][e]) for e in range(4)], 1)
    _close(got["y"], (p.unsqueeze(-1) * outs).sum(1).numpy(), 1e-13)


def test_zero_first_layer_closed_form():
    # W1 = 0: H = b1, A = GELU(b1), Y = W2 GELU(b1) + b2 for every row
    cfg = synth.MoEConfig("t", T=9, d=6, f=7, E=3, k=1, renorm=0, dtype="f32")
    inp = _inputs(cfg, seed=2)
    inp["W1"] = torch.zeros_like(inp["W1"])
    got = oracle.layer(inp, 1, 0, round_bf16=False, backward=False)
    for t in range(9):
        e = int(got["idx"][t, 0])
        b1 = inp["b1"][e].numpy()
        a = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in b1])
        yv = inp["W2"][e].numpy() @ a + inp["b2"][e].numpy()
        _close(got["y"][t], got["w"][t, 0] * yv, 1e-14)


def _topk_margin(L, k):
    s = np.sort(L, axis=1)[:, ::-1]
    gaps = [s[:, j] - s[:, j + 1] for j in range(min(k, L.shape[1] - 1))]
    return np.min(gaps) if gaps else np.inf


@pytest.mark.parametrize("k,renorm", [(1, 0), (2, 1), (2, 0)])
def test_finite_differences(k, renorm):
    cfg = synth.MoEConfig("t", T=6, d=5, f=7, E=4, k=k, renorm=renorm, dtype="f32")
    inp = _inputs(cfg, seed=21 + k)
    got = oracle.layer(inp, k, renorm, round_bf16=False)
    assert _topk_margin(got["logits"], k) > 1e-3   # routing cannot flip under h
    dy = inp["dy"].numpy()
    h = 1e-6
    rng = np.random.default_rng(0)

    def loss(mod):
        r = oracle.layer(mod, k, renorm, round_bf16=False, backward=False)
        return float((r["y"] * dy).sum())

    for name, gname in (("x", "dx"), ("Wg", "dWg"), ("W1", "dW1"), ("b1", "db1"),
                        ("W2", "dW2"), ("b2", "db2")):
        base = inp[name]
        for _ in range(6):
            i = tuple(rng.integers(0, s) for s in base.shape)
            plus, minus = dict(inp), dict(inp)
            bp, bm = base.clone(), base.clone()
            bp[i] += h
            bm[i] -= h
            plus[name], minus[name] = bp, bm
            fd = (loss(plus) - loss(minus)) / (2 * h)
            an = got[gname][i]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, i, fd, an)


def test_chunking_matches_unchunked():
    cfg = synth.MoEConfig("t", T=60, d=8, f=16, E=6, k=2, renorm=1, dtype="f32", zipf_s=1.1)
    inp = _inputs(cfg, seed=4)
    full = oracle.layer(inp, 2, 1, round_bf16=False)
    ch = oracle.layer(inp, 2, 1, round_bf16=False, chunk=16)
    for n in ("logits", "idx", "w", "y", "dx", "dw"):
        _close(ch[n], full[n], 1e-13)
    for n in ("dW1", "db1", "dW2", "db2", "dWg"):
        _close(ch[n], full[n], 1e-12)
    # per-chunk dispatch is the dispatch of that chunk's own slots
    for c, c0 in enumerate(range(0, 60, 16)):
        counts, offsets, pos, perm = oracle.dispatch(full["idx"][c0:c0 + 16], 6)
        np.testing.assert_array_equal(ch["offsets"][c], offsets)
        np.testing.assert_array_equal(ch["perm"][c], perm)


def test_bf16_storage_rounds_only_stored_activations():
    cfg = synth.MoEConfig("t", T=32, d=16, f=32, E=4, k=2, renorm=1, dtype="bf16")
    inp = _inputs(cfg, seed=8)
    r = oracle.layer(inp, 2, 1, round_bf16=True)
    for n in ("G", "A", "Y", "dY", "dH", "dX", "y", "dx"):
        np.testing.assert_array_equal(oracle.round_bf16_array(r[n]), r[n])
    full = oracle.layer(inp, 2, 1, round_bf16=False)
    # rounding moves results by about bf16 precision, not more
    for n in ("y", "dx", "dW1", "dW2", "dWg"):
        _close(r[n], full[n], 2e-2)


def test_h_storage_reading_single_expert_against_library():
    """The second reading of where the bf16 forward rounds: h itself is stored
    in bf16 and the backward takes GELU' of it.  With one expert the forward
    is a dense layer: G must equal torch's float64 autograd derivative of the
    exact GELU at bf16(h) (h from torch's float64 linear), while A and Y are
    those of the first reading (both come from the unrounded h)."""
    cfg = synth.MoEConfig("t", T=48, d=32, f=40, E=1, k=1, renorm=0, dtype="bf16")
    inp = _inputs(cfg, seed=13)
    X = inp["x"]
    offsets = np.array([0, cfg.T], np.int32)
    G2, A2, Y2 = oracle.expert_ffn_fwd(X, offsets, inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                       round_bf16=True, store_h=True)
    G1, A1, Y1 = oracle.expert_ffn_fwd(X, offsets, inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                       round_bf16=True)
    h = F.linear(X, inp["W1"][0], inp["b1"][0])
    hr = torch.from_numpy(oracle.round_bf16_array(h.numpy())).requires_grad_(True)
    F.gelu(hr, approximate="none").sum().backward()
    _close(G2, hr.grad.numpy(), 1e-13)
    # G of the first reading is a bf16 value, of the second in general not
    np.testing.assert_array_equal(oracle.round_bf16_array(G1), G1)
    assert not np.array_equal(oracle.round_bf16_array(G2), G2)
    np.testing.assert_array_equal(A2, A1)
    np.testing.assert_array_equal(Y2, Y1)


def test_h_storage_reading_changes_only_the_backward():
    cfg = synth.MoEConfig("t", T=40, d=16, f=32, E=4, k=2, renorm=1, dtype="bf16")
    inp = _inputs(cfg, seed=14)
    a = oracle.layer(inp, 2, 1, round_bf16=True)
    b = oracle.layer(inp, 2, 1, round_bf16=True, store_h=True)
    for n in ("y", "dw"):
        np.testing.assert_array_equal(a[n], b[n])
    # the two readings differ by about bf16 precision in the gradients
    for n in ("dx", "dW1", "db1", "dWg"):
        _close(b[n], a[n], 2e-2)
