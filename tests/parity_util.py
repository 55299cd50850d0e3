"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (per tensor):
  fp32 layer: max|gpu - ref| <= 1e-5 * max|ref|
  bf16 layer: max|gpu - ref| <= 2e-2 * max|ref|
  integer / index outputs: bit-exact.
"""
import numpy as np
import torch

TOL = {"f32": 1e-5, "bf16": 2e-2}


def np64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def assert_close(name, got, ref, dtype: str, rel: float | None = None):
    g, r = np64(got), np64(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    tol = TOL[dtype] if rel is None else rel
    scale = float(np.abs(r).max()) if r.size else 0.0
    err = float(np.abs(g - r).max()) if r.size else 0.0
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    assert err <= tol * max(scale, 1e-30), \
        f"{name}: max abs err {err:.3e} > {tol:g} * max|ref| = {tol * scale:.3e}"
    return err / max(scale, 1e-30)


def assert_equal(name, got, ref):
    g = got.cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    bad = np.flatnonzero(g.reshape(-1) != r.reshape(-1))
    assert bad.size == 0, f"{name}: {bad.size} mismatches, first at {bad[:5]}"


def to_dev(inp: dict, dev) -> dict:
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def topk_margin(L: np.ndarray, k: int) -> np.ndarray:
    """Per-row smallest gap among the k+1 largest logits (ties -> 0)."""
    s = -np.sort(-L, axis=1)
    m = min(k, L.shape[1] - 1)
    if m == 0:
        return np.full(L.shape[0], np.inf)
    return np.min(s[:, :m] - s[:, 1:m + 1], axis=1)
