"""Pins for the oracle's routing steps (A2 gate, A3 histogram / scan / stable
assignment, A4 permute): brute force against library sorts, exhaustive tie
patterns, invariants, and a hand-worked example from tests/golden/."""
import itertools
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _library_topk(L, k):
    """Top-k by Python's stable sort on (-logit): equal logits keep index
    order, so the lower expert index comes first."""
    order = sorted(range(len(L)), key=lambda e: -L[e])
    return order[:k]


@pytest.mark.parametrize("E", [1, 2, 3, 4])
def test_gate_exhaustive_ties(E):
    # every row of small integer logits in {-1, 0, 1}^E: ties everywhere
    rows = np.array(list(itertools.product([-1.0, 0.0, 1.0], repeat=E)))
    for k in range(1, E + 1):
        for renorm in (0, 1):
            idx, w = oracle.gate(rows, k, renorm)
            p = scipy.special.softmax(rows, axis=1)
            for t, L in enumerate(rows):
                sel = _library_topk(list(L), k)
                assert list(idx[t]) == sel
                ws = p[t, sel]
                if renorm:
                    ws = ws / ws.sum()
                np.testing.assert_allclose(w[t], ws, rtol=1e-14, atol=0)


def test_gate_weights_properties():
    rng = np.random.default_rng(1)
    L = rng.standard_normal((500, 16))
    for k in (2, 4, 8):
        _, w = oracle.gate(L, k, 1)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    # k = E with renorm is the full softmax, in descending order
    idx, w = oracle.gate(L, 16, 1)
    p = scipy.special.softmax(L, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-13)
    # k = 1 without renorm is the largest softmax probability
    idx, w = oracle.gate(L, 1, 0)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(L, 1))
    np.testing.assert_allclose(w[:, 0], p.max(1), rtol=1e-13)


def _random_idx(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 3, 2), (8, 4, 1), (8, 4, 4), (37, 5, 3)])
def test_dispatch_bruteforce(T, E, k):
    rng = np.random.default_rng(T * 100 + E * 10 + k)
    idx = _random_idx(rng, T, E, k)
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    # library: a stable sort of the slots by expert keeps token order inside
    # each expert
    slots = list(range(T * k))
    ref_perm = sorted(slots, key=lambda s: idx.reshape(-1)[s])
    np.testing.assert_array_equal(perm, ref_perm)
    ref_pos = np.empty(T * k, np.int64)
    ref_pos[np.array(ref_perm)] = np.arange(T * k)
    np.testing.assert_array_equal(pos.reshape(-1), ref_pos)
    np.testing.assert_array_equal(counts, np.bincount(idx.reshape(-1), minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))


def test_dispatch_invariants_large():
    rng = np.random.default_rng(7)
    T, E, k = 3000, 64, 8
    idx = _random_idx(rng, T, E, k)
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    assert counts.sum() == T * k and offsets[-1] == T * k
    assert sorted(perm.tolist()) == list(range(T * k))          # bijection
    np.testing.assert_array_equal(perm[pos.reshape(-1)], np.arange(T * k))
    for e in range(E):                                          # stability
        seg = perm[offsets[e]:offsets[e + 1]]
        tok = seg // k
        assert np.all(np.diff(tok) > 0)
        assert np.all(idx.reshape(-1)[seg] == e)


def test_permute_is_row_copy():
    rng = np.random.default_rng(3)
    T, E, k, d = 20, 4, 2, 6
    idx = _random_idx(rng, T, E, k)
    _, _, pos, perm = oracle.dispatch(idx, E)
    x = rng.standard_normal((T, d))
    Xp = oracle.permute(x, pos)
    np.testing.assert_array_equal(Xp, x[perm // k])


def _read_golden(name):
    data = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split("=", 1)
            data[key.strip()] = [float(v) for v in val.split()]
    return data


def test_dispatch_worked_example():
    g = _read_golden("dispatch_worked_example.txt")
    T, E, k = int(g["T"][0]), int(g["E"][0]), int(g["k"][0])
    L = np.array(g["logits"]).reshape(T, E)
    idx, _ = oracle.gate(L, k, 1)
    np.testing.assert_array_equal(idx.reshape(-1), np.array(g["idx"], np.int32))
    counts, offsets, pos, perm = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(counts, np.array(g["counts"], np.int32))
    np.testing.assert_array_equal(offsets, np.array(g["offsets"], np.int32))
    np.testing.assert_array_equal(pos.reshape(-1), np.array(g["pos"], np.int32))
    np.testing.assert_array_equal(perm, np.array(g["perm"], np.int32))


def test_oracle_rejects_invalid_routing_shapes():
    with pytest.raises(ValueError):
        oracle.gate(np.zeros((3, 1)), 2, 1)
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0], [3]], np.int32), 2)
