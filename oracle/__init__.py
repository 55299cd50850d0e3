"""CPU oracle for the MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never does, and
this package never imports the product's kernels or binding; both sides share
only the seeded input generator (``synth``), which holds none of the layer's
arithmetic.

The arithmetic lives in ``moe_oracle.c`` (plain C loops in double precision,
one function per step of the layer, each citing the passage it follows).
This wrapper compiles it with gcc on first use, marshals numpy float64
arrays, and composes the steps in the layer's order (``layer``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, OpenMP, portable flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def _declare(L):
    L.oracle_round_bf16.restype = ctypes.c_double
    L.oracle_round_bf16.argtypes = [ctypes.c_double]
    L.oracle_round_bf16_array.restype = None
    L.oracle_round_bf16_array.argtypes = [_i64, _D, _D]
    L.oracle_gelu.restype = ctypes.c_double
    L.oracle_gelu.argtypes = [ctypes.c_double]
    L.oracle_gelu_grad.restype = ctypes.c_double
    L.oracle_gelu_grad.argtypes = [ctypes.c_double]
    L.oracle_router_logits.argtypes = [_i64, _int, _int, _D, _D, _D, _D]
    L.oracle_gate.argtypes = [_i64, _int, _int, _int, _D, _I, _D]
    L.oracle_dispatch.argtypes = [_i64, _int, _int, _I, _I, _I, _I, _I]
    L.oracle_permute.argtypes = [_i64, _int, _int, _D, _I, _D]
    L.oracle_expert_ffn_fwd.argtypes = [_int, _int, _int, _I, _D, _D, _D, _D, _D,
                                        _D, _D, _D, _int]
    L.oracle_combine.argtypes = [_i64, _int, _int, _D, _I, _D, _D, _int]
    L.oracle_combine_bwd.argtypes = [_i64, _int, _int, _D, _D, _I, _D, _D, _D, _int]
    L.oracle_expert_ffn_bwd.argtypes = [_int, _int, _int, _I, _D, _D, _D, _D, _D, _D,
                                        _D, _D, _D, _D, _D, _D, _int, _int]
    L.oracle_router_bwd.argtypes = [_i64, _int, _int, _int, _int, _D, _D, _I, _D,
                                    _D, _D, _D, _D, _D, _int]
    for fn in ("oracle_router_logits", "oracle_gate", "oracle_dispatch",
               "oracle_permute", "oracle_expert_ffn_fwd", "oracle_combine",
               "oracle_combine_bwd", "oracle_expert_ffn_bwd", "oracle_router_bwd"):
        getattr(L, fn).restype = None


def _f64(a) -> np.ndarray:
    """Any array-like (numpy or torch, any float dtype) -> C-contiguous float64."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _pd(a):
    return None if a is None else a.ctypes.data_as(_D)


def _pi(a):
    return a.ctypes.data_as(_I)


# ---- scalar helpers ---------------------------------------------------------

def round_bf16(v: float) -> float:
    return lib().oracle_round_bf16(float(v))


def gelu(v: float) -> float:
    return lib().oracle_gelu(float(v))


def gelu_grad(v: float) -> float:
    return lib().oracle_gelu_grad(float(v))


def round_bf16_array(a) -> np.ndarray:
    a = _f64(a)
    out = np.empty_like(a)
    lib().oracle_round_bf16_array(a.size, _pd(a), _pd(out))
    return out


# ---- the layer's steps ----------------------------------------------------------

def router_logits(x, Wg, beta=None) -> np.ndarray:
    x, Wg = _f64(x), _f64(Wg)
    T, d = x.shape
    E = Wg.shape[0]
    b = None if beta is None else _f64(beta)
    out = np.empty((T, E), np.float64)
    lib().oracle_router_logits(T, d, E, _pd(x), _pd(Wg), _pd(b), _pd(out))
    return out


def gate(logits, k: int, renorm: int):
    L = _f64(logits)
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError(f"top-k needs 1 <= k <= E (k={k}, E={E})")
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_gate(T, E, k, int(renorm), _pd(L), _pi(idx), _pd(w))
    return idx, w


def dispatch(idx, E: int):
    idx = _i32(idx)
    T, k = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pos = np.empty((T, k), np.int32)
    perm = np.empty(T * k, np.int32)
    lib().oracle_dispatch(T, E, k, _pi(idx), _pi(counts), _pi(offsets), _pi(pos), _pi(perm))
    return counts, offsets, pos, perm


def permute(x, pos) -> np.ndarray:
    x, pos = _f64(x), _i32(pos)
    T, d = x.shape
    k = pos.shape[1]
    out = np.empty((T * k, d), np.float64)
    lib().oracle_permute(T, d, k, _pd(x), _pi(pos), _pd(out))
    return out


def expert_ffn_fwd(X, offsets, W1, b1, W2, b2, round_bf16: bool, store_h: bool = False):
    """Returns G = GELU'(h), A = GELU(h), Y.  With ``round_bf16`` the stored
    activations are rounded to bf16: G itself, or with ``store_h`` the
    pre-activation h that G is then taken of (the two readings of where a
    bf16 forward rounds; A and Y are the same in both)."""
    X, offsets = _f64(X), _i32(offsets)
    W1, b1, W2, b2 = _f64(W1), _f64(b1), _f64(W2), _f64(b2)
    P, d = X.shape
    E, f, _ = W1.shape
    G = np.zeros((P, f), np.float64)
    A = np.zeros((P, f), np.float64)
    Y = np.zeros((P, d), np.float64)
    lib().oracle_expert_ffn_fwd(d, f, E, _pi(offsets), _pd(X), _pd(W1), _pd(b1),
                                _pd(W2), _pd(b2), _pd(G), _pd(A), _pd(Y),
                                (2 if store_h else 1) if round_bf16 else 0)
    return G, A, Y


def combine(Y, pos, w, round_bf16: bool) -> np.ndarray:
    Y, pos = _f64(Y), _i32(pos)
    T, k = pos.shape
    d = Y.shape[1]
    wa = None if w is None else _f64(w)
    y = np.empty((T, d), np.float64)
    lib().oracle_combine(T, d, k, _pd(Y), _pi(pos), _pd(wa), _pd(y), int(round_bf16))
    return y


def combine_bwd(dy, Y, pos, w, round_bf16: bool):
    dy, Y, pos, w = _f64(dy), _f64(Y), _i32(pos), _f64(w)
    T, d = dy.shape
    k = pos.shape[1]
    dY = np.zeros((T * k, d), np.float64)
    dw = np.empty((T, k), np.float64)
    lib().oracle_combine_bwd(T, d, k, _pd(dy), _pd(Y), _pi(pos), _pd(w), _pd(dY),
                             _pd(dw), int(round_bf16))
    return dY, dw


def expert_ffn_bwd(dY, X, G, A, offsets, W1, W2, round_bf16: bool, grads=None):
    """Returns dH, dX, dW1, db1, dW2, db2 (G = GELU'(h) from the forward).
    ``grads`` (a dict with dW1, db1, dW2, db2 float64 arrays) makes the weight
    gradients accumulate into it."""
    dY, X, G, A = _f64(dY), _f64(X), _f64(G), _f64(A)
    offsets, W1, W2 = _i32(offsets), _f64(W1), _f64(W2)
    P, d = X.shape
    E, f, _ = W1.shape
    dH = np.zeros((P, f), np.float64)
    dX = np.zeros((P, d), np.float64)
    acc = grads is not None
    if grads is None:
        grads = dict(dW1=np.empty((E, f, d)), db1=np.empty((E, f)),
                     dW2=np.empty((E, d, f)), db2=np.empty((E, d)))
    lib().oracle_expert_ffn_bwd(d, f, E, _pi(offsets), _pd(dY), _pd(X), _pd(G), _pd(A),
                                _pd(W1), _pd(W2), _pd(dH), _pd(dX), _pd(grads["dW1"]),
                                _pd(grads["db1"]), _pd(grads["dW2"]), _pd(grads["db2"]),
                                int(acc), int(round_bf16))
    return dH, dX, grads["dW1"], grads["db1"], grads["dW2"], grads["db2"]


def router_bwd(dw, logits, idx, w, x, Wg, renorm: int, dWg=None):
    """Returns dL [T,E], dx_router [T,d], dWg [E,d] (accumulated into ``dWg``
    when it is given)."""
    dw, L, idx, w = _f64(dw), _f64(logits), _i32(idx), _f64(w)
    x, Wg = _f64(x), _f64(Wg)
    T, k = idx.shape
    E, d = Wg.shape
    dL = np.empty((T, E), np.float64)
    dxr = np.empty((T, d), np.float64)
    acc = dWg is not None
    if dWg is None:
        dWg = np.empty((E, d), np.float64)
    lib().oracle_router_bwd(T, d, E, k, int(renorm), _pd(dw), _pd(L), _pi(idx), _pd(w),
                            _pd(x), _pd(Wg), _pd(dL), _pd(dxr), _pd(dWg), int(acc))
    return dL, dxr, dWg


# ---- the whole layer -------------------------------------------------------------

def layer(inp: dict, k: int, renorm: int, round_bf16: bool, chunk: int | None = None,
          logits=None, backward: bool = True, store_h: bool = False) -> dict:
    """Forward and backward of the MoE layer, steps A1..A10 in order.

    ``inp`` holds x, Wg, W1, b1, W2, b2, dy and beta (see ``synth``).
    ``logits`` (optional, [T,E]) replaces A1: both sides can then take the
    routing decision on identical logits.  ``chunk`` splits the tokens into
    consecutive dispatch chunks; routing is per token, the histogram,
    offsets and positions are per chunk, and the weight gradients accumulate
    over chunks in chunk order.  Returns every intermediate, per chunk for the
    dispatch tensors.  ``store_h`` selects the other reading of where the
    bf16 forward rounds (see ``expert_ffn_fwd``)."""
    x = _f64(inp["x"])
    T = x.shape[0]
    Wg, W1, b1, W2, b2 = (_f64(inp[n]) for n in ("Wg", "W1", "b1", "W2", "b2"))
    E = Wg.shape[0]
    beta = inp.get("beta")
    dy = _f64(inp["dy"]) if backward else None
    C = chunk or T
    out = dict(logits=[], idx=[], w=[], counts=[], offsets=[], pos=[], perm=[],
               y=[], dw=[], dx=[], dL=[])
    grads = None
    dWg = None
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        xc = x[c0:c1]
        Lc = router_logits(xc, Wg, beta) if logits is None else _f64(logits)[c0:c1]
        idx, w = gate(Lc, k, renorm)
        counts, offsets, pos, perm = dispatch(idx, E)
        X = permute(xc, pos)
        G, A, Y = expert_ffn_fwd(X, offsets, W1, b1, W2, b2, round_bf16, store_h)
        y = combine(Y, pos, w, round_bf16)
        for name, v in (("logits", Lc), ("idx", idx), ("w", w), ("counts", counts),
                        ("offsets", offsets), ("pos", pos), ("perm", perm), ("y", y)):
            out[name].append(v)
        if not backward:
            continue
        dY, dw = combine_bwd(dy[c0:c1], Y, pos, w, round_bf16)
        if grads is None:
            res = expert_ffn_bwd(dY, X, G, A, offsets, W1, W2, round_bf16)
            grads = dict(zip(("dW1", "db1", "dW2", "db2"), res[2:]))
        else:
            res = expert_ffn_bwd(dY, X, G, A, offsets, W1, W2, round_bf16, grads)
        dX = res[1]
        dx_perm = combine(dX, pos, None, False)
        dL, dxr, dWg = router_bwd(dw, Lc, idx, w, xc, Wg, renorm, dWg)
        dx = dx_perm + dxr
        if round_bf16:
            dx = round_bf16_array(dx)
        out["dw"].append(dw)
        out["dx"].append(dx)
        out["dL"].append(dL)
        if chunk is None:
            out.update(X=X, G=G, A=A, Y=Y, dY=dY, dH=res[0], dX=dX)
    res = {}
    for name, v in out.items():
        if isinstance(v, list):
            if not v:
                continue
            if name in ("counts", "offsets", "pos", "perm"):
                res[name] = v if chunk else v[0]
            else:
                res[name] = np.concatenate(v, axis=0)
        else:
            res[name] = v
    if backward:
        res.update(grads)
        res["dWg"] = dWg
    return res
