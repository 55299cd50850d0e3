"""One MoE layer forward + backward pass, composed from the C-ABI entry
points in the layer's order (route, permute, expert FFN, combine; then combine
backward, expert FFN backward, permute backward, router backward).

Tokens are processed in consecutive dispatch chunks of at most ``chunk``
tokens, the bounded dispatch chunk of PipelinedLLEP ("Flattening Every Memory
Peak in Long-Context Mixture-of-Experts Training", abstract): routing is per
token, the histogram / offsets / positions are per chunk, and the weight
gradients accumulate over chunks in fp32 in chunk order.  The activations a
chunk's backward needs (X_perm, G = GELU'(h), A, Y_perm) stay resident in HBM between
the forward and the backward; the backward's transient buffers (dY_perm,
dX_perm and the library workspace) are shared by all chunks.

All buffers are allocated once, up front, by ``LayerPass``; ``forward`` and
``backward`` only launch work on the current CUDA stream (no allocation, no
host synchronisation).  This module does no arithmetic of its own.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import ops


def _pad4(n: int) -> int:
    return (n + 3) // 4 * 4


class LayerPass:
    """Preallocated buffers and launch sequence for one layer configuration.

    Parameters: T tokens, d model width, f expert hidden width, E experts,
    k experts per token, dtype (torch.bfloat16 or torch.float32), renorm,
    chunk (dispatch chunk cap; None = one chunk)."""

    def __init__(self, T: int, d: int, f: int, E: int, k: int, dtype: torch.dtype,
                 renorm: int, chunk: Optional[int] = None, device="cuda"):
        self.T, self.d, self.f, self.E, self.k = T, d, f, E, k
        self.dtype, self.renorm = dtype, int(renorm)
        C = chunk if chunk else T
        if C % 4 and C < T:
            raise ValueError("chunk must be a multiple of 4")
        self.C = C
        self.chunks = [(c0, min(T, c0 + C)) for c0 in range(0, T, C)] or [(0, 0)]
        nch = len(self.chunks)
        dev = torch.device(device)
        f32, i32 = torch.float32, torch.int32
        z = lambda *s, dt=dtype: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.shapes = [ops.make_shape(c1 - c0, d, f, E, k, dtype, renorm) for c0, c1 in self.chunks]
        # routing (per token; per chunk rows padded to 16-byte multiples)
        self.logits = z(T, E, dt=f32)
        self.idx = z(T, k, dt=i32)
        self.w = z(T, k, dt=f32)
        self.pos = z(T, k, dt=i32)
        self.perm = z(T * k, dt=i32)
        self.counts = z(nch, _pad4(E), dt=i32)
        self.offsets = z(nch, _pad4(E + 1), dt=i32)
        # saved activations of every chunk
        self.X_perm = z(T * k, d)
        self.G = z(T * k, f)
        self.A = z(T * k, f)
        self.Y_perm = z(T * k, d)
        self.y = z(T, d)
        # backward
        self.dw = z(T, k, dt=f32)
        self.dx = z(T, d)
        self.dY_perm = z(C * k, d)
        self.dX_perm = z(C * k, d)
        self.dW1 = z(E, f, d, dt=f32)
        self.db1 = z(E, f, dt=f32)
        self.dW2 = z(E, d, f, dt=f32)
        self.db2 = z(E, d, dt=f32)
        self.dWg = z(E, d, dt=f32)
        ws = max(ops.moe_workspace_size(s) for s in self.shapes)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)

    # -- per-chunk views ------------------------------------------------------------
    def _rows(self, t: torch.Tensor, c0: int, c1: int, mult: int = 1) -> torch.Tensor:
        return t[c0 * mult:c1 * mult]

    def forward(self, x, Wg, W1, b1, W2, b2, beta=None, compute_logits: bool = True,
                logits: Optional[torch.Tensor] = None):
        """x [T,d]; Wg [E,d]; W1 [E,f,d]; b1 [E,f]; W2 [E,d,f]; b2 [E,d]
        (storage dtype); beta [E] fp32 or None.  With compute_logits False the
        router logits are taken from ``logits`` [T,E] fp32 instead of x Wg^T.
        Returns y [T,d] (a buffer owned by this object)."""
        k = self.k
        if not compute_logits:
            self.logits.copy_(logits)
        for ci, ((c0, c1), s) in enumerate(zip(self.chunks, self.shapes)):
            if c1 == c0:
                continue
            xc = self._rows(x, c0, c1)
            pos = self._rows(self.pos, c0, c1)
            perm = self._rows(self.perm, c0, c1, k)
            offs = self.offsets[ci]
            ops.moe_route(s, xc, Wg, beta, self._rows(self.logits, c0, c1), int(compute_logits),
                          self._rows(self.idx, c0, c1), self._rows(self.w, c0, c1),
                          self.counts[ci], offs, pos, perm, self.ws, self.status)
            Xp = self._rows(self.X_perm, c0, c1, k)
            ops.moe_permute(s, xc, pos, Xp)
            Yp = self._rows(self.Y_perm, c0, c1, k)
            ops.moe_expert_ffn_fwd(s, Xp, offs, W1, b1, W2, b2, self._rows(self.G, c0, c1, k),
                                   self._rows(self.A, c0, c1, k), Yp, self.ws, self.status)
            ops.moe_combine_fwd(s, Yp, pos, self._rows(self.w, c0, c1), self._rows(self.y, c0, c1))
        return self.y

    def backward(self, dy, x, Wg, W1, W2):
        """Backward of the last ``forward``: dy [T,d].  Fills dx, dw, dW1, db1,
        dW2, db2, dWg (buffers owned by this object)."""
        k = self.k
        for ci, ((c0, c1), s) in enumerate(zip(self.chunks, self.shapes)):
            acc = int(ci > 0)
            if c1 == c0:
                continue
            n = (c1 - c0) * k
            pos = self._rows(self.pos, c0, c1)
            w = self._rows(self.w, c0, c1)
            offs = self.offsets[ci]
            dYp = self.dY_perm[:n]
            dXp = self.dX_perm[:n]
            ops.moe_combine_bwd(s, self._rows(dy, c0, c1), self._rows(self.Y_perm, c0, c1, k), pos,
                                w, dYp, self._rows(self.dw, c0, c1))
            ops.moe_expert_ffn_bwd(s, dYp, self._rows(self.X_perm, c0, c1, k),
                                   self._rows(self.G, c0, c1, k), self._rows(self.A, c0, c1, k),
                                   offs, W1, W2, dXp, self.dW1, self.db1, self.dW2, self.db2, acc,
                                   self.ws, self.status)
            # permute backward (A9) fused into the router backward (A10)
            ops.moe_route_bwd(s, self._rows(self.dw, c0, c1), self._rows(self.logits, c0, c1),
                              self._rows(self.idx, c0, c1), w, self._rows(self.perm, c0, c1, k),
                              offs, self._rows(x, c0, c1), Wg, dXp, pos,
                              self._rows(self.dx, c0, c1), self.dWg, acc, self.ws, self.status)
        return self.dx

    def offsets_of(self, ci: int) -> torch.Tensor:
        return self.offsets[ci, :self.E + 1]

    def counts_of(self, ci: int) -> torch.Tensor:
        return self.counts[ci, :self.E]

    def check_status(self):
        """Synchronises and raises if a kernel reported a device-side error."""
        code = int(self.status.item())
        if code != ops.MOE_OK:
            raise ops.MoEError("device", code, ops.moe_status_string(code))


def expert_flops(T: int, d: int, f: int, k: int) -> float:
    """Algorithmic expert FLOPs of forward + backward: 12 T k d f."""
    return 12.0 * T * k * d * f


def router_flops(T: int, d: int, E: int) -> float:
    return 6.0 * T * d * E


def _ceil(a: int, b: int) -> int:
    return math.ceil(a / b)
