"""One MoE layer forward + backward pass, composed from the C-ABI entry
points in the layer's order (route, permute, expert FFN, combine; then combine
backward, expert FFN backward, permute backward, router backward).

With ``gather`` the permute is fused into the expert GEMMs: the first GEMM of
the forward and the dW1 GEMM of the backward load the rows of x that the
dispatch's perm names (row r of the expert-sorted activations is
x[perm[r] / k]) instead of reading a permuted copy, so X_perm is never written
or kept.  The results are those of the unfused sequence, bit for bit.  It is
not the default: each TMA tile::gather4 load moves four 128-byte rows, and at
that rate the loads, not the tensor cores, bound those GEMMs.

Tokens are processed in consecutive dispatch chunks of at most ``chunk``
tokens, the bounded dispatch chunk of PipelinedLLEP ("Flattening Every Memory
Peak in Long-Context Mixture-of-Experts Training", abstract): routing is per
token, the histogram / offsets / positions are per chunk, and the weight
gradients accumulate over chunks in fp32 in chunk order.  The activations a
chunk's backward needs (G = GELU'(h), A, Y_perm; X_perm when unfused) stay resident in HBM between
the forward and the backward; the backward's transient buffers (dY_perm,
dX_perm and the library workspace) are shared by all chunks.

With more than one chunk the chunks are pipelined on two streams (the
micro-batch overlap of MPipeMoE, "research method", and ES-MoE's overlap of
the permutation with compute): a side stream routes and permutes chunk i+1
and combines chunk i-1 while the current stream runs chunk i's expert GEMMs
(on 64 of the GPU's 76 CTA pairs, so that it has SMs of its own), and in the
backward it
runs chunk i+1's combine backward and chunk i's router backward next to chunk
i's expert backward.  The side stream has its own library workspace, dY_perm
and dX_perm are double-buffered, and events order every reuse.  Each fp32
gradient still accumulates in chunk order on one stream (dW, db on the current
one, dWg on the side one), so the results equal the serial loop's bit for bit.

With more than one chunk (and the activations kept) the weight gradients are
not accumulated chunk by chunk: dY_perm and dH of every chunk are kept, each
chunk's backward computes only its activation gradients (and db1), and one
weight-gradient pass after the last chunk sums each expert's rows over all
chunks (``moe_expert_ffn_bwd_weights``).  Every dW tile is then written once
per pass instead of being read, added to and written back once per chunk, and
experts with few rows per chunk get one longer reduction instead of many
short ones.  ``defer_wgrad=False`` keeps the per-chunk accumulation.

With ``recompute`` the activations are not kept between the forward and the
backward (MPipeMoE, "research method": recomputation to cut activation
memory): only the routing results are, and the backward re-runs each chunk's
permute and expert forward into one chunk's buffers before its backward, for
the cost of those kernels again.  The results are the saved mode's, bit for
bit (the same kernels on the same inputs).  This mode runs on one stream.

All buffers are allocated once, up front, by ``LayerPass``; ``forward`` and
``backward`` only launch work on the current CUDA stream and the side stream
joined to it (no allocation, no host synchronisation).  This module does no
arithmetic of its own.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import ops


def _pad4(n: int) -> int:
    return (n + 3) // 4 * 4


# CTA pairs of the per-chunk expert GEMMs when the chunks are pipelined (of the
# 76 a GB300 holds; 0 = all): the cap leaves SMs to the side stream's routing,
# permute, combine backward and router backward.  On the long-context workload
# 64 gave 88.3-88.6 ms per step against 90.0 ms with every pair (56: 92.2,
# 68: 88.7), on one box.
GEMM_UNITS_PIPELINED = 64


class LayerPass:
    """Preallocated buffers and launch sequence for one layer configuration.

    Parameters: T tokens, d model width, f expert hidden width, E experts,
    k experts per token, dtype (torch.bfloat16 or torch.float32), renorm,
    chunk (dispatch chunk cap; None = one chunk), pipeline (two-stream chunk
    pipelining when there is more than one chunk; False keeps one stream),
    recompute (keep only the routing between forward and backward and re-run
    each chunk's permute and expert forward in the backward; one stream),
    defer_wgrad (one weight-gradient pass over all chunks after the last
    chunk's backward; default: with more than one chunk, unless recompute),
    gather (the permute fused into the expert GEMMs' operand loads: no X_perm
    is written; the first GEMM and the dW1 GEMM read x through the dispatch's
    perm.  False: moe_permute writes X_perm and the GEMMs read it),
    gemm_units (with the chunk pipeline: the CTA pairs the per-chunk expert
    GEMMs of the forward and of the backward's data half may use, leaving the
    other SMs to the side stream's routing, permute, combine backward and
    router backward; None = GEMM_UNITS_PIPELINED, 0 = all.  The weight
    gradients always use every pair)."""

    def __init__(self, T: int, d: int, f: int, E: int, k: int, dtype: torch.dtype,
                 renorm: int, chunk: Optional[int] = None, device="cuda",
                 pipeline: bool = True, recompute: bool = False,
                 defer_wgrad: Optional[bool] = None, gather: bool = False,
                 gemm_units: Optional[int] = None):
        self.T, self.d, self.f, self.E, self.k = T, d, f, E, k
        self.dtype, self.renorm = dtype, int(renorm)
        C = chunk if chunk else T
        if C % 4 and C < T:
            raise ValueError("chunk must be a multiple of 4")
        self.C = C
        self.chunks = [(c0, min(T, c0 + C)) for c0 in range(0, T, C)] or [(0, 0)]
        nch = len(self.chunks)
        self.recompute = bool(recompute)
        self.pipeline = bool(pipeline) and nch > 1 and not self.recompute
        if defer_wgrad is None:
            defer_wgrad = nch > 1
        self.defer_wgrad = bool(defer_wgrad) and not self.recompute
        self.gather = bool(gather)
        if gemm_units is None:
            gemm_units = GEMM_UNITS_PIPELINED if self.pipeline else 0
        self.gemm_units = int(gemm_units) if self.pipeline else 0
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
        # activations: of every chunk (kept for the backward), or of one chunk
        # (recompute)
        R = C * k if self.recompute else T * k
        self.X_perm = None if self.gather else z(R, d)
        self.G = z(R, f)
        self.A = z(R, f)
        self.Y_perm = z(R, d)
        self._params = None   # recompute: the forward's W1, b1, W2, b2
        self.y = z(T, d)
        # backward
        self.dw = z(T, k, dt=f32)
        self.dx = z(T, d)
        nbuf = 2 if self.pipeline else 1
        if self.defer_wgrad:
            # every chunk's rows, kept for the one weight-gradient pass
            self.dY_perm = z(T * k, d)
            self.dH = z(T * k, f)
            self.chunk_T = [c1 - c0 for c0, c1 in self.chunks]
            self.wshape = ops.make_shape(T, d, f, E, k, dtype, renorm)
            # scratch of the weight-gradient pass (split reductions; fp32 partials)
            wn = ops.moe_expert_ffn_bwd_weights_workspace_size(self.wshape, self.chunk_T)
            self.wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=dev)
        else:
            self.dY_perm = z(nbuf, C * k, d)
            if self.gather:
                # per chunk: dH for the weight half, which reads x through perm
                self.dH = z(nbuf, C * k, f)
                self.wshapes = [ops.make_shape(c1 - c0, d, f, E, k, dtype, renorm)
                                for c0, c1 in self.chunks]
                wn = max(ops.moe_expert_ffn_bwd_weights_workspace_size(
                    ws_, [c1 - c0]) for ws_, (c0, c1) in zip(self.wshapes, self.chunks))
                self.wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=dev)
        self.dX_perm = z(nbuf, C * k, d)
        self.dW1 = z(E, f, d, dt=f32)
        self.db1 = z(E, f, dt=f32)
        self.dW2 = z(E, d, f, dt=f32)
        self.db2 = z(E, d, dt=f32)
        self.dWg = z(E, d, dt=f32)
        ws = max(ops.moe_workspace_size(s) for s in self.shapes)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        if self.pipeline:
            self.side = torch.cuda.Stream(device=dev)
            self.ws2 = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
            ev = lambda: [torch.cuda.Event() for _ in range(nch)]  # noqa: E731
            self._ev_routed, self._ev_cb, self._ev_ffn, self._ev_rb = ev(), ev(), ev(), ev()
            self._ev_fwd = ev()
            self._ev_fork, self._ev_join = torch.cuda.Event(), torch.cuda.Event()

    # -- per-chunk views ------------------------------------------------------------
    def _rows(self, t: torch.Tensor, c0: int, c1: int, mult: int = 1) -> torch.Tensor:
        return t[c0 * mult:c1 * mult]

    def _act(self, t: torch.Tensor, c0: int, c1: int) -> torch.Tensor:
        """A chunk's rows of an activation buffer (X_perm, G, A, Y_perm)."""
        if self.recompute:
            return t[:(c1 - c0) * self.k]
        return t[c0 * self.k:c1 * self.k]

    def forward(self, x, Wg, W1, b1, W2, b2, beta=None, compute_logits: bool = True,
                logits: Optional[torch.Tensor] = None):
        """x [T,d]; Wg [E,d]; W1 [E,f,d]; b1 [E,f]; W2 [E,d,f]; b2 [E,d]
        (storage dtype); beta [E] fp32 or None.  With compute_logits False the
        router logits are taken from ``logits`` [T,E] fp32 instead of x Wg^T.
        Returns y [T,d] (a buffer owned by this object)."""
        k = self.k
        if not compute_logits:
            self.logits.copy_(logits)
        if self.recompute:
            self._params = (W1, b1, W2, b2)
        main = torch.cuda.current_stream()
        if self.pipeline:
            self._ev_fork.record(main)
            self.side.wait_event(self._ev_fork)

        def combine(ci):       # A6 of chunk ci
            c0, c1 = self.chunks[ci]
            ops.moe_combine_fwd(self.shapes[ci], self._act(self.Y_perm, c0, c1),
                                self._rows(self.pos, c0, c1), self._rows(self.w, c0, c1),
                                self._rows(self.y, c0, c1))

        prev = None            # pipelined: the chunk whose combine is still due
        for ci, ((c0, c1), s) in enumerate(zip(self.chunks, self.shapes)):
            if c1 == c0:
                continue
            xc = self._rows(x, c0, c1)
            pos = self._rows(self.pos, c0, c1)
            perm = self._rows(self.perm, c0, c1, k)
            offs = self.offsets[ci]
            # routing and permute of this chunk: on the side stream when
            # pipelined (chunks are independent there: own rows, own workspace)
            with torch.cuda.stream(self.side if self.pipeline else main):
                ops.moe_route(s, xc, Wg, beta, self._rows(self.logits, c0, c1),
                              int(compute_logits), self._rows(self.idx, c0, c1),
                              self._rows(self.w, c0, c1), self.counts[ci], offs, pos, perm,
                              self.ws2 if self.pipeline else self.ws, self.status)
                if not self.gather:
                    ops.moe_permute(s, xc, pos, self._act(self.X_perm, c0, c1))
                if self.pipeline:
                    self._ev_routed[ci].record(self.side)
                    # the previous chunk's combine, after its expert GEMMs and
                    # after this chunk's routing (which runs beside them)
                    if prev is not None:
                        self.side.wait_event(self._ev_fwd[prev])
                        combine(prev)
            if self.pipeline:
                main.wait_event(self._ev_routed[ci])
            Yp = self._act(self.Y_perm, c0, c1)
            ops.moe_set_gemm_max_units(self.gemm_units)
            if self.gather:   # A4 fused into A5: x rows through perm
                ops.moe_expert_ffn_fwd_gather(s, xc, perm, offs, W1, b1, W2, b2,
                                              self._act(self.G, c0, c1), self._act(self.A, c0, c1),
                                              Yp, self.ws, self.status)
            else:
                ops.moe_expert_ffn_fwd(s, self._act(self.X_perm, c0, c1), offs, W1, b1, W2, b2,
                                       self._act(self.G, c0, c1), self._act(self.A, c0, c1), Yp,
                                       self.ws, self.status)
            ops.moe_set_gemm_max_units(0)
            if self.pipeline:
                self._ev_fwd[ci].record(main)
                prev = ci
            else:
                combine(ci)
        if self.pipeline:
            if prev is not None:
                with torch.cuda.stream(self.side):
                    self.side.wait_event(self._ev_fwd[prev])
                    combine(prev)
            self._ev_join.record(self.side)
            main.wait_event(self._ev_join)
        return self.y

    def backward(self, dy, x, Wg, W1, W2):
        """Backward of the last ``forward``: dy [T,d].  Fills dx, dw, dW1, db1,
        dW2, db2, dWg (buffers owned by this object)."""
        k = self.k
        main = torch.cuda.current_stream()
        live = [ci for ci, (c0, c1) in enumerate(self.chunks) if c1 > c0]

        def views(ci):
            c0, c1 = self.chunks[ci]
            n = (c1 - c0) * k
            b = ci % 2 if self.pipeline else 0
            dYp = self.dY_perm[c0 * k:c1 * k] if self.defer_wgrad else self.dY_perm[b, :n]
            return c0, c1, dYp, self.dX_perm[b, :n]

        def combine_bwd(ci):   # A7: dY_perm and dw of chunk ci
            c0, c1, dYp, _ = views(ci)
            ops.moe_combine_bwd(self.shapes[ci], self._rows(dy, c0, c1),
                                self._act(self.Y_perm, c0, c1), self._rows(self.pos, c0, c1),
                                self._rows(self.w, c0, c1), dYp, self._rows(self.dw, c0, c1))

        def ffn_bwd(ci):       # A8: dX_perm of chunk ci; dW1, db1, dW2, db2 accumulate
            c0, c1, dYp, dXp = views(ci)
            if self.defer_wgrad:   # the activation half; db1 accumulates here
                ops.moe_set_gemm_max_units(self.gemm_units)
                ops.moe_expert_ffn_bwd_data(self.shapes[ci], dYp, self._act(self.G, c0, c1),
                                            self.offsets[ci], W1, W2, self.dH[c0 * k:c1 * k],
                                            dXp, self.db1, int(ci > 0), self.ws, self.status)
                ops.moe_set_gemm_max_units(0)
                return
            if self.gather:   # data half, then the weight half reading x through perm
                dH = self.dH[ci % 2 if self.pipeline else 0, :(c1 - c0) * k]
                ops.moe_set_gemm_max_units(self.gemm_units)
                ops.moe_expert_ffn_bwd_data(self.shapes[ci], dYp, self._act(self.G, c0, c1),
                                            self.offsets[ci], W1, W2, dH, dXp, self.db1,
                                            int(ci > 0), self.ws, self.status)
                ops.moe_set_gemm_max_units(0)
                ops.moe_expert_ffn_bwd_weights_gather(
                    self.wshapes[ci], [c1 - c0], self.offsets[ci:ci + 1], dYp,
                    self._rows(x, c0, c1), self._rows(self.perm, c0, c1, k), (c1 - c0) * k, dH,
                    self._act(self.A, c0, c1), self.dW1, self.dW2, self.db2, int(ci > 0),
                    self.wws, self.status)
                return
            ops.moe_expert_ffn_bwd(self.shapes[ci], dYp, self._act(self.X_perm, c0, c1),
                                   self._act(self.G, c0, c1), self._act(self.A, c0, c1),
                                   self.offsets[ci], W1, W2, dXp, self.dW1, self.db1, self.dW2,
                                   self.db2, int(ci > 0), self.ws, self.status)

        def route_bwd(ci, ws):  # A9 (permute backward) fused into A10; dWg accumulates
            c0, c1, _, dXp = views(ci)
            ops.moe_route_bwd(self.shapes[ci], self._rows(self.dw, c0, c1),
                              self._rows(self.logits, c0, c1), self._rows(self.idx, c0, c1),
                              self._rows(self.w, c0, c1), self._rows(self.perm, c0, c1, k),
                              self.offsets[ci], self._rows(x, c0, c1), Wg, dXp,
                              self._rows(self.pos, c0, c1), self._rows(self.dx, c0, c1),
                              self.dWg, int(ci > 0), ws, self.status)

        def refill(ci):        # recompute: A4 and A5 of chunk ci again
            c0, c1 = self.chunks[ci]
            W1_, b1_, W2_, b2_ = self._params
            s = self.shapes[ci]
            if self.gather:
                ops.moe_expert_ffn_fwd_gather(s, self._rows(x, c0, c1),
                                              self._rows(self.perm, c0, c1, k), self.offsets[ci],
                                              W1_, b1_, W2_, b2_, self._act(self.G, c0, c1),
                                              self._act(self.A, c0, c1),
                                              self._act(self.Y_perm, c0, c1), self.ws,
                                              self.status)
                return
            Xp = self._act(self.X_perm, c0, c1)
            ops.moe_permute(s, self._rows(x, c0, c1), self._rows(self.pos, c0, c1), Xp)
            ops.moe_expert_ffn_fwd(s, Xp, self.offsets[ci], W1_, b1_, W2_, b2_,
                                   self._act(self.G, c0, c1), self._act(self.A, c0, c1),
                                   self._act(self.Y_perm, c0, c1), self.ws, self.status)

        if self.recompute and self._params is None:
            raise RuntimeError("recompute: backward needs the forward's parameters")
        def weights():         # A8, weight half: every chunk's rows in one pass
            if self.defer_wgrad and self.gather:   # X through each chunk's perm
                ops.moe_expert_ffn_bwd_weights_gather(self.wshape, self.chunk_T, self.offsets,
                                                      self.dY_perm, x, self.perm, self.C * k,
                                                      self.dH, self.A, self.dW1, self.dW2,
                                                      self.db2, 0, self.wws, self.status)
            elif self.defer_wgrad:
                ops.moe_expert_ffn_bwd_weights(self.wshape, self.chunk_T, self.offsets,
                                               self.dY_perm, self.X_perm, self.dH, self.A,
                                               self.dW1, self.dW2, self.db2, 0, self.wws,
                                               self.status)

        if not self.pipeline:
            for ci in live:
                if self.recompute:
                    refill(ci)
                combine_bwd(ci)
                ffn_bwd(ci)
                route_bwd(ci, self.ws)
            weights()
            return self.dx
        # two streams: the side stream runs combine backward one chunk ahead and
        # router backward one chunk behind the current stream's expert backward
        side = self.side
        self._ev_fork.record(main)
        side.wait_event(self._ev_fork)
        with torch.cuda.stream(side):
            combine_bwd(live[0])
            self._ev_cb[live[0]].record(side)
        for i, ci in enumerate(live):
            main.wait_event(self._ev_cb[ci])
            if i >= 2:
                main.wait_event(self._ev_rb[live[i - 2]])   # its dX_perm buffer is free
            ffn_bwd(ci)
            self._ev_ffn[ci].record(main)
            with torch.cuda.stream(side):
                if i + 1 < len(live):
                    if i >= 1 and not self.defer_wgrad:
                        side.wait_event(self._ev_ffn[live[i - 1]])   # its dY_perm buffer is free
                    combine_bwd(live[i + 1])
                    self._ev_cb[live[i + 1]].record(side)
                side.wait_event(self._ev_ffn[ci])
                route_bwd(ci, self.ws2)
                self._ev_rb[ci].record(side)
        weights()
        self._ev_join.record(side)
        main.wait_event(self._ev_join)
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

