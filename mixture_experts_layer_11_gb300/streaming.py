"""The MoE layer pass with the expert weights kept in host memory and streamed
to the GPU one group of experts at a time, overlapped with the previous
group's compute (ES-MoE: Scaling Beyond the GPU Memory Limit for Large
Mixture-of-Experts Model Training, review, section 3, "expert-wise offloading
and processing": experts are uploaded one after another and each upload
overlaps the previous expert's computation).  On a Grace-Blackwell node the
host memory is LPDDR behind NVLink-C2C, so an expert count whose weights (and
fp32 weight gradients) exceed HBM still trains on one GPU.

Order of a step (expert-major, so that each expert's weights cross the link
once per pass, not once per dispatch chunk):

forward:  route + permute every chunk; for each expert group g: wait for its
          weights (copy stream), run the expert FFN of g over every chunk's
          rows of g's experts, release the slot for group g+2's upload; then
          combine every chunk.
backward: combine backward of every chunk; for each group g (weights streamed
          again): the data half of the expert backward over every chunk
          (dH, dX_perm rows of g's experts, db1 of g), then the weight half over
          all chunks at once into a device slot, whose fp32 dW1 / dW2 are read
          back to pinned host memory on the copy stream; then the router
          backward (with the permute backward) of every chunk.

Two device slots hold a group's W1, b1, W2, b2 (and two more its dW1, dW2);
events order every reuse.  The per-expert kernels are the ones of
``layer.LayerPass``: a group is an expert sub-range of the same entry points
(offsets, weights and bias gradients at the group's first expert).  This
module does no arithmetic of its own.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import ops


def _pad4(n: int) -> int:
    return (n + 3) // 4 * 4


class ExpertStreamingPass:
    """Preallocated device buffers for one layer configuration whose expert
    weights live in pinned host memory.  ``group`` experts are streamed at a
    time (a multiple of 4).  The host weight gradients dW1_host [E,f,d] and
    dW2_host [E,d,f] (fp32, pinned) are filled by ``backward``; db1, db2, dWg
    and the activation gradients stay on the device."""

    def __init__(self, T: int, d: int, f: int, E: int, k: int, dtype: torch.dtype,
                 renorm: int, chunk: Optional[int] = None, group: int = 16, device="cuda"):
        if group % 4 or group < 4:
            raise ValueError("group must be a positive multiple of 4")
        self.T, self.d, self.f, self.E, self.k = T, d, f, E, k
        self.dtype, self.renorm = dtype, int(renorm)
        C = chunk if chunk else T
        if C % 4 and C < T:
            raise ValueError("chunk must be a multiple of 4")
        self.chunks = [(c0, min(T, c0 + C)) for c0 in range(0, T, C)] or [(0, 0)]
        nch = len(self.chunks)
        self.groups = [(e0, min(E, e0 + group)) for e0 in range(0, E, group)]
        dev = torch.device(device)
        f32, i32 = torch.float32, torch.int32
        z = lambda *s, dt=dtype: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.shapes = [ops.make_shape(c1 - c0, d, f, E, k, dtype, renorm) for c0, c1 in self.chunks]
        # routing and activations of every chunk
        self.logits = z(T, E, dt=f32)
        self.idx = z(T, k, dt=i32)
        self.w = z(T, k, dt=f32)
        self.pos = z(T, k, dt=i32)
        self.perm = z(T * k, dt=i32)
        self.counts = z(nch, _pad4(E), dt=i32)
        self.offsets = z(nch, _pad4(E + 1), dt=i32)
        self.X_perm = z(T * k, d)
        self.G = z(T * k, f)
        self.A = z(T * k, f)
        self.Y_perm = z(T * k, d)
        self.y = z(T, d)
        self.dw = z(T, k, dt=f32)
        self.dx = z(T, d)
        self.dY_perm = z(T * k, d)
        self.dX_perm = z(T * k, d)
        self.dH = z(T * k, f)
        self.db1 = z(E, f, dt=f32)
        self.db2 = z(E, d, dt=f32)
        self.dWg = z(E, d, dt=f32)
        # streamed weights and weight gradients: two slots each
        self.W1s = [z(group, f, d) for _ in range(2)]
        self.b1s = [z(group, f) for _ in range(2)]
        self.W2s = [z(group, d, f) for _ in range(2)]
        self.b2s = [z(group, d) for _ in range(2)]
        self.dW1s = [z(group, f, d, dt=f32) for _ in range(2)]
        self.dW2s = [z(group, d, f, dt=f32) for _ in range(2)]
        self.dW1_host = torch.empty(E, f, d, dtype=f32, pin_memory=True)
        self.dW2_host = torch.empty(E, d, f, dtype=f32, pin_memory=True)
        ws = max(ops.moe_workspace_size(s) for s in self.shapes)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        # the expert FFN calls see a chunk as T*k rows with k = 1 and E = the group
        self.rows = [(c1 - c0) * k for c0, c1 in self.chunks]
        gshape = ops.make_shape(T * k, d, f, group, 1, dtype, renorm)
        wn = ops.moe_expert_ffn_bwd_weights_workspace_size(gshape, self.rows)
        self.wws = torch.empty(max(wn, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.copy = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        self._ev_loaded, self._ev_used, self._ev_grad, self._ev_read = ev(), ev(), ev(), ev()

    def _gshape(self, ci: int, e0: int, e1: int, rows: Optional[int] = None):
        return ops.make_shape(self.rows[ci] if rows is None else rows, self.d, self.f, e1 - e0, 1,
                              self.dtype, self.renorm)

    def _act(self, t, ci):
        c0, c1 = self.chunks[ci]
        return t[c0 * self.k:c1 * self.k]

    def _upload(self, gi: int, host: dict, names):
        """Copy group gi's weights into slot gi % 2 on the copy stream, after
        the compute that used the slot last."""
        e0, e1 = self.groups[gi]
        s = gi % 2
        slots = {"W1": self.W1s, "b1": self.b1s, "W2": self.W2s, "b2": self.b2s}
        with torch.cuda.stream(self.copy):
            self.copy.wait_event(self._ev_used[s])
            for n in names:
                slots[n][s][:e1 - e0].copy_(host[n][e0:e1], non_blocking=True)
            self._ev_loaded[s].record(self.copy)

    def _release_slots(self):
        main = torch.cuda.current_stream()
        for s in range(2):
            self._ev_used[s].record(main)

    def forward(self, x, Wg, W1_host, b1_host, W2_host, b2_host, beta=None):
        """x [T,d], Wg [E,d] on the device; W1_host [E,f,d], b1_host [E,f],
        W2_host [E,d,f], b2_host [E,d] in pinned host memory; beta [E] fp32 or
        None.  Returns y [T,d]."""
        k = self.k
        main = torch.cuda.current_stream()
        host = dict(W1=W1_host, b1=b1_host, W2=W2_host, b2=b2_host)
        names = ("W1", "b1", "W2", "b2")
        self._release_slots()
        for gi in range(min(2, len(self.groups))):
            self._upload(gi, host, names)
        live = [ci for ci, (c0, c1) in enumerate(self.chunks) if c1 > c0]
        for ci in live:
            c0, c1 = self.chunks[ci]
            s = self.shapes[ci]
            ops.moe_route(s, x[c0:c1], Wg, beta, self.logits[c0:c1], 1, self.idx[c0:c1],
                          self.w[c0:c1], self.counts[ci], self.offsets[ci], self.pos[c0:c1],
                          self.perm[c0 * k:c1 * k], self.ws, self.status)
            ops.moe_permute(s, x[c0:c1], self.pos[c0:c1], self._act(self.X_perm, ci))
        for gi, (e0, e1) in enumerate(self.groups):
            sl = gi % 2
            main.wait_event(self._ev_loaded[sl])
            n = e1 - e0
            for ci in live:
                ops.moe_expert_ffn_fwd(self._gshape(ci, e0, e1), self._act(self.X_perm, ci),
                                       self.offsets[ci, e0:], self.W1s[sl][:n], self.b1s[sl][:n],
                                       self.W2s[sl][:n], self.b2s[sl][:n],
                                       self._act(self.G, ci), self._act(self.A, ci),
                                       self._act(self.Y_perm, ci), self.ws, self.status)
            self._ev_used[sl].record(main)
            if gi + 2 < len(self.groups):
                self._upload(gi + 2, host, names)
        for ci in live:
            c0, c1 = self.chunks[ci]
            ops.moe_combine_fwd(self.shapes[ci], self._act(self.Y_perm, ci), self.pos[c0:c1],
                                self.w[c0:c1], self.y[c0:c1])
        return self.y

    def backward(self, dy, x, Wg, W1_host, W2_host):
        """Backward of the last ``forward``: fills dx, dw, db1, db2, dWg on the
        device and dW1_host, dW2_host (read back on the copy stream; call
        ``synchronize`` or synchronise the device before reading them)."""
        k = self.k
        main = torch.cuda.current_stream()
        host = dict(W1=W1_host, W2=W2_host)
        names = ("W1", "W2")
        live = [ci for ci, (c0, c1) in enumerate(self.chunks) if c1 > c0]
        for ci in live:
            c0, c1 = self.chunks[ci]
            ops.moe_combine_bwd(self.shapes[ci], dy[c0:c1], self._act(self.Y_perm, ci),
                                self.pos[c0:c1], self.w[c0:c1], self._act(self.dY_perm, ci),
                                self.dw[c0:c1])
        self._release_slots()
        for s in range(2):
            self._ev_read[s].record(main)
        for gi in range(min(2, len(self.groups))):
            self._upload(gi, host, names)
        for gi, (e0, e1) in enumerate(self.groups):
            sl = gi % 2
            n = e1 - e0
            main.wait_event(self._ev_loaded[sl])
            for j, ci in enumerate(live):
                ops.moe_expert_ffn_bwd_data(self._gshape(ci, e0, e1), self._act(self.dY_perm, ci),
                                            self._act(self.G, ci), self.offsets[ci, e0:],
                                            self.W1s[sl][:n], self.W2s[sl][:n],
                                            self._act(self.dH, ci), self._act(self.dX_perm, ci),
                                            self.db1[e0:e1], int(j > 0), self.ws, self.status)
            self._ev_used[sl].record(main)
            if gi + 2 < len(self.groups):
                self._upload(gi + 2, host, names)
            # the gradient slot's previous contents have been read back
            main.wait_event(self._ev_read[sl])
            ops.moe_expert_ffn_bwd_weights(self._gshape(0, e0, e1, rows=self.T * k),
                                           [self.rows[ci] for ci in live],
                                           self.offsets[live[0]:live[-1] + 1, e0:] if live
                                           else self.offsets[:1, e0:],
                                           self.dY_perm, self.X_perm, self.dH, self.A,
                                           self.dW1s[sl][:n], self.dW2s[sl][:n],
                                           self.db2[e0:e1], 0, self.wws, self.status)
            self._ev_grad[sl].record(main)
            with torch.cuda.stream(self.copy):
                self.copy.wait_event(self._ev_grad[sl])
                self.dW1_host[e0:e1].copy_(self.dW1s[sl][:n], non_blocking=True)
                self.dW2_host[e0:e1].copy_(self.dW2s[sl][:n], non_blocking=True)
                self._ev_read[sl].record(self.copy)
        for j, ci in enumerate(live):
            c0, c1 = self.chunks[ci]
            ops.moe_route_bwd(self.shapes[ci], self.dw[c0:c1], self.logits[c0:c1],
                              self.idx[c0:c1], self.w[c0:c1], self.perm[c0 * k:c1 * k],
                              self.offsets[ci], x[c0:c1], Wg, self._act(self.dX_perm, ci),
                              self.pos[c0:c1], self.dx[c0:c1], self.dWg, int(j > 0), self.ws,
                              self.status)
        # the host gradients are complete once the copy stream has drained
        main.wait_stream(self.copy)
        return self.dx

    def check_status(self):
        """Synchronises and raises if a kernel reported a device-side error."""
        code = int(self.status.item())
        if code != ops.MOE_OK:
            raise ops.MoEError("device", code, ops.moe_status_string(code))
