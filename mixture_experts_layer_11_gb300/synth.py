"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers and fixes shapes; it contains none of
the layer's arithmetic.  Both the CUDA path (tests, benchmark) and the CPU
oracle take their inputs from here, so that they see identical values.

Workloads (the layer sizes the MoE systems in the literature train; all
inputs synthetic):

* ``tiny_f32``      T=256, d_model=64, d_ffn=128, E=4, top-1, fp32 throughout.
* ``moe_s_bf16``    T=8192 (8 x 1024), d=768, f=3072, E=8, top-2 renormalised
                    (the MoE-S layer shape of the ES-MoE throughput table).
* ``skewed64_bf16`` T=16384, d=768, f=3072, E=64, top-1 Switch-style gate,
                    logits shifted by 2*ln(Zipf(s=1.2) rank weight) so that a
                    few experts take most tokens and many take none.
* ``moe_l_bf16``    T=16384 (16 x 1024), d=2048, f=8192, E=16, top-2 renorm.
* ``longctx128_bf16`` T=262144, d=4096, f=1024, E=128, top-8 renorm, Zipf
                    s=1.1 logit shift, processed in dispatch chunks of at most
                    32768 tokens (the bounded dispatch chunk of PipelinedLLEP,
                    "Flattening Every Memory Peak in Long-Context MoE
                    Training", abstract).

Draw recipe (one ``torch.Generator`` seeded with ``seed``, tensors drawn in
this fixed order): x ~ N(0,1) [T,d]; Wg ~ N(0,1/d) [E,d]; W1 ~ N(0,1/d)
[E,f,d]; b1 [E,f]; W2 ~ N(0,1/f) [E,d,f]; b2 [E,d]; dy ~ N(0,1) [T,d].
Biases are zero unless ``random_bias`` is set (then N(0, 0.1^2), drawn in
their slot of the order).  bf16 workloads draw in fp32 and round to bf16.
The Zipf logit shift beta_e = c * ln((e+1)^-s) is a fixed input, not a
parameter.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    renorm: int
    dtype: str                     # "f32" or "bf16"
    zipf_s: Optional[float] = None  # Zipf exponent of the logit shift
    zipf_c: float = 2.0            # scale of the logit shift
    chunk: Optional[int] = None    # dispatch chunk cap (tokens)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def chunk_tokens(self) -> int:
        return self.chunk if self.chunk else self.T

    def scaled(self, **kw) -> "MoEConfig":
        """Same workload family at other sizes (for tests the oracle finishes
        in seconds)."""
        return dataclasses.replace(self, **kw)

    # Algorithmic work of one forward + backward pass (no padding, no dense
    # dispatch mask counted).
    def expert_flops(self) -> float:
        return 12.0 * self.T * self.k * self.d * self.f

    def router_flops(self) -> float:
        return 6.0 * self.T * self.d * self.E


CONFIGS = {
    c.name: c
    for c in [
        MoEConfig("tiny_f32", T=256, d=64, f=128, E=4, k=1, renorm=0, dtype="f32"),
        MoEConfig("moe_s_bf16", T=8192, d=768, f=3072, E=8, k=2, renorm=1, dtype="bf16"),
        MoEConfig("skewed64_bf16", T=16384, d=768, f=3072, E=64, k=1, renorm=0,
                  dtype="bf16", zipf_s=1.2),
        MoEConfig("moe_l_bf16", T=16384, d=2048, f=8192, E=16, k=2, renorm=1, dtype="bf16"),
        MoEConfig("longctx128_bf16", T=262144, d=4096, f=1024, E=128, k=8, renorm=1,
                  dtype="bf16", zipf_s=1.1, chunk=32768),
    ]
}


def zipf_logit_bias(E: int, s: float, c: float) -> torch.Tensor:
    """beta_e = c * ln((e+1)^-s), fp32 [E]."""
    return torch.tensor([c * (-s) * math.log(e + 1.0) for e in range(E)],
                        dtype=torch.float32)


def make_inputs(cfg: MoEConfig, seed: int = 0, device: str = "cpu",
                random_bias: bool = False) -> dict:
    """Draw every input of one forward + backward pass.

    Returns a dict of tensors in the workload's storage dtype (the logit
    shift ``beta`` is fp32 or None)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = cfg.torch_dtype

    def normal(shape, std):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(dt)

    def bias(shape):
        if random_bias:
            return normal(shape, 0.1)
        return torch.zeros(shape, device=device, dtype=dt)

    x = normal((cfg.T, cfg.d), 1.0)
    Wg = normal((cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d))
    W1 = normal((cfg.E, cfg.f, cfg.d), 1.0 / math.sqrt(cfg.d))
    b1 = bias((cfg.E, cfg.f))
    W2 = normal((cfg.E, cfg.d, cfg.f), 1.0 / math.sqrt(cfg.f))
    b2 = bias((cfg.E, cfg.d))
    dy = normal((cfg.T, cfg.d), 1.0)
    beta = None
    if cfg.zipf_s is not None:
        beta = zipf_logit_bias(cfg.E, cfg.zipf_s, cfg.zipf_c).to(device)
    return dict(x=x, Wg=Wg, W1=W1, b1=b1, W2=W2, b2=b2, dy=dy, beta=beta)


def make_logits(T: int, E: int, seed: int = 0, ties: bool = False) -> torch.Tensor:
    """Synthetic fp32 router logits for tests that feed identical logits to
    both sides.  With ``ties`` the values are small integers so that equal
    logits are frequent."""
    g = torch.Generator()
    g.manual_seed(seed)
    if ties:
        return torch.randint(-2, 3, (T, E), generator=g).to(torch.float32)
    return torch.randn((T, E), generator=g, dtype=torch.float32)
