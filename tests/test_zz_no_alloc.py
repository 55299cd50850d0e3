"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such a caller (for example a plug-in whose host framework owns every
allocation and passes it only the tensors it reads and writes) has no
workspace to give the library, so this entry point keeps the histogram
scratch in a fixed array inside libmoe.so.  These tests call it through the C
ABI and check it against moe_route (which takes a caller workspace) on the
same inputs, on calls in a row with different inputs, so that each call runs
on scratch the one before left behind: a smaller histogram after a larger one,
then a larger one again, then an empty batch (T = 0), whose counts and
offsets must come out as zeros whatever the array holds.  Integer outputs must match
bit for bit; logits and gate weights come from the same kernels and are held
to the fp32 tolerance of the other GPU tests."""
import pytest
import torch

from mixture_experts_layer_11_gb300 import ops, synth
from parity_util import assert_close, assert_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buffers(T, E, k):
    z = lambda *s, dt: torch.empty(*s, dtype=dt, device=DEV)  # noqa: E731
    return dict(logits=z(T, E, dt=torch.float32), idx=z(T, k, dt=torch.int32),
                w=z(T, k, dt=torch.float32), counts=z(E, dt=torch.int32),
                offsets=z(E + 1, dt=torch.int32), pos=z(T, k, dt=torch.int32),
                perm=z(max(T * k, 1), dt=torch.int32),
                status=torch.zeros(1, dtype=torch.int32, device=DEV))


CALLS = [  # calls in a row, different shapes and inputs
    synth.CONFIGS["longctx128_bf16"].scaled(T=3000, d=256, chunk=None),   # 128 x 47 entries
    synth.CONFIGS["moe_s_bf16"].scaled(T=1111, d=768),                    # 8 x 18
    synth.CONFIGS["longctx128_bf16"].scaled(T=9000, d=128, chunk=None),   # 128 x 141
]


def test_noalloc_route_matches_route_on_calls_in_a_row():
    for i, cfg in enumerate(CALLS):
        inp = synth.make_inputs(cfg, seed=10 + i)
        x, Wg = inp["x"].to(DEV), inp["Wg"].to(DEV)
        beta = None if inp["beta"] is None else inp["beta"].to(DEV)
        s = ops.make_shape(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.dtype, cfg.renorm)
        ref = _buffers(cfg.T, cfg.E, cfg.k)
        ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device=DEV)
        ops.moe_route(s, x, Wg, beta, ref["logits"], 1, ref["idx"], ref["w"], ref["counts"],
                      ref["offsets"], ref["pos"], ref["perm"], ws, ref["status"])
        got = _buffers(cfg.T, cfg.E, cfg.k)
        ops.moe_route_noalloc(s, x, Wg, beta, got["logits"], 1, got["idx"], got["w"],
                              got["counts"], got["offsets"], got["pos"], got["perm"],
                              got["status"])
        torch.cuda.synchronize()
        assert int(ref["status"].item()) == 0 and int(got["status"].item()) == 0
        for n in ("idx", "counts", "offsets", "pos", "perm"):
            assert_equal(f"call {i} {n}", got[n], ref[n].cpu().numpy())
        assert_close(f"call {i} logits", got["logits"], ref["logits"].cpu(), "f32")
        assert_close(f"call {i} w", got["w"], ref["w"].cpu(), "f32")


def test_noalloc_empty_batch_after_a_full_one():
    # a non-empty call leaves its histogram in the array; T = 0 must still
    # give all-zero counts and offsets (only the scan runs)
    cfg = synth.CONFIGS["moe_s_bf16"].scaled(T=2000, d=256)
    inp = synth.make_inputs(cfg, seed=21)
    s = ops.make_shape(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.dtype, cfg.renorm)
    b = _buffers(cfg.T, cfg.E, cfg.k)
    ops.moe_route_noalloc(s, inp["x"].to(DEV), inp["Wg"].to(DEV), None, b["logits"], 1,
                          b["idx"], b["w"], b["counts"], b["offsets"], b["pos"], b["perm"],
                          b["status"])
    s0 = ops.make_shape(0, cfg.d, cfg.f, cfg.E, cfg.k, cfg.dtype, cfg.renorm)
    counts = torch.full((cfg.E,), -1, dtype=torch.int32, device=DEV)
    offsets = torch.full((cfg.E + 1,), -1, dtype=torch.int32, device=DEV)
    ops.moe_route_noalloc(s0, None, None, None, None, 1, None, None, counts, offsets, None,
                          None, b["status"])
    torch.cuda.synchronize()
    assert int(b["status"].item()) == 0
    assert int(b["counts"].sum().item()) == cfg.T * cfg.k
    assert_equal("counts (T = 0)", counts, torch.zeros(cfg.E, dtype=torch.int32).numpy())
    assert_equal("offsets (T = 0)", offsets, torch.zeros(cfg.E + 1, dtype=torch.int32).numpy())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # E * ceil(T / 64) > MOE_ROUTE_NOALLOC_MAX_SCRATCH: refused on the host
    E = 256
    T = 64 * (ops.ROUTE_NOALLOC_MAX_SCRATCH // E) + 64
    s = ops.make_shape(T, 64, 64, E, 1, "f32", 0)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    with pytest.raises(ops.MoEError) as ei:
        ops.moe_route_noalloc(s, None, None, None, dummy.view(torch.float32), 0, dummy,
                              dummy.view(torch.float32), dummy, dummy, dummy, dummy, dummy)
    assert ei.value.code == ops.MOE_ERR_UNSUPPORTED
