"""Failure detection on the GPU without a GPU fault: a bounded wait on a flag
that nothing sets must come back with MOE_ERR_TIMEOUT in the status word
while the context stays usable; bad arguments never launch."""
import time

import pytest
import torch

from mixture_experts_layer_11_gb300 import ops

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    ops.moe_debug_bounded_wait(200_000_000, st)  # 0.2 s
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(st.item()) == ops.MOE_ERR_TIMEOUT
    assert 0.15 < dt < 5.0
    # the context still works
    x = torch.arange(10, device="cuda").sum()
    assert int(x.item()) == 45


def test_first_error_wins():
    st = torch.full((1,), ops.MOE_ERR_NONFINITE, dtype=torch.int32, device="cuda")
    ops.moe_debug_bounded_wait(1_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == ops.MOE_ERR_NONFINITE


def test_invalid_arguments_raise_without_launch():
    s = ops.make_shape(100, 64, 64, 4, 1, "f32", 0)
    x = torch.zeros(100, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(ops.MoEError) as ei:
        ops.moe_permute(s, x, None, x)
    assert ei.value.code == ops.MOE_ERR_INVALID


def test_wrong_dtype_buffer_rejected_at_the_binding():
    # an fp32 gradient slot given a float64 tensor would be written as fp32
    # bit patterns into doubles; the binding refuses it before any launch
    s = ops.make_shape(8, 64, 64, 4, 1, "f32", 0)
    dw = torch.zeros(8, 1, dtype=torch.float64, device="cuda")
    y = torch.zeros(8, 64, dtype=torch.float32, device="cuda")
    pos = torch.zeros(8, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(ops.MoEError) as ei:
        ops.moe_combine_bwd(s, y, y, pos, dw, y, dw)
    assert ei.value.code == ops.MOE_ERR_INVALID


@pytest.mark.parametrize("shape", ["pairs", "single_cta"])
def test_gemm_timeout_teardown(shape, monkeypatch):
    """The grouped GEMM's own timeout path.  With MOE_DEBUG_GEMM_WITHHOLD the
    producer of the CTA (pair) holding work unit 0 issues nothing from K block
    1 on (no expect_tx and no copy for that stage, so nothing is left in
    flight for it).  That CTA's MMA warp waits on the stage for the default
    1 s, raises the abort, the other roles stop, the copies already issued
    are waited for, tensor memory is freed, and MOE_ERR_TIMEOUT lands in the
    status word.  Afterwards the context is usable and a normal call gives
    the same result as before."""
    from mixture_experts_layer_11_gb300 import synth
    if shape == "single_cta":
        monkeypatch.setenv("MOE_GEMM_PAIR", "0")
    T, d, f, E, k = 600, 256, 512, 4, 2
    cfg = synth.MoEConfig("t", T=T, d=d, f=f, E=E, k=k, renorm=1, dtype="bf16")
    inp = {n: (v.cuda() if v is not None else None)
           for n, v in synth.make_inputs(cfg, seed=3, random_bias=True).items()}
    P = T * k
    offs = torch.tensor([0, 500, 600, 1100, P], dtype=torch.int32, device="cuda")
    X = torch.randn(P, d, device="cuda").to(torch.bfloat16)
    s = ops.make_shape(T, d, f, E, k, "bf16", 1)
    ws = torch.empty(ops.moe_workspace_size(s), dtype=torch.uint8, device="cuda")

    def run(st):
        G, A, Y = (torch.empty(P, n, dtype=torch.bfloat16, device="cuda") for n in (f, f, d))
        ops.moe_expert_ffn_fwd(s, X, offs, inp["W1"], inp["b1"], inp["W2"], inp["b2"], G, A, Y,
                               ws, st)
        return G, A, Y

    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    good = run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    monkeypatch.setenv("MOE_DEBUG_GEMM_WITHHOLD", "0:1")
    t0 = time.time()
    run(st)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(st.item()) == ops.MOE_ERR_TIMEOUT
    assert 0.9 < dt < 20.0
    monkeypatch.delenv("MOE_DEBUG_GEMM_WITHHOLD")
    st.zero_()
    again = run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a, b in zip(good, again):
        assert torch.equal(a, b)
