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
