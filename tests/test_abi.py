"""The C-ABI library loads, exports every entry point include/moe.h declares,
and rejects bad arguments on the host before launching anything (no GPU
needed: these calls return before any CUDA call)."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_11_gb300 import build as mbuild
from mixture_experts_layer_11_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return ops.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn_fwd", "moe_expert_ffn_bwd",
              "moe_combine_fwd", "moe_combine_bwd", "moe_route_bwd", "moe_workspace_size",
              "moe_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(ops.ENTRY_POINTS) >= set(_declared())


def test_status_strings(lib):
    for code in range(6):
        s = ops.moe_status_string(code)
        assert s.startswith("MOE_")
    assert "unknown" in ops.moe_status_string(99)


def _shape(**kw):
    base = dict(T=1024, d=256, f=512, E=8, k=2, dtype="bf16", renorm=1)
    base.update(kw)
    return ops.make_shape(**base)


def test_workspace_size(lib):
    s = _shape()
    n = ops.moe_workspace_size(s)
    # at least dH of the expert backward: T*k*f bf16
    assert n >= 1024 * 2 * 512 * 2
    assert ops.moe_workspace_size(_shape(E=0)) == 0
    assert ops.moe_workspace_size(_shape(k=9, E=8)) == 0
    assert ops.moe_workspace_size(_shape(T=0)) > 0


@pytest.mark.parametrize("bad", [dict(E=0), dict(E=300), dict(k=0), dict(k=17, E=32),
                                 dict(k=5, E=4), dict(T=-1), dict(d=0), dict(dtype=7),
                                 dict(renorm=2)])
def test_invalid_shapes_rejected(lib, bad):
    s = _shape(**bad)
    code = lib.moe_permute(ctypes.byref(s), 16, 16, 16, None)
    assert code == ops.MOE_ERR_INVALID


def test_unsupported_shapes(lib):
    # bf16 expert GEMMs need d, f multiples of 64
    s = _shape(d=72)
    code = lib.moe_expert_ffn_fwd(ctypes.byref(s), *([16] * 10), None, None)
    assert code == ops.MOE_ERR_UNSUPPORTED
    s = _shape(d=12)  # rows must be whole 16-byte vectors
    assert lib.moe_permute(ctypes.byref(s), 16, 16, 16, None) == ops.MOE_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected(lib):
    s = _shape()
    assert lib.moe_permute(None, 16, 16, 16, None) == ops.MOE_ERR_INVALID
    assert lib.moe_permute(ctypes.byref(s), None, 16, 16, None) == ops.MOE_ERR_INVALID
    assert lib.moe_permute(ctypes.byref(s), 24, 16, 16, None) == ops.MOE_ERR_INVALID
    assert lib.moe_combine_fwd(ctypes.byref(s), 16, 16, 8, 16, None) == ops.MOE_ERR_INVALID
    assert lib.moe_debug_bounded_wait(1000, None, None) == ops.MOE_ERR_INVALID
    with pytest.raises(ops.MoEError) as ei:
        ops.moe_permute(s, 16, None, 16, stream=0)
    assert ei.value.code == ops.MOE_ERR_INVALID


def test_empty_calls_do_nothing(lib):
    s = _shape(T=0)
    # no tokens: nothing to launch, bad (dangling) buffers are never touched
    assert lib.moe_permute(ctypes.byref(s), 16, 16, 16, None) == ops.MOE_OK
    assert lib.moe_combine_fwd(ctypes.byref(s), 16, 16, None, 16, None) == ops.MOE_OK
    assert lib.moe_combine_bwd(ctypes.byref(s), 16, 16, 16, 16, 16, 16, None) == ops.MOE_OK


def test_gather_entry_points_reject_bad_arguments(lib):
    """The fused-permute calls check their extra arguments on the host: a null
    perm, a perm stride shorter than a chunk's entries."""
    s = _shape()
    assert lib.moe_expert_ffn_fwd_gather(ctypes.byref(s), 16, None, 16, 16, None, 16, None,
                                         16, 16, 16, 16, 16, None) == ops.MOE_ERR_INVALID
    T = ctypes.c_int64(int(s.T))
    arr = (ctypes.c_int64 * 1)(T.value)
    short = int(s.T) * int(s.k) - 1
    args = [16, 16, ctypes.c_int64(short), 16, 16, 16, 16, 16, 0, 16, 4096, 16, None]
    assert lib.moe_expert_ffn_bwd_weights_gather(ctypes.byref(s), 1, arr, 16, 12, 16, *args) \
        == ops.MOE_ERR_INVALID
    args[1] = None   # no perm
    args[2] = ctypes.c_int64(int(s.T) * int(s.k))
    assert lib.moe_expert_ffn_bwd_weights_gather(ctypes.byref(s), 1, arr, 16, 12, 16, *args) \
        == ops.MOE_ERR_INVALID


def test_gemm_max_units_option(lib):
    assert lib.moe_set_gemm_max_units(-1) == ops.MOE_ERR_INVALID
    assert lib.moe_set_gemm_max_units(8) == ops.MOE_OK
    assert lib.moe_set_gemm_max_units(0) == ops.MOE_OK
