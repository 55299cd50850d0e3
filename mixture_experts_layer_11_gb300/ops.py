"""Thin Python binding of libmoe.so (include/moe.h): same entry-point names,
argument marshalling only.  Every step of the layer runs in the library's CUDA
kernels; there is no Python or CPU fallback.  If the library has not been
built, the first call raises.

Tensors are torch CUDA tensors (any pointer-like argument may also be a raw
device address as an int, or None where the C ABI allows NULL).  Work is
enqueued on the current torch CUDA stream unless ``stream`` is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_NONFINITE = range(6)
MOE_F32, MOE_BF16 = 0, 1

ENTRY_POINTS = ("moe_status_string", "moe_workspace_size", "moe_route", "moe_permute",
                "moe_expert_ffn_fwd", "moe_combine_fwd", "moe_combine_bwd",
                "moe_expert_ffn_bwd", "moe_route_bwd", "moe_debug_bounded_wait",
                "moe_debug_gelu", "moe_route_noalloc", "moe_expert_ffn_bwd_data",
                "moe_expert_ffn_bwd_weights", "moe_expert_ffn_fwd_gather",
                "moe_expert_ffn_bwd_weights_gather", "moe_set_gemm_max_units",
                "moe_expert_ffn_bwd_weights_workspace_size")


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {msg}")
        self.code = code


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("renorm", ctypes.c_int32)]


def make_shape(T: int, d: int, f: int, E: int, k: int, dtype, renorm: int) -> moe_shape:
    if isinstance(dtype, torch.dtype):
        dt = MOE_BF16 if dtype == torch.bfloat16 else MOE_F32
    elif isinstance(dtype, str):
        dt = MOE_BF16 if dtype == "bf16" else MOE_F32
    else:
        dt = int(dtype)
    return moe_shape(int(T), int(d), int(f), int(E), int(k), dt, int(renorm))


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_SP = ctypes.POINTER(moe_shape)


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_status_string.argtypes = [ctypes.c_int]
            L.moe_workspace_size.restype = ctypes.c_size_t
            L.moe_workspace_size.argtypes = [_SP]
            L.moe_route.argtypes = [_SP, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P]
            L.moe_permute.argtypes = [_SP, _P, _P, _P, _P]
            L.moe_expert_ffn_fwd.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
            L.moe_combine_fwd.argtypes = [_SP, _P, _P, _P, _P, _P]
            L.moe_combine_bwd.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P]
            L.moe_expert_ffn_bwd.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, ctypes.c_int, _P, _P, _P]
            L.moe_route_bwd.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_int, _P, _P, _P]
            L.moe_debug_bounded_wait.argtypes = [ctypes.c_uint64, _P, _P]
            L.moe_debug_gelu.argtypes = [ctypes.c_int64, _P, _P, _P, ctypes.c_int, _P]
            L.moe_route_noalloc.argtypes = [_SP, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P, _P,
                                            _P, _P, _P, _P]
            L.moe_expert_ffn_bwd_data.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, _P,
                                                  ctypes.c_int, _P, _P, _P]
            L.moe_expert_ffn_bwd_weights.argtypes = [_SP, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_int64), _P,
                                                     ctypes.c_int, _P, _P, _P, _P, _P, _P, _P,
                                                     ctypes.c_int, _P, ctypes.c_size_t, _P, _P]
            L.moe_set_gemm_max_units.argtypes = [ctypes.c_int]
            L.moe_expert_ffn_fwd_gather.argtypes = [_SP] + [_P] * 13
            L.moe_expert_ffn_bwd_weights_gather.argtypes = [
                _SP, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), _P, ctypes.c_int, _P, _P,
                _P, ctypes.c_int64, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P,
                _P]
            L.moe_expert_ffn_bwd_weights_workspace_size.restype = ctypes.c_size_t
            L.moe_expert_ffn_bwd_weights_workspace_size.argtypes = [
                _SP, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]
            for fn in ENTRY_POINTS[2:]:
                if not fn.endswith("_workspace_size"):
                    getattr(L, fn).restype = ctypes.c_int
            _lib = L
    return _lib


_F32, _I32 = torch.float32, torch.int32


def _act(s: moe_shape):
    return torch.bfloat16 if s.dtype == MOE_BF16 else torch.float32


def _ptr(t, want=None):
    """Device address of a tensor (None -> NULL; ints pass through).  Tensors
    must be CUDA, contiguous, and of the element type the C ABI expects for
    that argument: the library reads raw pointers and cannot check this."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise MoEError("argument", MOE_ERR_INVALID, "tensor is not on a CUDA device")
    if not t.is_contiguous():
        raise MoEError("argument", MOE_ERR_INVALID, "tensor is not contiguous")
    if want is not None and t.dtype != want:
        raise MoEError("argument", MOE_ERR_INVALID, f"tensor dtype {t.dtype}, expected {want}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, code: int):
    if code != MOE_OK:
        raise MoEError(fn, code, moe_status_string(code))


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def moe_workspace_size(s: moe_shape) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(s)))


def moe_route(s, x, Wg, logit_bias, logits, compute_logits, idx, w, counts, offsets, pos, perm,
              ws, dev_status, stream=None):
    _check("moe_route", lib().moe_route(
        ctypes.byref(s), _ptr(x, _act(s)), _ptr(Wg, _act(s)), _ptr(logit_bias, _F32),
        _ptr(logits, _F32), int(compute_logits), _ptr(idx, _I32), _ptr(w, _F32),
        _ptr(counts, _I32), _ptr(offsets, _I32), _ptr(pos, _I32), _ptr(perm, _I32), _ptr(ws),
        _ptr(dev_status, _I32), _stream(stream)))


def moe_permute(s, x, pos, x_perm, stream=None):
    _check("moe_permute", lib().moe_permute(ctypes.byref(s), _ptr(x, _act(s)), _ptr(pos, _I32),
                                            _ptr(x_perm, _act(s)), _stream(stream)))


def moe_expert_ffn_fwd(s, x_perm, offsets, W1, b1, W2, b2, G, A, y_perm, ws, dev_status,
                       stream=None):
    _check("moe_expert_ffn_fwd", lib().moe_expert_ffn_fwd(
        ctypes.byref(s), _ptr(x_perm, _act(s)), _ptr(offsets, _I32), _ptr(W1, _act(s)),
        _ptr(b1, _act(s)), _ptr(W2, _act(s)), _ptr(b2, _act(s)), _ptr(G, _act(s)),
        _ptr(A, _act(s)), _ptr(y_perm, _act(s)), _ptr(ws), _ptr(dev_status, _I32),
        _stream(stream)))


def moe_expert_ffn_fwd_gather(s, x, perm, offsets, W1, b1, W2, b2, G, A, y_perm, ws,
                              dev_status, stream=None):
    """moe_expert_ffn_fwd with the permute fused in: x [T,d] and the dispatch's
    perm [T*k] instead of X_perm."""
    _check("moe_expert_ffn_fwd_gather", lib().moe_expert_ffn_fwd_gather(
        ctypes.byref(s), _ptr(x, _act(s)), _ptr(perm, _I32), _ptr(offsets, _I32),
        _ptr(W1, _act(s)), _ptr(b1, _act(s)), _ptr(W2, _act(s)), _ptr(b2, _act(s)),
        _ptr(G, _act(s)), _ptr(A, _act(s)), _ptr(y_perm, _act(s)), _ptr(ws),
        _ptr(dev_status, _I32), _stream(stream)))


def moe_combine_fwd(s, y_perm, pos, w, y, stream=None):
    _check("moe_combine_fwd", lib().moe_combine_fwd(
        ctypes.byref(s), _ptr(y_perm, _act(s)), _ptr(pos, _I32), _ptr(w, _F32), _ptr(y, _act(s)),
        _stream(stream)))


def moe_combine_bwd(s, dy, y_perm, pos, w, dy_perm, dw, stream=None):
    _check("moe_combine_bwd", lib().moe_combine_bwd(
        ctypes.byref(s), _ptr(dy, _act(s)), _ptr(y_perm, _act(s)), _ptr(pos, _I32), _ptr(w, _F32),
        _ptr(dy_perm, _act(s)), _ptr(dw, _F32), _stream(stream)))


def moe_expert_ffn_bwd(s, dy_perm, x_perm, G, A, offsets, W1, W2, dx_perm, dW1, db1, dW2, db2,
                       accumulate, ws, dev_status, stream=None):
    _check("moe_expert_ffn_bwd", lib().moe_expert_ffn_bwd(
        ctypes.byref(s), _ptr(dy_perm, _act(s)), _ptr(x_perm, _act(s)), _ptr(G, _act(s)),
        _ptr(A, _act(s)), _ptr(offsets, _I32), _ptr(W1, _act(s)), _ptr(W2, _act(s)),
        _ptr(dx_perm, _act(s)), _ptr(dW1, _F32), _ptr(db1, _F32), _ptr(dW2, _F32),
        _ptr(db2, _F32), int(accumulate), _ptr(ws), _ptr(dev_status, _I32), _stream(stream)))


def moe_expert_ffn_bwd_data(s, dy_perm, G, offsets, W1, W2, dH, dx_perm, db1, accumulate, ws,
                            dev_status, stream=None):
    _check("moe_expert_ffn_bwd_data", lib().moe_expert_ffn_bwd_data(
        ctypes.byref(s), _ptr(dy_perm, _act(s)), _ptr(G, _act(s)), _ptr(offsets, _I32),
        _ptr(W1, _act(s)), _ptr(W2, _act(s)), _ptr(dH, _act(s)), _ptr(dx_perm, _act(s)),
        _ptr(db1, _F32), int(accumulate), _ptr(ws), _ptr(dev_status, _I32), _stream(stream)))


def moe_expert_ffn_bwd_weights_workspace_size(s, chunk_T) -> int:
    n = len(chunk_T)
    arr = (ctypes.c_int64 * n)(*[int(t) for t in chunk_T])
    return int(lib().moe_expert_ffn_bwd_weights_workspace_size(ctypes.byref(s), n, arr))


def moe_expert_ffn_bwd_weights(s, chunk_T, offsets, dy_perm, x_perm, dH, A, dW1, dW2, db2,
                               accumulate, ws, dev_status, stream=None):
    """chunk_T: tokens of each dispatch chunk (a host sequence of ints);
    offsets: int32 device tensor [nchunks, >= E+1] whose rows are the chunks'
    expert offsets; it may be a column slice of a wider array (row stride a
    multiple of 4 elements, columns contiguous), for a range of experts.  ws: a
    uint8 device tensor (its size is passed) or None."""
    n = len(chunk_T)
    arr = (ctypes.c_int64 * n)(*[int(t) for t in chunk_T])
    fn = "moe_expert_ffn_bwd_weights"
    stride = _offsets_stride(fn, offsets, n)
    _check(fn, lib().moe_expert_ffn_bwd_weights(
        ctypes.byref(s), n, arr, offsets.data_ptr(), stride, _ptr(dy_perm, _act(s)),
        _ptr(x_perm, _act(s)), _ptr(dH, _act(s)), _ptr(A, _act(s)), _ptr(dW1, _F32),
        _ptr(dW2, _F32), _ptr(db2, _F32), int(accumulate), _ptr(ws),
        0 if ws is None else int(ws.numel() * ws.element_size()), _ptr(dev_status, _I32),
        _stream(stream)))


def _offsets_stride(fn, offsets, n):
    if not isinstance(offsets, torch.Tensor) or offsets.dim() != 2 or offsets.shape[0] != n:
        raise MoEError(fn, MOE_ERR_INVALID, "offsets must be a [nchunks, stride] tensor")
    if not offsets.is_cuda or offsets.dtype != _I32 or offsets.stride(1) != 1:
        raise MoEError(fn, MOE_ERR_INVALID, "offsets must be int32 CUDA rows")
    return int(offsets.stride(0)) if n > 1 else max(int(offsets.shape[1]) + 3 & ~3, 4)


def moe_expert_ffn_bwd_weights_gather(s, chunk_T, offsets, dy_perm, x, perm, perm_stride, dH,
                                      A, dW1, dW2, db2, accumulate, ws, dev_status,
                                      stream=None):
    """moe_expert_ffn_bwd_weights reading X through each chunk's perm: x holds
    the chunks' tokens one chunk after the other; chunk c's perm starts at
    element c * perm_stride of ``perm``."""
    n = len(chunk_T)
    arr = (ctypes.c_int64 * n)(*[int(t) for t in chunk_T])
    fn = "moe_expert_ffn_bwd_weights_gather"
    stride = _offsets_stride(fn, offsets, n)
    _check(fn, lib().moe_expert_ffn_bwd_weights_gather(
        ctypes.byref(s), n, arr, offsets.data_ptr(), stride, _ptr(dy_perm, _act(s)),
        _ptr(x, _act(s)), _ptr(perm, _I32), ctypes.c_int64(int(perm_stride)), _ptr(dH, _act(s)),
        _ptr(A, _act(s)), _ptr(dW1, _F32), _ptr(dW2, _F32), _ptr(db2, _F32), int(accumulate),
        _ptr(ws), 0 if ws is None else int(ws.numel() * ws.element_size()),
        _ptr(dev_status, _I32), _stream(stream)))


def moe_route_bwd(s, dw, logits, idx, w, perm, offsets, x, Wg, dx_perm, pos, dx, dWg,
                  accumulate, ws, dev_status, stream=None):
    _check("moe_route_bwd", lib().moe_route_bwd(
        ctypes.byref(s), _ptr(dw, _F32), _ptr(logits, _F32), _ptr(idx, _I32), _ptr(w, _F32),
        _ptr(perm, _I32), _ptr(offsets, _I32), _ptr(x, _act(s)), _ptr(Wg, _act(s)),
        _ptr(dx_perm, _act(s)), _ptr(pos, _I32), _ptr(dx, _act(s)), _ptr(dWg, _F32),
        int(accumulate), _ptr(ws), _ptr(dev_status, _I32), _stream(stream)))


def moe_set_gemm_max_units(units: int):
    """Cap the CTA pairs of the tensor-core GEMMs this host thread launches
    (0 = no cap); see include/moe.h."""
    _check("moe_set_gemm_max_units", lib().moe_set_gemm_max_units(int(units)))


def moe_debug_bounded_wait(limit_ns: int, dev_status, stream=None):
    _check("moe_debug_bounded_wait", lib().moe_debug_bounded_wait(
        int(limit_ns), _ptr(dev_status, _I32), _stream(stream)))


def moe_debug_gelu(x, gelu, gelu_grad, fast: int, stream=None):
    _check("moe_debug_gelu", lib().moe_debug_gelu(
        int(x.numel()), _ptr(x, _F32), _ptr(gelu, _F32), _ptr(gelu_grad, _F32), int(fast),
        _stream(stream)))


ROUTE_NOALLOC_MAX_SCRATCH = 1 << 18  # MOE_ROUTE_NOALLOC_MAX_SCRATCH in include/moe.h


def moe_route_noalloc(s, x, Wg, logit_bias, logits, compute_logits, idx, w, counts, offsets,
                      pos, perm, dev_status, stream=None):
    """moe_route without a workspace argument: for callers that cannot
    allocate device memory (see include/moe.h)."""
    _check("moe_route_noalloc", lib().moe_route_noalloc(
        ctypes.byref(s), _ptr(x, _act(s)), _ptr(Wg, _act(s)), _ptr(logit_bias, _F32),
        _ptr(logits, _F32), int(compute_logits), _ptr(idx, _I32), _ptr(w, _F32),
        _ptr(counts, _I32), _ptr(offsets, _I32), _ptr(pos, _I32), _ptr(perm, _I32),
        _ptr(dev_status, _I32), _stream(stream)))
