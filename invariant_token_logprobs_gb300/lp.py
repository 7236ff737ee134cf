"""ctypes binding of liblp (the C ABI in include/lp.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of liblp.  PyTorch is used for device memory and the current stream.
There is no fallback: if the library cannot be loaded, or the current device is
not a GB300 (compute capability 10.3), calls raise :class:`LpError`.

The ``lp_*`` functions mirror the C entry points one to one and take tensors
instead of raw pointers; the short names below them (``logprob_from_logits``,
``linear_logprob``, ...) allocate the outputs and workspace with torch.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

from . import _build_lib

__all__ = [
    "LpError",
    "STATUS",
    "STATE_FLOATS",
    "load",
    "declared_symbols",
    "lp_logprob_from_logits",
    "lp_logprob_partials_from_logits",
    "lp_merge_partials",
    "lp_vocab_shard_range",
    "lp_linear_logprob_workspace_size",
    "lp_linear_logprob",
    "lp_linear_logprob_noalloc",
    "lp_linear_logprob_partials_workspace_size",
    "lp_linear_logprob_partials",
    "lp_logprob_from_logits_temperature",
    "lp_logprob_from_logits_lse",
    "lp_logprob_from_logits_backward",
    "lp_merge_partials_lse",
    "lp_logprob_partials_from_logits_backward",
    "logprob_from_logits_lse",
    "logprob_from_logits_backward",
    "lp_logprob_partials_from_logits_temperature",
    "lp_linear_logprob_temperature",
    "lp_linear_logprob_partials_temperature",
    "lp_linear_logprob_backward_workspace_size",
    "lp_linear_logprob_lse",
    "lp_linear_logprob_backward",
    "lp_linear_logprob_backward_ex",
    "lp_linear_logprob_partials_backward_workspace_size",
    "lp_linear_logprob_partials_backward",
    "lp_merge_grad_h_partials",
    "linear_logprob_partials_backward",
    "merge_grad_h_partials",
    "GRAD_W_FLOAT32",
    "GRAD_W_BFLOAT16",
    "GRAD_W_FLOAT32_ACCUMULATE",
    "linear_logprob_lse",
    "linear_logprob_backward",
    "lp_get_device_error",
    "lp_set_persistent_grid_limit",
    "lp_set_kernel_timing_events",
    "lp_set_fault_injection",
    "lp_get_check_word",
    "lp_status_string",
    "lp_backend_id",
    "logprob_from_logits",
    "logprob_partials_from_logits",
    "merge_partials",
    "linear_logprob",
    "linear_logprob_partials",
    "vocab_shard_range",
]

# floats per quarter state in the partials layout [T][quarters][STATE_FLOATS]
STATE_FLOATS = 8

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lp.h")

STATUS = {
    0: "LP_OK",
    1: "LP_ERR_INVALID_ARGUMENT",
    2: "LP_ERR_MISALIGNED",
    3: "LP_ERR_UNSUPPORTED_DEVICE",
    4: "LP_ERR_WORKSPACE_TOO_SMALL",
    5: "LP_ERR_CUDA",
    6: "LP_ERR_TIMEOUT",
}


class LpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


_lib: Optional[ctypes.CDLL] = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t

_SIGNATURES = {
    "lp_logprob_from_logits": (_int, [_vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp]),
    "lp_vocab_shard_range": (_int, [_i64, _int, _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "lp_logprob_partials_from_logits": (_int, [_vp, _i64, _vp, _i64, _i64, _int, _int, _vp, _vp]),
    "lp_merge_partials": (_int, [ctypes.POINTER(_vp), _int, _i64, _vp, _vp, _vp]),
    "lp_linear_logprob_workspace_size": (_sz, [_i64, _i64, _i64]),
    "lp_linear_logprob": (_int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _sz, _vp]),
    "lp_linear_logprob_noalloc": (_int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "lp_linear_logprob_partials_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "lp_linear_logprob_partials": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _int, _int, _vp, _vp, _sz, _vp]),
    "lp_logprob_from_logits_temperature": (
        _int, [_vp, _i64, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp]),
    "lp_logprob_from_logits_lse": (
        _int, [_vp, _i64, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp]),
    "lp_logprob_from_logits_backward": (
        _int, [_vp, _i64, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "lp_merge_partials_lse": (_int, [ctypes.POINTER(_vp), _int, _i64, _vp, _vp, _vp, _vp]),
    "lp_logprob_partials_from_logits_backward": (
        _int, [_vp, _i64, _vp, _i64, _i64, _int, _int, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
               _i64, _vp]),
    "lp_logprob_partials_from_logits_temperature": (
        _int, [_vp, _i64, _vp, _i64, _i64, _int, _int, ctypes.c_float, _vp, _vp]),
    "lp_linear_logprob_temperature": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _sz, _vp]),
    "lp_linear_logprob_partials_temperature": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _int, _int, ctypes.c_float, _vp, _vp,
               _sz, _vp]),
    "lp_linear_logprob_backward_workspace_size": (_sz, [_i64, _i64, _i64]),
    "lp_linear_logprob_lse": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp,
               _sz, _vp]),
    "lp_linear_logprob_backward": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp,
               _vp, _vp, _vp, _sz, _vp]),
    "lp_linear_logprob_backward_ex": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp,
               _vp, _vp, _int, _vp, _sz, _vp]),
    "lp_linear_logprob_partials_backward_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "lp_linear_logprob_partials_backward": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _int, _int, ctypes.c_float, _vp, _vp,
               _vp, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "lp_merge_grad_h_partials": (_int, [ctypes.POINTER(_vp), _int, _i64, _i64, _vp, _vp]),
    "lp_get_device_error": (_int, [_vp, _sz, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "lp_set_persistent_grid_limit": (_int, [_int]),
    "lp_set_kernel_timing_events": (_int, [_vp, _vp]),
    "lp_set_fault_injection": (_int, [_int]),
    "lp_get_check_word": (_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "lp_status_string": (ctypes.c_char_p, [_int]),
    "lp_backend_id": (ctypes.c_char_p, []),
}


def declared_symbols() -> list[str]:
    """Names of the entry points include/lp.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^LP_API\s+[\w\s\*]+?\b(lp_\w+)\s*\(", text, flags=re.M)


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load liblp.so (building it first when it is missing or stale).

    The environment variable LP_LIBRARY names another build of the same
    library to load instead (for comparing builds); it is never a fallback.
    """
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("LP_LIBRARY", _build_lib.LIB)
    if build_if_needed and path == _build_lib.LIB and _build_lib._stale():
        _build_lib.build()
    if not os.path.exists(path):
        raise LpError("load", 5)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise LpError(fn, status)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _row_stride(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with contiguous rows")
    return t.stride(0)


# ----------------------------------------------------------------- C entry points

def lp_logprob_from_logits(logits, targets, logp, entropy=None, stream=None) -> None:
    if logits.dtype != torch.float32 or targets.dtype != torch.int64:
        raise TypeError("logits must be float32 and targets int64")
    T, V = logits.shape
    _check("lp_logprob_from_logits", load().lp_logprob_from_logits(
        _ptr(logits), _row_stride(logits), _ptr(targets), T, V, _ptr(logp), _ptr(entropy),
        _stream(stream)))


def lp_vocab_shard_range(vocab_total: int, shard_index: int, n_shards: int) -> tuple[int, int]:
    b, e = _i64(), _i64()
    _check("lp_vocab_shard_range",
           load().lp_vocab_shard_range(vocab_total, shard_index, n_shards, ctypes.byref(b), ctypes.byref(e)))
    return b.value, e.value


def lp_logprob_partials_from_logits(logits_shard, targets, vocab_total, shard_index, n_shards,
                                    partials, stream=None) -> None:
    if logits_shard.dtype != torch.float32 or targets.dtype != torch.int64:
        raise TypeError("logits must be float32 and targets int64")
    T = logits_shard.shape[0]
    _check("lp_logprob_partials_from_logits", load().lp_logprob_partials_from_logits(
        _ptr(logits_shard), _row_stride(logits_shard), _ptr(targets), T, vocab_total,
        shard_index, n_shards, _ptr(partials), _stream(stream)))


def lp_merge_partials(shard_partials: Sequence[torch.Tensor], T: int, logp, entropy=None,
                      stream=None) -> None:
    arr = (_vp * len(shard_partials))(*[p.data_ptr() for p in shard_partials])
    _check("lp_merge_partials", load().lp_merge_partials(
        arr, len(shard_partials), T, _ptr(logp), _ptr(entropy), _stream(stream)))


def lp_merge_partials_lse(shard_partials: Sequence[torch.Tensor], T: int, logp, entropy, lse,
                          stream=None) -> None:
    arr = (_vp * len(shard_partials))(*[p.data_ptr() for p in shard_partials])
    _check("lp_merge_partials_lse", load().lp_merge_partials_lse(
        arr, len(shard_partials), T, _ptr(logp), _ptr(entropy), _ptr(lse), _stream(stream)))


def lp_logprob_partials_from_logits_backward(logits_shard, targets, vocab_total, shard_index,
                                             n_shards, temperature, saved_lse, saved_entropy,
                                             grad_logp, grad_entropy, grad_shard,
                                             stream=None) -> None:
    if logits_shard.dtype != torch.float32 or grad_shard.dtype != torch.float32 \
            or targets.dtype != torch.int64:
        raise TypeError("logits and gradient must be float32 and targets int64")
    if tuple(grad_shard.shape) != tuple(logits_shard.shape):
        raise ValueError("grad_shard must have the shard's shape")
    T = logits_shard.shape[0]
    _check("lp_logprob_partials_from_logits_backward",
           load().lp_logprob_partials_from_logits_backward(
               _ptr(logits_shard), _row_stride(logits_shard), _ptr(targets), T, vocab_total,
               shard_index, n_shards, float(temperature), _ptr(saved_lse), _ptr(saved_entropy),
               _ptr(grad_logp), _ptr(grad_entropy), _ptr(grad_shard), _row_stride(grad_shard),
               _stream(stream)))


def lp_linear_logprob_workspace_size(T: int, d: int, V: int) -> int:
    return int(load().lp_linear_logprob_workspace_size(T, d, V))


def lp_linear_logprob_partials_workspace_size(T: int, d: int, vocab_total: int, n_shards: int) -> int:
    return int(load().lp_linear_logprob_partials_workspace_size(T, d, vocab_total, n_shards))


def _check_bf16(H, W, targets):
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or targets.dtype != torch.int64:
        raise TypeError("H and W must be bfloat16 and targets int64")


def lp_linear_logprob(H, W, targets, logp, entropy, workspace, stream=None) -> None:
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    _check("lp_linear_logprob", load().lp_linear_logprob(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        _ptr(logp), _ptr(entropy), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def lp_linear_logprob_noalloc(H, W, targets, logp, entropy=None, stream=None) -> None:
    """lp_linear_logprob with the library's fixed device scratch instead of a
    workspace: for callers that cannot allocate device memory (see lp.h)."""
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    _check("lp_linear_logprob_noalloc", load().lp_linear_logprob_noalloc(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        _ptr(logp), _ptr(entropy), _stream(stream)))


def lp_linear_logprob_partials(H, W_shard, targets, vocab_total, shard_index, n_shards,
                               partials, workspace, stream=None) -> None:
    _check_bf16(H, W_shard, targets)
    T, d = H.shape
    _check("lp_linear_logprob_partials", load().lp_linear_logprob_partials(
        _ptr(H), _row_stride(H), _ptr(W_shard), _row_stride(W_shard), _ptr(targets), T, d,
        vocab_total, shard_index, n_shards, _ptr(partials), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lp_logprob_from_logits_temperature(logits, targets, temperature, logp, entropy=None,
                                       stream=None) -> None:
    if logits.dtype != torch.float32 or targets.dtype != torch.int64:
        raise TypeError("logits must be float32 and targets int64")
    T, V = logits.shape
    _check("lp_logprob_from_logits_temperature", load().lp_logprob_from_logits_temperature(
        _ptr(logits), _row_stride(logits), _ptr(targets), T, V, float(temperature), _ptr(logp),
        _ptr(entropy), _stream(stream)))


def lp_logprob_from_logits_lse(logits, targets, temperature, logp, entropy, lse,
                               stream=None) -> None:
    if logits.dtype != torch.float32 or targets.dtype != torch.int64:
        raise TypeError("logits must be float32 and targets int64")
    T, V = logits.shape
    _check("lp_logprob_from_logits_lse", load().lp_logprob_from_logits_lse(
        _ptr(logits), _row_stride(logits), _ptr(targets), T, V, float(temperature), _ptr(logp),
        _ptr(entropy), _ptr(lse), _stream(stream)))


def lp_logprob_from_logits_backward(logits, targets, temperature, saved_lse, saved_entropy,
                                    grad_logp, grad_entropy, grad_logits, stream=None) -> None:
    if logits.dtype != torch.float32 or grad_logits.dtype != torch.float32 \
            or targets.dtype != torch.int64:
        raise TypeError("logits and grad_logits must be float32 and targets int64")
    T, V = logits.shape
    if tuple(grad_logits.shape) != (T, V):
        raise ValueError("grad_logits must have the logits' shape")
    _check("lp_logprob_from_logits_backward", load().lp_logprob_from_logits_backward(
        _ptr(logits), _row_stride(logits), _ptr(targets), T, V, float(temperature),
        _ptr(saved_lse), _ptr(saved_entropy), _ptr(grad_logp), _ptr(grad_entropy),
        _ptr(grad_logits), _row_stride(grad_logits), _stream(stream)))


def lp_logprob_partials_from_logits_temperature(logits_shard, targets, vocab_total, shard_index,
                                                n_shards, temperature, partials,
                                                stream=None) -> None:
    if logits_shard.dtype != torch.float32 or targets.dtype != torch.int64:
        raise TypeError("logits must be float32 and targets int64")
    T = logits_shard.shape[0]
    _check("lp_logprob_partials_from_logits_temperature",
           load().lp_logprob_partials_from_logits_temperature(
               _ptr(logits_shard), _row_stride(logits_shard), _ptr(targets), T, vocab_total,
               shard_index, n_shards, float(temperature), _ptr(partials), _stream(stream)))


def lp_linear_logprob_temperature(H, W, targets, temperature, logp, entropy, workspace,
                                  stream=None) -> None:
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    _check("lp_linear_logprob_temperature", load().lp_linear_logprob_temperature(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        float(temperature), _ptr(logp), _ptr(entropy), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lp_linear_logprob_partials_temperature(H, W_shard, targets, vocab_total, shard_index, n_shards,
                                           temperature, partials, workspace, stream=None) -> None:
    _check_bf16(H, W_shard, targets)
    T, d = H.shape
    _check("lp_linear_logprob_partials_temperature", load().lp_linear_logprob_partials_temperature(
        _ptr(H), _row_stride(H), _ptr(W_shard), _row_stride(W_shard), _ptr(targets), T, d,
        vocab_total, shard_index, n_shards, float(temperature), _ptr(partials), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lp_linear_logprob_backward_workspace_size(T: int, d: int, V: int) -> int:
    return int(load().lp_linear_logprob_backward_workspace_size(T, d, V))


def lp_linear_logprob_lse(H, W, targets, temperature, logp, entropy, lse, workspace,
                          stream=None) -> None:
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    _check("lp_linear_logprob_lse", load().lp_linear_logprob_lse(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        float(temperature), _ptr(logp), _ptr(entropy), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lp_linear_logprob_backward(H, W, targets, temperature, saved_lse, saved_entropy, grad_logp,
                               grad_entropy, grad_H, grad_W, workspace, stream=None) -> None:
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    _check("lp_linear_logprob_backward", load().lp_linear_logprob_backward(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        float(temperature), _ptr(saved_lse), _ptr(saved_entropy), _ptr(grad_logp),
        _ptr(grad_entropy), _ptr(grad_H), _ptr(grad_W), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


GRAD_W_FLOAT32 = 0
GRAD_W_BFLOAT16 = 1
GRAD_W_FLOAT32_ACCUMULATE = 2


def _grad_w_dtype_code(grad_W, accumulate: bool = False) -> int:
    if accumulate:
        if grad_W is None or grad_W.dtype != torch.float32:
            raise TypeError("accumulating needs a float32 grad_W")
        return GRAD_W_FLOAT32_ACCUMULATE
    if grad_W is None or grad_W.dtype == torch.float32:
        return GRAD_W_FLOAT32
    if grad_W.dtype == torch.bfloat16:
        return GRAD_W_BFLOAT16
    raise TypeError("grad_W must be float32 or bfloat16")


def lp_linear_logprob_backward_ex(H, W, targets, temperature, saved_lse, saved_entropy,
                                  grad_logp, grad_entropy, grad_H, grad_W, workspace,
                                  stream=None, accumulate: bool = False) -> None:
    """The backward with grad_W float32 or bfloat16 (taken from grad_W's dtype);
    accumulate=True adds the product into the float32 grad_W instead."""
    _check_bf16(H, W, targets)
    T, d = H.shape
    V = W.shape[0]
    dtype = _grad_w_dtype_code(grad_W, accumulate)
    _check("lp_linear_logprob_backward_ex", load().lp_linear_logprob_backward_ex(
        _ptr(H), _row_stride(H), _ptr(W), _row_stride(W), _ptr(targets), T, d, V,
        float(temperature), _ptr(saved_lse), _ptr(saved_entropy), _ptr(grad_logp),
        _ptr(grad_entropy), _ptr(grad_H), _ptr(grad_W), dtype, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))




def lp_linear_logprob_partials_backward_workspace_size(T: int, d: int, vocab_total: int,
                                                       n_shards: int) -> int:
    return int(load().lp_linear_logprob_partials_backward_workspace_size(T, d, vocab_total,
                                                                         n_shards))


def lp_linear_logprob_partials_backward(H, W_shard, targets, vocab_total, shard_index, n_shards,
                                        temperature, saved_lse, saved_entropy, grad_logp,
                                        grad_entropy, grad_H_partial, grad_W_shard, workspace,
                                        stream=None, accumulate: bool = False) -> None:
    """The shard's backward (grad_W_shard float32 or bfloat16, from its dtype, or None;
    accumulate=True adds into the float32 grad_W_shard)."""
    _check_bf16(H, W_shard, targets)
    T, d = H.shape
    _check("lp_linear_logprob_partials_backward", load().lp_linear_logprob_partials_backward(
        _ptr(H), _row_stride(H), _ptr(W_shard), _row_stride(W_shard), _ptr(targets), T, d,
        vocab_total, shard_index, n_shards, float(temperature), _ptr(saved_lse),
        _ptr(saved_entropy), _ptr(grad_logp), _ptr(grad_entropy), _ptr(grad_H_partial),
        _ptr(grad_W_shard), _grad_w_dtype_code(grad_W_shard, accumulate), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lp_merge_grad_h_partials(shard_grad_h: Sequence[torch.Tensor], grad_H, stream=None) -> None:
    T, d = grad_H.shape
    for p in shard_grad_h:
        if p.dtype != torch.float32 or tuple(p.shape) != (T, d) or not p.is_contiguous():
            raise ValueError("partials must be contiguous float32 [T, d]")
    arr = (_vp * len(shard_grad_h))(*[p.data_ptr() for p in shard_grad_h])
    _check("lp_merge_grad_h_partials", load().lp_merge_grad_h_partials(
        arr, len(shard_grad_h), T, d, _ptr(grad_H), _stream(stream)))


def linear_logprob_partials_backward(H, W_shard, y, vocab_total, shard_index, n_shards,
                                     saved_lse, saved_entropy, grad_logp=None, grad_entropy=None,
                                     temperature: float = 1.0, with_grad_W: bool = True,
                                     grad_W_dtype=torch.float32, workspace=None, stream=None,
                                     accumulate_into=None):
    """(grad_H partial [T, d] fp32, grad_W_shard [rows of W_shard, d] or None) of one
    vocabulary shard, from the merged rows' log Z and entropy; with accumulate_into
    (float32 [rows of W_shard, d]) the shard's grad_W is added into it."""
    T, d = H.shape
    if workspace is None:
        workspace = _workspace(
            lp_linear_logprob_partials_backward_workspace_size(T, d, vocab_total, n_shards),
            H.device)
    gH = torch.empty((T, d), dtype=torch.float32, device=H.device)
    if accumulate_into is not None:
        gW = accumulate_into
    else:
        gW = (torch.empty((W_shard.shape[0], d), dtype=grad_W_dtype, device=H.device)
              if with_grad_W else None)
    lp_linear_logprob_partials_backward(H, W_shard, y, vocab_total, shard_index, n_shards,
                                        temperature, saved_lse, saved_entropy, grad_logp,
                                        grad_entropy, gH, gW, workspace, stream,
                                        accumulate=accumulate_into is not None)
    return gH, gW


def merge_grad_h_partials(shard_grad_h: Sequence[torch.Tensor], stream=None) -> torch.Tensor:
    """grad_H [T, d] fp32 from the shards' partials, in shard order."""
    out = torch.empty_like(shard_grad_h[0])
    lp_merge_grad_h_partials(shard_grad_h, out, stream)
    return out


def linear_logprob_lse(H, W, y, temperature: float = 1.0, workspace=None, stream=None):
    """(logp, entropy, lse) [T] fp32 of the fused path; keep entropy and lse for the backward."""
    T, d = H.shape
    V = W.shape[0]
    if workspace is None:
        workspace = _workspace(lp_linear_logprob_workspace_size(T, d, V), H.device)
    out = [torch.empty(T, dtype=torch.float32, device=H.device) for _ in range(3)]
    lp_linear_logprob_lse(H, W, y, temperature, out[0], out[1], out[2], workspace, stream)
    return tuple(out)


def linear_logprob_backward(H, W, y, grad_logp=None, grad_entropy=None, temperature: float = 1.0,
                            with_grad_W: bool = True, saved_lse=None, saved_entropy=None,
                            workspace=None, stream=None, grad_W_dtype=torch.float32,
                            accumulate_into=None):
    """(grad_H [T, d] fp32, grad_W [V, d] fp32 / bf16 or None) of the fused path;
    with accumulate_into (a float32 [V, d] tensor, e.g. a main gradient) the
    product is added into it and it is returned as grad_W."""
    T, d = H.shape
    V = W.shape[0]
    if workspace is None:
        workspace = _workspace(lp_linear_logprob_backward_workspace_size(T, d, V), H.device)
    gH = torch.empty((T, d), dtype=torch.float32, device=H.device)
    if accumulate_into is not None:
        lp_linear_logprob_backward_ex(H, W, y, temperature, saved_lse, saved_entropy, grad_logp,
                                      grad_entropy, gH, accumulate_into, workspace, stream,
                                      accumulate=True)
        return gH, accumulate_into
    gW = torch.empty((V, d), dtype=grad_W_dtype, device=H.device) if with_grad_W else None
    if grad_W_dtype == torch.float32:
        lp_linear_logprob_backward(H, W, y, temperature, saved_lse, saved_entropy, grad_logp,
                                   grad_entropy, gH, gW, workspace, stream)
    else:
        lp_linear_logprob_backward_ex(H, W, y, temperature, saved_lse, saved_entropy, grad_logp,
                                      grad_entropy, gH, gW, workspace, stream)
    return gH, gW


def lp_get_device_error(workspace, stream=None) -> int:
    """The workspace error word (0: no device-side wait gave up)."""
    word = ctypes.c_uint32(0)
    st = load().lp_get_device_error(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                    ctypes.byref(word), _stream(stream))
    if st not in (0, 6):
        raise LpError("lp_get_device_error", st)
    return int(word.value)


def lp_set_persistent_grid_limit(max_ctas: int) -> None:
    _check("lp_set_persistent_grid_limit", load().lp_set_persistent_grid_limit(max_ctas))


def lp_set_kernel_timing_events(start_event=None, stop_event=None) -> None:
    """Record torch.cuda.Event pairs around the fused path's tensor-core kernel."""
    a = None if start_event is None else start_event.cuda_event
    b = None if stop_event is None else stop_event.cuda_event
    _check("lp_set_kernel_timing_events", load().lp_set_kernel_timing_events(a, b))


def lp_set_fault_injection(mode: int) -> None:
    _check("lp_set_fault_injection", load().lp_set_fault_injection(mode))


def lp_get_check_word() -> int:
    """The OR of the check words of the checked build since the last read (0 in
    the normal build); synchronises the device."""
    word = ctypes.c_uint32(0)
    _check("lp_get_check_word", load().lp_get_check_word(ctypes.byref(word)))
    return int(word.value)


def lp_status_string(status: int) -> str:
    return load().lp_status_string(status).decode()


def lp_backend_id() -> str:
    return load().lp_backend_id().decode()


# ------------------------------------------------------------ allocating helpers

def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def logprob_from_logits(z: torch.Tensor, y: torch.Tensor, with_entropy: bool = True, stream=None,
                        temperature: Optional[float] = None):
    T = z.shape[0]
    logp = torch.empty(T, dtype=torch.float32, device=z.device)
    ent = torch.empty(T, dtype=torch.float32, device=z.device) if with_entropy else None
    if temperature is None:
        lp_logprob_from_logits(z, y, logp, ent, stream)
    else:
        lp_logprob_from_logits_temperature(z, y, temperature, logp, ent, stream)
    return logp, ent


def logprob_from_logits_lse(z: torch.Tensor, y: torch.Tensor, temperature: float = 1.0,
                            stream=None):
    """(logp, entropy, lse) [T] fp32 of the logits path; keep entropy and lse for the backward."""
    T = z.shape[0]
    out = [torch.empty(T, dtype=torch.float32, device=z.device) for _ in range(3)]
    lp_logprob_from_logits_lse(z, y, temperature, out[0], out[1], out[2], stream)
    return tuple(out)


def logprob_from_logits_backward(z: torch.Tensor, y: torch.Tensor, grad_logp=None,
                                 grad_entropy=None, temperature: float = 1.0, saved_lse=None,
                                 saved_entropy=None, stream=None) -> torch.Tensor:
    """dL/dz [T, V] fp32 for L = sum grad_logp * logp + grad_entropy * entropy; log Z and
    the entropy are taken from the forward when given, else computed first."""
    if saved_lse is None or saved_entropy is None:
        _, saved_entropy, saved_lse = logprob_from_logits_lse(z, y, temperature, stream)
    grad = torch.empty(z.shape, dtype=torch.float32, device=z.device)
    lp_logprob_from_logits_backward(z, y, temperature, saved_lse, saved_entropy, grad_logp,
                                    grad_entropy, grad, stream)
    return grad


def vocab_shard_range(vocab_total: int, shard_index: int, n_shards: int) -> tuple[int, int]:
    return lp_vocab_shard_range(vocab_total, shard_index, n_shards)


def logprob_partials_from_logits(z_shard, y, vocab_total, shard_index, n_shards, stream=None,
                                 temperature: Optional[float] = None):
    T = z_shard.shape[0]
    partials = torch.empty((T, 4 // n_shards, STATE_FLOATS), dtype=torch.float32,
                           device=z_shard.device)
    if temperature is None:
        lp_logprob_partials_from_logits(z_shard, y, vocab_total, shard_index, n_shards, partials,
                                        stream)
    else:
        lp_logprob_partials_from_logits_temperature(z_shard, y, vocab_total, shard_index, n_shards,
                                                    temperature, partials, stream)
    return partials


def merge_partials(shard_partials: Sequence[torch.Tensor], with_entropy: bool = True, stream=None):
    T = shard_partials[0].shape[0]
    dev = shard_partials[0].device
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    ent = torch.empty(T, dtype=torch.float32, device=dev) if with_entropy else None
    lp_merge_partials(shard_partials, T, logp, ent, stream)
    return logp, ent


def linear_logprob(H, W, y, with_entropy: bool = True, workspace=None, stream=None,
                   temperature: Optional[float] = None):
    T, d = H.shape
    V = W.shape[0]
    if workspace is None:
        workspace = _workspace(lp_linear_logprob_workspace_size(T, d, V), H.device)
    logp = torch.empty(T, dtype=torch.float32, device=H.device)
    ent = torch.empty(T, dtype=torch.float32, device=H.device) if with_entropy else None
    if temperature is None:
        lp_linear_logprob(H, W, y, logp, ent, workspace, stream)
    else:
        lp_linear_logprob_temperature(H, W, y, temperature, logp, ent, workspace, stream)
    return logp, ent


def linear_logprob_partials(H, W_shard, y, vocab_total, shard_index, n_shards, workspace=None,
                            stream=None, temperature: Optional[float] = None):
    T, d = H.shape
    if workspace is None:
        workspace = _workspace(
            lp_linear_logprob_partials_workspace_size(T, d, vocab_total, n_shards), H.device)
    partials = torch.empty((T, 4 // n_shards, STATE_FLOATS), dtype=torch.float32, device=H.device)
    if temperature is None:
        lp_linear_logprob_partials(H, W_shard, y, vocab_total, shard_index, n_shards, partials,
                                   workspace, stream)
    else:
        lp_linear_logprob_partials_temperature(H, W_shard, y, vocab_total, shard_index, n_shards,
                                               temperature, partials, workspace, stream)
    return partials
