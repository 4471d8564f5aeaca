"""PyTorch-facing wrappers of the logits-input fused log-prob (include/fused_logp.h).

Argument marshalling only; the computation runs in ``liblinear_logp.so``.
logits [N, V] (or [..., V]) bf16, fp16 or fp32, contiguous, on a CUDA device;
targets int64 with the logits' leading shape.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from .ops import on_tensor_device

IGNORE_INDEX = -100
_DTYPES = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(logits: torch.Tensor, targets: torch.Tensor):
    if not isinstance(logits, torch.Tensor) or logits.device.type != "cuda":
        raise ValueError("logits must be a CUDA tensor; this op has no CPU path")
    if logits.dtype not in _DTYPES:
        raise TypeError(f"logits must be bf16, fp16 or fp32, got {logits.dtype}")
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [N, V] tensor")
    if targets.dtype != torch.int64 or targets.device != logits.device or targets.shape != (logits.shape[0],):
        raise ValueError("targets must be int64 [N] on the logits' device")
    if not targets.is_contiguous():
        raise ValueError("targets must be contiguous")


@on_tensor_device
def fused_logp_fwd(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = IGNORE_INDEX,
                   workspace: Optional[torch.Tensor] = None):
    """(logp, row_max, log_sum), each fp32 [N]; lse = row_max + log_sum."""
    _check(logits, targets)
    N, V = logits.shape
    lib = _lib.load()
    dev = logits.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    row_max = torch.empty(N, dtype=torch.float32, device=dev)
    log_sum = torch.empty(N, dtype=torch.float32, device=dev)
    nbytes = int(lib.fused_logp_workspace_bytes(N, V))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    st = lib.fused_logp_fwd(_ptr(logits), _DTYPES[logits.dtype], N, V, _ptr(targets), int(ignore_index),
                            _ptr(logp), _ptr(row_max), _ptr(log_sum), _ptr(workspace), workspace.numel(),
                            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    _lib.check("fused_logp_fwd", st)
    return logp, row_max, log_sum


@on_tensor_device
def fused_logp_bwd(grad_logp: torch.Tensor, row_max: torch.Tensor, log_sum: torch.Tensor, logits: torch.Tensor,
                   targets: torch.Tensor, ignore_index: int = IGNORE_INDEX,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad_logits [N, V] in the logits' dtype."""
    _check(logits, targets)
    N, V = logits.shape
    for name, t in (("grad_logp", grad_logp), ("row_max", row_max), ("log_sum", log_sum)):
        if t.dtype != torch.float32 or t.shape != (N,) or t.device != logits.device or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 [N] tensor on the logits' device")
    grad = torch.empty_like(logits) if out is None else out
    lib = _lib.load()
    st = lib.fused_logp_bwd(_ptr(grad_logp), _ptr(row_max), _ptr(log_sum), _ptr(logits), _DTYPES[logits.dtype], N, V,
                            _ptr(targets), int(ignore_index), _ptr(grad),
                            ctypes.c_void_p(torch.cuda.current_stream(logits.device).cuda_stream))
    _lib.check("fused_logp_bwd", st)
    return grad


def _indices(indices: torch.Tensor, device) -> torch.Tensor:
    if not isinstance(indices, torch.Tensor) or indices.dtype != torch.int64 or indices.device != device:
        raise TypeError("indices must be an int64 tensor on the logits' device")
    return indices.reshape(-1).contiguous()


@on_tensor_device
def fused_logp_fwd_indexed(logits: torch.Tensor, targets: torch.Tensor, indices: torch.Tensor,
                           ignore_index: int = IGNORE_INDEX,
                           out: Optional[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]] = None):
    """Forward on the rows named by ``indices`` (duplicates count once, out of range
    ignored).  Selected entries of (logp, row_max, log_sum) get the dense forward's
    values; the others keep their contents (new buffers start as 0 / -inf / 0)."""
    _check(logits, targets)
    N, V = logits.shape
    dev = logits.device
    idx = _indices(indices, dev)
    if out is None:
        logp = torch.zeros(N, dtype=torch.float32, device=dev)
        row_max = torch.full((N,), float("-inf"), dtype=torch.float32, device=dev)
        log_sum = torch.zeros(N, dtype=torch.float32, device=dev)
    else:
        logp, row_max, log_sum = out
    lib = _lib.load()
    K = idx.numel()
    ws = torch.empty(max(int(lib.fused_logp_fwd_indexed_workspace_bytes(N, V, K)), 1), dtype=torch.uint8, device=dev)
    st = lib.fused_logp_fwd_indexed(_ptr(logits), _DTYPES[logits.dtype], N, V, _ptr(targets), int(ignore_index),
                                    _ptr(idx), K, _ptr(logp), _ptr(row_max), _ptr(log_sum), _ptr(ws), ws.numel(),
                                    ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    _lib.check("fused_logp_fwd_indexed", st)
    return logp, row_max, log_sum


@on_tensor_device
def fused_logp_bwd_indexed(grad_logp: torch.Tensor, row_max: torch.Tensor, log_sum: torch.Tensor,
                           logits: torch.Tensor, targets: torch.Tensor, indices: torch.Tensor,
                           ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """grad_logits [N, V] of sum over the selected rows of grad_logp * logp: rows
    not selected are zero."""
    _check(logits, targets)
    N, V = logits.shape
    dev = logits.device
    idx = _indices(indices, dev)
    for name, t in (("grad_logp", grad_logp), ("row_max", row_max), ("log_sum", log_sum)):
        if t.dtype != torch.float32 or t.shape != (N,) or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 [N] tensor on the logits' device")
    grad = torch.empty_like(logits)
    lib = _lib.load()
    K = idx.numel()
    ws = torch.empty(max(int(lib.fused_logp_bwd_indexed_workspace_bytes(N, K)), 1), dtype=torch.uint8, device=dev)
    st = lib.fused_logp_bwd_indexed(_ptr(grad_logp), _ptr(row_max), _ptr(log_sum), _ptr(logits),
                                    _DTYPES[logits.dtype], N, V, _ptr(targets), int(ignore_index), _ptr(idx), K,
                                    _ptr(grad), _ptr(ws), ws.numel(),
                                    ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    _lib.check("fused_logp_bwd_indexed", st)
    return grad


class _FusedLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, targets, ignore_index):
        logp, row_max, log_sum = fused_logp_fwd(logits, targets, ignore_index)
        ctx.save_for_backward(logits, targets, row_max, log_sum)
        ctx.ignore_index = ignore_index
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        logits, targets, row_max, log_sum = ctx.saved_tensors
        g = fused_logp_bwd(grad_logp.contiguous().float(), row_max, log_sum, logits, targets, ctx.ignore_index)
        return g, None, None


def fused_logp(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """log_softmax(logits)[targets] in fp32 with autograd; logits [..., V], targets [...]."""
    V = logits.shape[-1]
    out = _FusedLogp.apply(logits.reshape(-1, V).contiguous(), targets.reshape(-1).contiguous(), int(ignore_index))
    return out.reshape(targets.shape)
