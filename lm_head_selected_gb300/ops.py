"""PyTorch-facing wrappers over the C ABI (include/linear_logp.h).

PyTorch supplies device memory and the current stream; every step of the
computation runs in the CUDA kernels of ``liblinear_logp.so``.  Inputs are
checked here and rejected (no fallback, no casting): hidden/weight bf16 (or
both fp16 for the plain and row-subset forward / backward and ``linear_logp``),
bias/temperature/grad fp32, targets int64, all contiguous on one CUDA device.

Entry points mirror the C ABI names:
  * ``linear_logp_fwd``  -> (logp [N] fp32, lse [N] fp32)
  * ``linear_logp_bwd``  -> (grad_hidden | None, grad_weight | None, grad_bias fp32 | None), the
    16-bit gradients in the inputs' dtype
  * ``linear_logp``      -> autograd-aware op with leading shapes, the interface
    of "Fused Linear LogP" (Entry Point): hidden [B,S,D] or [N,D], targets [B,S]
    or [N], optional bias; gradients flow into hidden, weight and bias.
"""
from __future__ import annotations

import ctypes
import functools
import itertools
from typing import Optional, Tuple

import torch

from . import _lib

IGNORE_INDEX = -100


def on_tensor_device(fn):
    """Run a wrapper with its first CUDA tensor argument's device current: the C
    ABI launches on the current device, which need not be the tensors' one."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        for a in itertools.chain(args, kwargs.values()):
            if isinstance(a, torch.Tensor) and a.is_cuda:
                with torch.cuda.device(a.device):
                    return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return wrapper


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_inputs(hidden, weight, targets, bias, temperature, allow_f16=False):
    if not isinstance(hidden, torch.Tensor) or hidden.device.type != "cuda":
        raise ValueError("hidden must be a CUDA tensor; this op has no CPU path")
    dev = hidden.device
    dt = torch.float16 if (allow_f16 and hidden.dtype == torch.float16) else torch.bfloat16
    _need(hidden, "hidden", dt, dev, 2)
    _need(weight, "weight", dt, dev, 2)
    N, D = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != D:
        raise ValueError(f"weight must be [V, {D}], got {tuple(weight.shape)}")
    _need(targets, "targets", torch.int64, dev, 1)
    if targets.shape[0] != N:
        raise ValueError("targets must have N entries")
    if bias is not None:
        _need(bias, "bias", torch.float32, dev, 1)
        if bias.shape[0] != V:
            raise ValueError("bias must have V entries")
    if temperature is not None:
        _need(temperature, "temperature", torch.float32, dev, 1)
        if temperature.shape[0] != N:
            raise ValueError("temperature must have N entries")
    return dev, N, D, V


def fwd_workspace_bytes(N: int, D: int, V: int) -> int:
    return int(_lib.load().linear_logp_fwd_workspace_bytes(N, D, V))


def bwd_workspace_bytes(N: int, D: int, V: int, has_bias: bool) -> int:
    return int(_lib.load().linear_logp_bwd_workspace_bytes(N, D, V, int(bool(has_bias))))


def _workspace(nbytes: int, device, given: Optional[torch.Tensor]):
    if given is not None:
        if given.device != device or given.dtype != torch.uint8 or given.numel() < nbytes:
            raise ValueError("workspace must be a uint8 CUDA tensor of at least the queried size")
        return given
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


@on_tensor_device
def linear_logp_fwd(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                    bias: Optional[torch.Tensor] = None, temperature: Optional[torch.Tensor] = None,
                    ignore_index: int = IGNORE_INDEX, workspace: Optional[torch.Tensor] = None,
                    out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """Per-token log-prob of the target and the row log-sum-exp (both fp32 [N]).
    hidden / weight are both bf16 or both fp16."""
    dev, N, D, V = _check_inputs(hidden, weight, targets, bias, temperature, allow_f16=True)
    lib = _lib.load()
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    nbytes = int(lib.linear_logp_fwd_workspace_bytes(N, D, V))
    ws = _workspace(nbytes, dev, workspace)
    name = "linear_logp_fwd_f16" if hidden.dtype == torch.float16 else "linear_logp_fwd"
    st = getattr(lib, name)(_ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), _ptr(temperature),
                            N, D, V, int(ignore_index), _ptr(logp), _ptr(lse), _ptr(ws), ws.numel(), _stream(dev))
    _lib.check(name, st)
    return logp, lse


@on_tensor_device
def linear_logp_fwd_noalloc(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                            bias: Optional[torch.Tensor] = None, temperature: Optional[torch.Tensor] = None,
                            ignore_index: int = IGNORE_INDEX,
                            out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """Forward through ``linear_logp_fwd_noalloc``: no workspace, for callers that
    cannot allocate device memory themselves (the library uses its own fixed
    16 MiB device array; pass preallocated ``out`` buffers to allocate nothing
    here either).  Calls that overlap on the GPU share that array and race."""
    dev, N, D, V = _check_inputs(hidden, weight, targets, bias, temperature)
    lib = _lib.load()
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    st = lib.linear_logp_fwd_noalloc(_ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), _ptr(temperature),
                                     N, D, V, int(ignore_index), _ptr(logp), _ptr(lse), _stream(dev))
    _lib.check("linear_logp_fwd_noalloc", st)
    return logp, lse


@on_tensor_device
def linear_logp_bwd(grad_logp: torch.Tensor, saved_lse: torch.Tensor, hidden: torch.Tensor,
                    weight: torch.Tensor, targets: torch.Tensor, bias: Optional[torch.Tensor] = None,
                    temperature: Optional[torch.Tensor] = None, ignore_index: int = IGNORE_INDEX,
                    need_hidden: bool = True, need_weight: bool = True, need_bias: bool = True,
                    workspace: Optional[torch.Tensor] = None):
    """Gradients of sum_n grad_logp[n] * logp[n] w.r.t. hidden, weight and bias
    (hidden / weight gradients in the inputs' dtype, bf16 or fp16)."""
    dev, N, D, V = _check_inputs(hidden, weight, targets, bias, temperature, allow_f16=True)
    _need(grad_logp, "grad_logp", torch.float32, dev, 1)
    _need(saved_lse, "saved_lse", torch.float32, dev, 1)
    if grad_logp.shape[0] != N or saved_lse.shape[0] != N:
        raise ValueError("grad_logp and saved_lse must have N entries")
    lib = _lib.load()
    gh = torch.empty((N, D), dtype=hidden.dtype, device=dev) if need_hidden else None
    gw = torch.empty((V, D), dtype=hidden.dtype, device=dev) if need_weight else None
    gb = torch.empty(V, dtype=torch.float32, device=dev) if (need_bias and bias is not None) else None
    nbytes = int(lib.linear_logp_bwd_workspace_bytes(N, D, V, int(bias is not None)))
    ws = _workspace(nbytes, dev, workspace)
    name = "linear_logp_bwd_f16" if hidden.dtype == torch.float16 else "linear_logp_bwd"
    st = getattr(lib, name)(_ptr(grad_logp), _ptr(saved_lse), _ptr(hidden), _ptr(weight), _ptr(bias),
                            _ptr(targets), _ptr(temperature), N, D, V, int(ignore_index),
                            _ptr(gh), _ptr(gw), _ptr(gb), _ptr(ws), ws.numel(), _stream(dev))
    _lib.check(name, st)
    return gh, gw, gb


def _check_indices(indices: torch.Tensor, device) -> torch.Tensor:
    if not isinstance(indices, torch.Tensor) or indices.dtype != torch.int64 or indices.device != device:
        raise TypeError("indices must be an int64 tensor on the inputs' device")
    return indices.reshape(-1).contiguous()


@on_tensor_device
def linear_logp_fwd_indexed(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                            indices: torch.Tensor, bias: Optional[torch.Tensor] = None,
                            temperature: Optional[torch.Tensor] = None, ignore_index: int = IGNORE_INDEX,
                            out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """Forward on the rows named by ``indices`` only (duplicates count once, out of
    range ignored).  Selected rows of ``out`` get the plain forward's values; the
    others keep their contents (new buffers start as logp 0 / lse -inf).  hidden /
    weight are both bf16 or both fp16."""
    dev, N, D, V = _check_inputs(hidden, weight, targets, bias, temperature, allow_f16=True)
    idx = _check_indices(indices, dev)
    lib = _lib.load()
    if out is None:
        logp = torch.zeros(N, dtype=torch.float32, device=dev)
        lse = torch.full((N,), float("-inf"), dtype=torch.float32, device=dev)
    else:
        logp, lse = out
    K = idx.numel()
    ws = _workspace(int(lib.linear_logp_fwd_indexed_workspace_bytes(N, D, V, K)), dev, None)
    name = "linear_logp_fwd_indexed_f16" if hidden.dtype == torch.float16 else "linear_logp_fwd_indexed"
    st = getattr(lib, name)(_ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets), _ptr(temperature),
                            N, D, V, int(ignore_index), _ptr(idx), K, _ptr(logp), _ptr(lse), _ptr(ws),
                            ws.numel(), _stream(dev))
    _lib.check(name, st)
    return logp, lse


@on_tensor_device
def linear_logp_bwd_indexed(grad_logp: torch.Tensor, saved_lse: torch.Tensor, hidden: torch.Tensor,
                            weight: torch.Tensor, targets: torch.Tensor, indices: torch.Tensor,
                            bias: Optional[torch.Tensor] = None, temperature: Optional[torch.Tensor] = None,
                            ignore_index: int = IGNORE_INDEX, need_hidden: bool = True, need_weight: bool = True,
                            need_bias: bool = True):
    """Gradients of the sum over the selected rows of grad_logp * logp; grad_hidden
    rows that are not selected are zero; 16-bit gradients in the inputs' dtype."""
    dev, N, D, V = _check_inputs(hidden, weight, targets, bias, temperature, allow_f16=True)
    idx = _check_indices(indices, dev)
    _need(grad_logp, "grad_logp", torch.float32, dev, 1)
    _need(saved_lse, "saved_lse", torch.float32, dev, 1)
    lib = _lib.load()
    gh = torch.empty((N, D), dtype=hidden.dtype, device=dev) if need_hidden else None
    gw = torch.empty((V, D), dtype=hidden.dtype, device=dev) if need_weight else None
    gb = torch.empty(V, dtype=torch.float32, device=dev) if (need_bias and bias is not None) else None
    K = idx.numel()
    ws = _workspace(int(lib.linear_logp_bwd_indexed_workspace_bytes(N, D, V, K, int(bias is not None))), dev, None)
    name = "linear_logp_bwd_indexed_f16" if hidden.dtype == torch.float16 else "linear_logp_bwd_indexed"
    st = getattr(lib, name)(_ptr(grad_logp), _ptr(saved_lse), _ptr(hidden), _ptr(weight), _ptr(bias),
                            _ptr(targets), _ptr(temperature), N, D, V, int(ignore_index), _ptr(idx), K,
                            _ptr(gh), _ptr(gw), _ptr(gb), _ptr(ws), ws.numel(), _stream(dev))
    _lib.check(name, st)
    return gh, gw, gb


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the kernel status word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    code = ctypes.c_uint(0)
    with torch.cuda.device(dev):
        st = _lib.load().linear_logp_device_status(_stream(dev), ctypes.byref(code))
    if st not in (_lib.LLP_OK, _lib.LLP_ERR_DEVICE_TIMEOUT):
        _lib.check("linear_logp_device_status", st)
    return int(code.value)


class _LinearLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, bias, targets, temperature, ignore_index):
        logp, lse = linear_logp_fwd(hidden, weight, targets, bias, temperature, ignore_index)
        ctx.save_for_backward(hidden, weight, bias, targets, temperature, lse)
        ctx.ignore_index = ignore_index
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        hidden, weight, bias, targets, temperature, lse = ctx.saved_tensors
        need_h, need_w, need_b = ctx.needs_input_grad[0], ctx.needs_input_grad[1], ctx.needs_input_grad[2]
        gh, gw, gb = linear_logp_bwd(grad_logp.contiguous().float(), lse, hidden, weight, targets, bias,
                                     temperature, ctx.ignore_index, need_h, need_w, need_b)
        return gh, gw, gb, None, None, None


def linear_logp(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                bias: Optional[torch.Tensor] = None, temperature: Optional[torch.Tensor] = None,
                ignore_index: int = IGNORE_INDEX, *, tp_group=None, vocab_start_index: int = 0,
                global_vocab_size: Optional[int] = None) -> torch.Tensor:
    """log_softmax((hidden @ weight^T + bias) / temperature)[targets], fp32, with autograd.

    hidden [..., D] and weight [V, D] both bf16 or both fp16, targets [...] int64,
    bias [V] fp32, temperature [...] fp32 (per token).  Returns fp32 with the
    leading shape of targets.  Gradients reach hidden and weight in their dtype
    and bias as fp32.

    The "Fused Linear LogP" entry point's vocab-parallel arguments: with a
    ``tp_group``, ``weight`` / ``bias`` are this rank's rows ``vocab_start_index
    .. + V_local - 1`` of a head of ``global_vocab_size`` rows (default: the sum
    of the ranks' V_local), targets are global ids, and the shards' statistics
    are merged in ascending rank order (see ``tp.linear_logp_vocab_parallel``).
    """
    lead = targets.shape
    D = hidden.shape[-1]
    h2 = hidden.reshape(-1, D)
    t1 = targets.reshape(-1)
    tau = None if temperature is None else temperature.reshape(-1)
    if h2.shape[0] != t1.shape[0]:
        raise ValueError("hidden and targets must share the leading shape")
    tau = None if tau is None else tau.contiguous()
    if tp_group is not None:
        from . import tp
        if global_vocab_size is None:
            import torch.distributed as dist
            n = torch.tensor([weight.shape[0]], dtype=torch.int64, device=weight.device)
            dist.all_reduce(n, group=tp_group)
            global_vocab_size = int(n.item())
        out = tp.linear_logp_vocab_parallel(h2.contiguous(), weight, t1.contiguous(), bias, tau, group=tp_group,
                                            vocab_start=vocab_start_index, global_vocab_size=global_vocab_size,
                                            ignore_index=ignore_index)
        return out.reshape(lead)
    if vocab_start_index != 0 or global_vocab_size not in (None, weight.shape[0]):
        raise ValueError("vocab_start_index / global_vocab_size describe a vocab shard: pass tp_group too")
    out = _LinearLogp.apply(h2.contiguous(), weight, bias, t1.contiguous(), tau, int(ignore_index))
    return out.reshape(lead)
