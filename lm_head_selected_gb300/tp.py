"""Vocab-parallel (tensor-parallel) fused linear log-prob.

"Fused Linear LogP", Tensor Parallel Vocab Shards: each rank holds a contiguous
weight shard [V_local, D] (and bias shard) starting at global vocab id
``vocab_start``; the shards partition [0, global_vocab_size).  Each rank
computes its shard's per-row (max, sum of exp, target logit); the ranks
all-gather these triples and merge them in ascending rank order; in the
backward every rank forms its local dlogits with the merged lse, and the fp32
grad_hidden contributions are summed over ranks in ascending rank order and
rounded once to bf16 (the page's all-reduce of hidden.grad); the weight / bias
gradients stay local.  Summing in a fixed rank order (instead of an all-reduce
whose summation order belongs to the collective library) keeps the result
independent of collective timing.

The grad_hidden sum is a reduce-scatter done by hand: an all_to_all hands rank
q every rank's contribution to the q-th block of token rows, rank q sums its
block in ascending rank order and rounds it once, and an all_gather of the
rounded blocks gives every rank the whole gradient.  Per rank that moves
(R-1)/R * N*D*(4 + 2) bytes, against (R-1) * N*D*4 bytes (and an R*N*D*4-byte
buffer) for all-gathering every contribution; each element's sum has the same
terms in the same order either way, so both give the same bits
(``grad_hidden_exchange="gather"`` keeps the gather form).

The device work is in ``liblinear_logp.so``; torch.distributed moves the
triples and partials.  ``ShardOps`` groups the device operations; the default
is the CUDA library.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Callable, Optional

import torch
import torch.distributed as dist

from . import _lib
from .ops import IGNORE_INDEX, _check_inputs, _need, _ptr, _stream, _workspace, on_tensor_device


@on_tensor_device
def fwd_shard(hidden, weight_local, targets, vocab_start, bias_local=None, temperature=None,
              ignore_index=IGNORE_INDEX):
    """-> stats fp32 [3, N]: (max, sum of exp(z - max), target logit or -inf) of this shard.
    hidden / weight_local are both bf16 or both fp16."""
    dev, N, D, V = _check_inputs(hidden, weight_local, targets, bias_local, temperature, allow_f16=True)
    lib = _lib.load()
    stats = torch.empty((3, N), dtype=torch.float32, device=dev)
    ws = _workspace(int(lib.linear_logp_fwd_workspace_bytes(N, D, V)), dev, None)
    name = "linear_logp_fwd_shard_f16" if hidden.dtype == torch.float16 else "linear_logp_fwd_shard"
    st = getattr(lib, name)(_ptr(hidden), _ptr(weight_local), _ptr(bias_local), _ptr(targets), _ptr(temperature),
                            N, D, V, int(vocab_start), int(ignore_index), _ptr(stats[0]), _ptr(stats[1]),
                            _ptr(stats[2]), _ptr(ws), ws.numel(), _stream(dev))
    _lib.check(name, st)
    return stats


@on_tensor_device
def merge_shards(gathered, targets, global_vocab_size, ignore_index=IGNORE_INDEX):
    """gathered fp32 [R, 3, N] in rank order -> (logp, lse)."""
    R, three, N = gathered.shape
    assert three == 3
    dev = gathered.device
    g = gathered.permute(1, 0, 2).contiguous()  # [3, R, N]
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    st = _lib.load().linear_logp_merge_shards(_ptr(g[0]), _ptr(g[1]), _ptr(g[2]), R, N, _ptr(targets),
                                              int(global_vocab_size), int(ignore_index), _ptr(logp), _ptr(lse),
                                              _stream(dev))
    _lib.check("linear_logp_merge_shards", st)
    return logp, lse


@on_tensor_device
def bwd_shard(grad_logp, lse, hidden, weight_local, targets, vocab_start, global_vocab_size, bias_local=None,
              temperature=None, ignore_index=IGNORE_INDEX, need_weight=True, need_bias=True):
    """-> (grad_hidden contribution fp32 [N, D], local grad_weight in the inputs' dtype, local grad_bias fp32)."""
    dev, N, D, V = _check_inputs(hidden, weight_local, targets, bias_local, temperature, allow_f16=True)
    _need(grad_logp, "grad_logp", torch.float32, dev, 1)
    _need(lse, "lse", torch.float32, dev, 1)
    lib = _lib.load()
    gh = torch.empty((N, D), dtype=torch.float32, device=dev)
    gw = torch.empty((V, D), dtype=hidden.dtype, device=dev) if need_weight else None
    gb = torch.empty(V, dtype=torch.float32, device=dev) if (need_bias and bias_local is not None) else None
    ws = _workspace(int(lib.linear_logp_bwd_workspace_bytes(N, D, V, int(bias_local is not None))), dev, None)
    name = "linear_logp_bwd_shard_f16" if hidden.dtype == torch.float16 else "linear_logp_bwd_shard"
    st = getattr(lib, name)(_ptr(grad_logp), _ptr(lse), _ptr(hidden), _ptr(weight_local), _ptr(bias_local),
                            _ptr(targets), _ptr(temperature), N, D, V, int(vocab_start), int(global_vocab_size),
                            int(ignore_index), _ptr(gh), _ptr(gw), _ptr(gb), _ptr(ws), ws.numel(), _stream(dev))
    _lib.check(name, st)
    return gh, gw, gb


@on_tensor_device
def sum_partials(parts, dtype=torch.bfloat16):
    """parts fp32 [R, ...] -> sum over R in ascending order, rounded once to dtype (bf16 or fp16)."""
    if dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("sum_partials returns bf16 or fp16")
    R = parts.shape[0]
    count = parts[0].numel()
    out = torch.empty(parts.shape[1:], dtype=dtype, device=parts.device)
    name = "linear_logp_sum_partials_f16" if dtype == torch.float16 else "linear_logp_sum_partials"
    st = getattr(_lib.load(), name)(_ptr(parts.contiguous()), R, count, _ptr(out), _stream(parts.device))
    _lib.check(name, st)
    return out


@dataclasses.dataclass
class ShardOps:
    """The device operations of the vocab-parallel path (CUDA library by default)."""
    fwd_shard: Callable = fwd_shard
    merge_shards: Callable = merge_shards
    bwd_shard: Callable = bwd_shard
    sum_partials: Callable = sum_partials


def _all_gather(t: torch.Tensor, group) -> torch.Tensor:
    """[R, *t.shape] with rank r's tensor at index r."""
    world = dist.get_world_size(group)
    outs = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(outs, t.contiguous(), group=group)
    return torch.stack(outs)


def rank_ordered_sum(part: torch.Tensor, group, dtype, ops: "ShardOps",
                     exchange: str = "reduce_scatter") -> torch.Tensor:
    """Sum over the ranks of ``group`` of each rank's fp32 ``part`` [N, D], in
    ascending rank order, rounded once to ``dtype``; the whole result on every rank.

    exchange="reduce_scatter": all_to_all of row blocks of ceil(N/R) rows (the
    last block zero-padded), an ordered sum of this rank's block, all_gather of
    the rounded blocks.  exchange="gather": all_gather of every rank's whole
    contribution, then the ordered sum of all of it.  Same terms, same order,
    same rounding per element: the same bits.
    """
    if exchange == "gather":
        return ops.sum_partials(_all_gather(part, group), dtype)
    if exchange != "reduce_scatter":
        raise ValueError(f"unknown grad_hidden exchange {exchange!r}")
    world = dist.get_world_size(group)
    N, D = part.shape
    rows = -(-N // world) if N else 0
    send = part.contiguous()
    if rows * world != N:
        send = torch.cat([send, send.new_zeros((rows * world - N, D))])
    recv = torch.empty_like(send)  # block r: rank r's contribution to this rank's rows
    dist.all_to_all_single(recv, send, group=group)
    mine = ops.sum_partials(recv.view(world, rows, D), dtype)
    out = mine.new_empty((world * rows, D))
    dist.all_gather_into_tensor(out, mine.contiguous(), group=group)
    return out[:N]


class _VocabParallelLinearLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight_local, bias_local, targets, temperature, group, vocab_start, global_v,
                ignore_index, ops, exchange):
        stats = ops.fwd_shard(hidden, weight_local, targets, vocab_start, bias_local, temperature, ignore_index)
        gathered = _all_gather(stats, group)
        logp, lse = ops.merge_shards(gathered, targets, global_v, ignore_index)
        ctx.save_for_backward(hidden, weight_local, bias_local, targets, temperature, lse)
        ctx.meta = (group, vocab_start, global_v, ignore_index, ops, exchange)
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        hidden, weight_local, bias_local, targets, temperature, lse = ctx.saved_tensors
        group, vocab_start, global_v, ignore_index, ops, exchange = ctx.meta
        gh_part, gw, gb = ops.bwd_shard(grad_logp.contiguous().float(), lse, hidden, weight_local, targets,
                                        vocab_start, global_v, bias_local, temperature, ignore_index,
                                        ctx.needs_input_grad[1], ctx.needs_input_grad[2])
        gh = rank_ordered_sum(gh_part, group, hidden.dtype, ops, exchange) if ctx.needs_input_grad[0] else None
        return gh, gw, gb, None, None, None, None, None, None, None, None


def linear_logp_vocab_parallel(hidden: torch.Tensor, weight_local: torch.Tensor, targets: torch.Tensor,
                               bias_local: Optional[torch.Tensor] = None,
                               temperature: Optional[torch.Tensor] = None, *, group=None, vocab_start: int,
                               global_vocab_size: int, ignore_index: int = IGNORE_INDEX,
                               ops: Optional[ShardOps] = None,
                               grad_hidden_exchange: str = "reduce_scatter") -> torch.Tensor:
    """Per-token log-prob with the LM head sharded over the vocab across ``group``.

    hidden [N, D] (replicated), weight_local [V_local, D] rows vocab_start ..
    vocab_start + V_local - 1 of the global head, targets [N] global ids
    (replicated), bias_local [V_local] optional.  Returns logp fp32 [N]; its
    backward gives grad_hidden (summed over ranks in ascending rank order; see
    ``rank_ordered_sum`` for the two exchanges) and the local weight / bias
    gradients.
    """
    if grad_hidden_exchange not in ("reduce_scatter", "gather"):
        raise ValueError(f"unknown grad_hidden exchange {grad_hidden_exchange!r}")
    return _VocabParallelLinearLogp.apply(hidden, weight_local, bias_local, targets, temperature, group,
                                          int(vocab_start), int(global_vocab_size), int(ignore_index),
                                          ops or ShardOps(), grad_hidden_exchange)
