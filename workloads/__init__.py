"""Seeded synthetic inputs for the fused linear selected-token log-probability.

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no logits, no softmax, no gradients), so both the FP64
oracle and the CUDA path can be fed from it without sharing any computation.

Every workload is shaped like the ones the pages describe: the Nemotron-3-Nano
LM head (hidden 2688, vocab 131072) from "Feat/nemotron h lm head logprob cuda"
(summary and Benchmark sections), scored as an RL post-training head, plus the
small correctness case and the larger training / long-context stress shapes.
All tensors are produced on the CPU with a ``torch.Generator`` seeded from the
workload's seed; callers copy them to the device themselves.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass
class Inputs:
    """One batch of inputs.  Shapes: hidden [N,D] bf16, weight [V,D] bf16,
    bias [V] fp32 or None, targets [N] int64, temperature [N] fp32 or None,
    grad_logp [N] fp32 (the upstream gradient of the per-token log-prob)."""

    hidden: torch.Tensor
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    targets: torch.Tensor
    temperature: Optional[torch.Tensor]
    grad_logp: torch.Tensor
    ignore_index: int = IGNORE_INDEX

    @property
    def N(self) -> int:
        return int(self.hidden.shape[0])

    @property
    def D(self) -> int:
        return int(self.hidden.shape[1])

    @property
    def V(self) -> int:
        return int(self.weight.shape[0])

    def rows(self, idx: torch.Tensor) -> "Inputs":
        """The same problem restricted to the given token rows (weight and bias shared)."""
        idx = torch.as_tensor(idx, dtype=torch.long)
        return Inputs(
            hidden=self.hidden[idx].contiguous(),
            weight=self.weight,
            bias=self.bias,
            targets=self.targets[idx].contiguous(),
            temperature=None if self.temperature is None else self.temperature[idx].contiguous(),
            grad_logp=self.grad_logp[idx].contiguous(),
            ignore_index=self.ignore_index,
        )


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _normal(shape, std: float, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def make_inputs(
    N: int,
    D: int,
    V: int,
    seed: int,
    *,
    hidden_std: float = 1.0,
    weight_std: float = 0.02,
    bias_std: Optional[float] = None,
    temperature_range: Optional[tuple] = None,
    n_ignore: int = 0,
    n_out_of_range: int = 0,
    grad_std: Optional[float] = None,
    dtype: torch.dtype = torch.bfloat16,
) -> Inputs:
    """Generic seeded problem.

    hidden ~ N(0, hidden_std^2) and weight ~ N(0, weight_std^2), rounded to
    ``dtype`` (bf16, or fp16);
    bias ~ N(0, bias_std^2) fp32 when ``bias_std`` is given; per-row temperature
    ~ U[lo, hi] when ``temperature_range`` is given; targets uniform in [0, V) with
    ``n_ignore`` rows set to the ignore index and ``n_out_of_range`` rows set to
    ids outside [0, V) (alternately -1-k and V+k); grad_logp is 1 unless
    ``grad_std`` is given, then N(0, grad_std^2).
    """
    g = _gen(seed)
    hidden = _normal((N, D), hidden_std, g).to(dtype)
    weight = _normal((V, D), weight_std, g).to(dtype)
    bias = None if bias_std is None else _normal((V,), bias_std, g)
    targets = torch.randint(0, V, (N,), generator=g, dtype=torch.int64)
    if N and (n_ignore or n_out_of_range):
        perm = torch.randperm(N, generator=g)
        ign = perm[: min(n_ignore, N)]
        targets[ign] = IGNORE_INDEX
        oor = perm[min(n_ignore, N): min(n_ignore + n_out_of_range, N)]
        for k, r in enumerate(oor.tolist()):
            targets[r] = (-1 - k) if k % 2 == 0 else (V + k)
    temperature = None
    if temperature_range is not None:
        lo, hi = temperature_range
        temperature = lo + (hi - lo) * torch.rand(N, generator=g, dtype=torch.float32)
    if grad_std is None:
        grad = torch.ones(N, dtype=torch.float32)
    else:
        grad = _normal((N,), grad_std, g)
    return Inputs(hidden, weight, bias, targets, temperature, grad)


# --------------------------------------------------------------------------------------
# The named workloads.  Seeds are 1000 + the workload's position in the list below.
# --------------------------------------------------------------------------------------

def tiny(seed: int = 1000) -> Inputs:
    """N=64, D=256, V=4096.  hidden ~ N(0,1) and W ~ N(0, (2/sqrt(D))^2) so that the
    logits have a standard deviation of about 2; bias ~ N(0, 0.1^2); tau = 1;
    4 rows carry the ignore index; grad_logp = 1."""
    D = 256
    return make_inputs(64, D, 4096, seed, hidden_std=1.0, weight_std=2.0 / math.sqrt(D),
                       bias_std=0.1, n_ignore=4)


def nemotron_head(N: int = 32, seed: int = 1001) -> Inputs:
    """Nemotron-3-Nano LM head, D=2688, V=131072, no bias, per-row temperature
    U[0.7, 1.3], uniform targets, hidden ~ N(0,1), W ~ N(0, 0.02^2).  N=32 is the
    batch 2 x seq 16 case; an N=512 pool of the same distribution feeds the
    batch-invariance subsets."""
    return make_inputs(N, 2688, 131072, seed, temperature_range=(0.7, 1.3))


def rl_scoring(N: int = 16384, D: int = 2688, V: int = 131072, seed: int = 1002,
               grad_std: Optional[float] = 1.0) -> Inputs:
    """RL rollout scoring shape (batch 32 x seq 512 at the default N): no bias, tau = 1.

    Target mix: 85% high-probability tokens, 10% uniform tokens, 5% ignore index.
    A high-probability target t is planted by adding gamma * W[t] / (D * 0.02^2) to
    the row's hidden state (gamma ~ U[11, 17]), which lifts that token's logit by about
    gamma above the N(0, ~1) background.  The background's log-mass is about
    log(V) + 1/2 = 12.3, so the planted token carries most of the row's probability
    (log-prob roughly -1.5 .. 0), as a token sampled from the model itself would.
    This draws such tokens without computing any logits or softmax here.
    grad_logp ~ N(0, 1) so the same batch also serves a training step.
    """
    g = _gen(seed)
    w_std = 0.02
    hidden = _normal((N, D), 1.0, g)
    weight = _normal((V, D), w_std, g).to(torch.bfloat16)
    targets = torch.randint(0, V, (N,), generator=g, dtype=torch.int64)
    kind = torch.rand(N, generator=g)
    planted = kind < 0.85
    ignored = kind >= 0.95
    gamma = 11.0 + 6.0 * torch.rand(N, generator=g)
    rows = torch.nonzero(planted).flatten()
    step = 4096
    for s in range(0, rows.numel(), step):
        r = rows[s: s + step]
        hidden[r] += (gamma[r] / (D * w_std * w_std))[:, None] * weight[targets[r]].float()
    targets[ignored] = IGNORE_INDEX
    grad = torch.ones(N) if grad_std is None else _normal((N,), grad_std, g)
    return Inputs(hidden.to(torch.bfloat16), weight, None, targets, None, grad)


def train(N: int = 16384, D: int = 4096, V: int = 128256, seed: int = 1003) -> Inputs:
    """Training step: bias ~ N(0, 0.1^2), grad_logp ~ N(0,1), uniform targets."""
    return make_inputs(N, D, V, seed, bias_std=0.1, grad_std=1.0)


LONG_SHIFT = 9984.0  # bf16(1e4): exactly representable, so the shifted row moves by 9984


def long_context(N: int = 65600, D: int = 2688, V: int = 131072, seed: int = 1004,
                 shift_row: int = 0) -> Inputs:
    """Long-context stress: N=65600 (not a power of two), no bias, tau = 1.

    One row's logits are all lifted by the same constant: hidden column D-1 is zero
    for every row, weight column D-1 is exactly 1.0, and the stress row gets
    hidden[row, D-1] = 9984 (bf16 of 1e4).  Its logits therefore move by exactly 9984
    and no other row changes.  Duplicate target ids across rows are guaranteed by
    copying the first 64 targets onto 64 other rows.
    """
    inp = make_inputs(N, D, V, seed)
    inp.hidden[:, D - 1] = 0
    inp.weight[:, D - 1] = 1.0
    if N > shift_row:
        inp.hidden[shift_row, D - 1] = LONG_SHIFT
    if N >= 128:
        inp.targets[64:128] = inp.targets[0:64]
    return inp


WORKLOADS = {
    "tiny": tiny,
    "nemotron_head": nemotron_head,
    "rl_scoring": rl_scoring,
    "train": train,
    "long_context": long_context,
}
