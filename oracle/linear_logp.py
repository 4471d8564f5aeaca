"""FP64 CPU oracle for the fused linear selected-token log-probability.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never imports, calls or links it, and
it imports nothing from the product path.

What it computes is the plain definition, written out in float64 with logits
materialised row chunk by row chunk:

* "Fused Linear LogP" (docs page), sections "Reference Semantics" and "Tensor
  Contract": ``log_softmax(hidden @ W^T + b)[target]`` per token, output float32
  there; here float64.
* "Feat/nemotron h lm head logprob cuda", summary: optional per-row temperature.
  Reading taken: the temperature divides the biased logit, z = (h.W + b) / tau,
  and the backward is the derivative of that forward, so dlogits carries 1/tau.
* "recursive deterministic LogP autograd on B200", "Summary by CodeRabbit":
  invalid token ids give a zero log-probability and a negative-infinity
  log-sum-exp; here a target equal to ``ignore_index`` or outside [0, V) is
  invalid and its row contributes nothing to any gradient.
* "add backward support for fused logp CUDA kernels", "Implementation
  details": the gradient w.r.t. the logits is grad_out * (one_hot(t) - softmax).

Every function takes numpy arrays.  bf16 and fp32 inputs convert to float64
exactly, so callers pass ``tensor.double().numpy()``.

Pins (checked by ``tests/test_oracle_pins.py`` against things other than this
file): the float64 library composition of the docs page's reference semantics
(incl. autograd), normalisation over all targets, zero-weight and bias-shift
closed forms, the temperature identity, central finite differences, the
zero-sum gradient identities, hand-derived worked examples in
``tests/golden/``, and brute force on duplicates.  No function here is
"parity unpinned".
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

ROW_CHUNK = 256


def valid_rows(targets: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    """Boolean mask of rows whose target is a real token id.

    A row is invalid when its target equals ``ignore_index`` or lies outside
    [0, V) ("recursive deterministic LogP autograd on B200", Summary: invalid
    token ids; "add backward support for fused logp CUDA kernels", review of the
    selected-token lookup: labels below zero or at least the vocab size give 0).
    """
    t = np.asarray(targets, dtype=np.int64)
    return (t != ignore_index) & (t >= 0) & (t < V)


def logits(hidden: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray],
           temperature: Optional[np.ndarray], rows: np.ndarray) -> np.ndarray:
    """z[r, v] = (hidden[r] . weight[v] + bias[v]) / tau[r] for the given rows.

    "Fused Linear LogP", Reference Semantics: ``F.linear(hidden, weight, bias)``;
    the per-row temperature of "Feat/nemotron h lm head logprob cuda" divides it.
    """
    z = hidden[rows] @ weight.T
    if bias is not None:
        z = z + bias[None, :]
    if temperature is not None:
        z = z / temperature[rows][:, None]
    return z


def _chunks(rows: np.ndarray, size: int = ROW_CHUNK):
    for s in range(0, rows.size, size):
        yield rows[s: s + size]


def forward(hidden: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray],
            targets: np.ndarray, temperature: Optional[np.ndarray],
            ignore_index: int = -100,
            rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """(logp, lse) for every row, or only for ``rows`` (others stay 0 / -inf).

    logp[n] = z[n, t_n] - lse[n],  lse[n] = log sum_v exp(z[n, v])
    ("Fused Linear LogP", Reference Semantics and Tensor Contract: the output is
    z[target] - logsumexp(z)).  The log-sum-exp is evaluated with the row maximum
    subtracted first, which is the textbook stable form in exact arithmetic.
    Invalid rows give logp = 0 and lse = -inf.
    """
    N = hidden.shape[0]
    V = weight.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    logp = np.zeros(N, dtype=np.float64)
    lse = np.full(N, -np.inf, dtype=np.float64)
    ok = valid_rows(t, V, ignore_index)
    sel = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    sel = sel[ok[sel]]
    for r in _chunks(sel):
        z = logits(hidden, weight, bias, temperature, r)
        m = z.max(axis=1)
        s = np.exp(z - m[:, None]).sum(axis=1)
        l = m + np.log(s)
        lse[r] = l
        logp[r] = z[np.arange(r.size), t[r]] - l
    return logp, lse


def dlogits(z: np.ndarray, lse: np.ndarray, t: np.ndarray, g: np.ndarray,
            inv_tau: np.ndarray) -> np.ndarray:
    """d logp / d logits scaled by the upstream gradient, for a block of valid rows.

    dz[r, v] = g_r / tau_r * (onehot(t_r)[v] - softmax(z_r)[v])
    ("add backward support for fused logp CUDA kernels", Implementation details:
    grad_out * (one_hot(token_id) - softmax(logits)); the 1/tau factor is the chain
    rule through z = (h.W + b) / tau).
    """
    p = np.exp(z - lse[:, None])
    onehot = np.zeros_like(p)
    onehot[np.arange(z.shape[0]), t] = 1.0
    return (g * inv_tau)[:, None] * (onehot - p)


def backward(grad_logp: np.ndarray, hidden: np.ndarray, weight: np.ndarray,
             bias: Optional[np.ndarray], targets: np.ndarray,
             temperature: Optional[np.ndarray], ignore_index: int = -100,
             rows: Optional[Sequence[int]] = None,
             need_weight: bool = True):
    """(grad_hidden [N,D], grad_weight [V,D], grad_bias [V] or None), float64.

    grad_hidden = dz @ W, grad_weight = dz^T @ h, grad_bias = sum_n dz
    ("Fused Linear LogP", intro: differentiable w.r.t. hidden, lm_head_weight and
    bias; the gradients of F.linear).  Invalid rows contribute nothing; their
    upstream gradient is never read, so a NaN there cannot leak.  When ``rows`` is
    given only those rows are differentiated (grad_hidden of other rows stays 0 and
    grad_weight / grad_bias then sum over those rows only).  The log-sum-exp is
    recomputed here from the definition; nothing is taken from any other path.
    """
    N, D = hidden.shape
    V = weight.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    g = np.asarray(grad_logp, dtype=np.float64)
    gh = np.zeros((N, D), dtype=np.float64)
    gw = np.zeros((V, D), dtype=np.float64) if need_weight else None
    gb = np.zeros(V, dtype=np.float64) if bias is not None else None
    ok = valid_rows(t, V, ignore_index)
    sel = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    sel = sel[ok[sel]]
    for r in _chunks(sel):
        z = logits(hidden, weight, bias, temperature, r)
        m = z.max(axis=1)
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        inv_tau = np.ones(r.size) if temperature is None else 1.0 / temperature[r]
        dz = dlogits(z, lse, t[r], g[r], inv_tau)
        gh[r] = dz @ weight
        if need_weight:
            gw += dz.T @ hidden[r]
        if gb is not None:
            gb += dz.sum(axis=0)
    return gh, gw, gb


def grad_weight_rows(grad_logp: np.ndarray, hidden: np.ndarray, weight: np.ndarray,
                     bias: Optional[np.ndarray], targets: np.ndarray,
                     temperature: Optional[np.ndarray], vocab_rows: Sequence[int],
                     ignore_index: int = -100) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """grad_weight[vocab_rows] and grad_bias[vocab_rows] without forming [V, D].

    Needs every valid row's log-sum-exp (a full pass over the logits, streamed in
    row chunks), then dz[:, vocab_rows] only.  Same definition as ``backward``.
    """
    N, D = hidden.shape
    V = weight.shape[0]
    vr = np.asarray(vocab_rows, dtype=np.int64)
    _, lse = forward(hidden, weight, bias, targets, temperature, ignore_index)
    t = np.asarray(targets, dtype=np.int64)
    g = np.asarray(grad_logp, dtype=np.float64)
    ok = valid_rows(t, V, ignore_index)
    sel = np.arange(N)[ok]
    gw = np.zeros((vr.size, D), dtype=np.float64)
    gb = np.zeros(vr.size, dtype=np.float64)
    for r in _chunks(sel, 4096):
        z = hidden[r] @ weight[vr].T
        if bias is not None:
            z = z + bias[vr][None, :]
        if temperature is not None:
            z = z / temperature[r][:, None]
        inv_tau = np.ones(r.size) if temperature is None else 1.0 / temperature[r]
        p = np.exp(z - lse[r][:, None])
        onehot = (t[r][:, None] == vr[None, :]).astype(np.float64)
        dz = (g[r] * inv_tau)[:, None] * (onehot - p)
        gw += dz.T @ hidden[r]
        gb += dz.sum(axis=0)
    return gw, (gb if bias is not None else None)
