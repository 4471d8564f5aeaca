"""FP64 CPU oracle for the logits-input fused log-probability.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle/linear_logp.py``: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; it imports nothing from the product path).

The op takes already materialised logits z [N, V] ("Fused Linear LogP" docs
page: "This differs from Fused LogP, which takes already-materialized logits as
input"), and computes

* forward: logp[n] = z[n, t_n] - lse[n], with the row statistics kept apart as
  row_max[n] = max_v z[n, v] and log_sum[n] = log sum_v exp(z[n, v] - row_max[n])
  ("add backward support for fused logp CUDA kernels", Summary and
  Implementation details: LSE-returning forward that returns row_max and
  log_sum separately, to keep precision under large constant logit shifts);
* backward from those saved statistics: grad_z[n, v] = g_n * (onehot(t_n)[v] -
  exp((z[n, v] - row_max[n]) - log_sum[n])) (same page, Implementation details:
  grad_out * (one_hot - softmax) without a logits-sized probability tensor);
* an invalid target (the ignore index, or outside [0, V)) gives logp 0, lse -inf
  and a zero gradient row ("recursive deterministic LogP autograd on B200",
  Summary).  Reading: for such rows row_max = -inf and log_sum = 0, so that
  lse = row_max + log_sum = -inf as well.

Pins: ``tests/test_oracle_pins_logits.py`` (float64 torch log_softmax and
autograd, agreement with the linear oracle when z = h.W^T + b, normalisation,
a +1e4 shift, finite differences, zero-sum gradient rows, ignored rows).
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

ROW_CHUNK = 512


def valid_rows(targets: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    t = np.asarray(targets, dtype=np.int64)
    return (t != ignore_index) & (t >= 0) & (t < V)


def forward(logits: np.ndarray, targets: np.ndarray, ignore_index: int = -100,
            rows: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(logp, row_max, log_sum), float64, for every row or only `rows`."""
    N, V = logits.shape
    t = np.asarray(targets, dtype=np.int64)
    logp = np.zeros(N)
    row_max = np.full(N, -np.inf)
    log_sum = np.zeros(N)
    ok = valid_rows(t, V, ignore_index)
    sel = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    sel = sel[ok[sel]]
    for s in range(0, sel.size, ROW_CHUNK):
        r = sel[s: s + ROW_CHUNK]
        z = logits[r]
        m = z.max(axis=1)
        ls = np.log(np.exp(z - m[:, None]).sum(axis=1))
        row_max[r] = m
        log_sum[r] = ls
        logp[r] = (z[np.arange(r.size), t[r]] - m) - ls
    return logp, row_max, log_sum


def backward(grad_logp: np.ndarray, logits: np.ndarray, targets: np.ndarray,
             ignore_index: int = -100) -> np.ndarray:
    """grad_logits [N, V], float64; the row statistics are recomputed here."""
    N, V = logits.shape
    t = np.asarray(targets, dtype=np.int64)
    g = np.asarray(grad_logp, dtype=np.float64)
    out = np.zeros((N, V))
    ok = valid_rows(t, V, ignore_index)
    sel = np.arange(N)[ok]
    for s in range(0, sel.size, ROW_CHUNK):
        r = sel[s: s + ROW_CHUNK]
        z = logits[r]
        m = z.max(axis=1)
        ls = np.log(np.exp(z - m[:, None]).sum(axis=1))
        p = np.exp((z - m[:, None]) - ls[:, None])
        onehot = np.zeros_like(p)
        onehot[np.arange(r.size), t[r]] = 1.0
        out[r] = g[r][:, None] * (onehot - p)
    return out
