"""Pins for the logits-input oracle (``oracle/logits_logp.py``), each checked
against something other than that file: the float64 torch composition
(log_softmax, logsumexp, autograd), the independently pinned linear oracle on
z = h.W^T + b, normalisation over all targets, a +1e4 constant shift, central
finite differences, and zero-sum gradient rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import logits_logp as lo


def _problem(N, V, seed, n_ignore=2, scale=2.0):
    g = np.random.default_rng(seed)
    z = g.standard_normal((N, V)) * scale
    t = g.integers(0, V, N)
    t[:n_ignore] = -100
    if N > n_ignore + 1:
        t[n_ignore] = V + 3  # out of range
    gl = g.standard_normal(N)
    return z, t, gl


def test_matches_torch_log_softmax_and_autograd():
    z, t, gl = _problem(11, 37, 1)
    logp, m, ls = lo.forward(z, t)
    gz = lo.backward(gl, z, t)
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    ok = torch.tensor(lo.valid_rows(t, 37, -100))
    tt = torch.where(ok, torch.tensor(t), torch.zeros(11, dtype=torch.long))
    ref = torch.log_softmax(zt, -1).gather(-1, tt[:, None]).squeeze(-1)
    ref = torch.where(ok, ref, torch.zeros_like(ref))
    (ref * torch.tensor(gl) * ok).sum().backward()
    np.testing.assert_allclose(logp, ref.detach().numpy(), rtol=0, atol=1e-13)
    lse_ref = torch.logsumexp(zt.detach(), -1).numpy()
    okn = ok.numpy()
    np.testing.assert_allclose((m + ls)[okn], lse_ref[okn], rtol=0, atol=1e-13)
    assert np.all(np.isneginf(m[~okn])) and np.all(ls[~okn] == 0)
    np.testing.assert_allclose(gz, zt.grad.numpy(), rtol=0, atol=1e-13)


def test_agrees_with_linear_oracle():
    """Logits formed as h.W^T + b give the same log-probs and the same dlogits
    (the linear oracle's gradients are dlogits contracted with W and h)."""
    g = np.random.default_rng(3)
    N, D, V = 9, 12, 29
    h = g.standard_normal((N, D))
    W = g.standard_normal((V, D)) * 0.4
    b = g.standard_normal(V) * 0.3
    t = g.integers(0, V, N)
    t[4] = -100
    gl = g.standard_normal(N)
    z = h @ W.T + b
    lp_lin, lse_lin = oracle.forward(h, W, b, t, None)
    lp, m, ls = lo.forward(z, t)
    np.testing.assert_allclose(lp, lp_lin, rtol=0, atol=1e-12)
    ok = lo.valid_rows(t, V, -100)
    np.testing.assert_allclose((m + ls)[ok], lse_lin[ok], rtol=0, atol=1e-12)
    gz = lo.backward(gl, z, t)
    gh, gw, gb = oracle.backward(gl, h, W, b, t, None)
    np.testing.assert_allclose(gz @ W, gh, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gz.T @ h, gw, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gz.sum(0), gb, rtol=0, atol=1e-12)


def test_normalisation_and_range():
    z, _, _ = _problem(3, 50, 5, n_ignore=0)
    V = 50
    zz = np.repeat(z, V, axis=0)
    tt = np.tile(np.arange(V), 3)
    logp, _, _ = lo.forward(zz, tt)
    np.testing.assert_allclose(np.exp(logp).reshape(3, V).sum(1), 1.0, rtol=0, atol=1e-13)
    assert np.all(logp <= 0)


def test_large_constant_shift():
    """Adding 1e4 to a row moves row_max by 1e4 and leaves logp and the gradient."""
    z, t, gl = _problem(6, 40, 7, n_ignore=0)
    zs = z.copy()
    zs[2] += 1e4
    lp0, m0, ls0 = lo.forward(z, t)
    lp1, m1, ls1 = lo.forward(zs, t)
    np.testing.assert_allclose(lp1, lp0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(m1[2] - m0[2], 1e4, rtol=0, atol=1e-9)
    np.testing.assert_allclose(ls1, ls0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lo.backward(gl, zs, t), lo.backward(gl, z, t), rtol=0, atol=1e-10)


def test_finite_differences():
    z, t, gl = _problem(4, 9, 11, n_ignore=1)
    gz = lo.backward(gl, z, t)
    eps = 1e-6
    num = np.zeros_like(z)
    for i in np.ndindex(z.shape):
        zp = z.copy(); zp[i] += eps
        zm = z.copy(); zm[i] -= eps
        num[i] = (np.dot(gl, lo.forward(zp, t)[0]) - np.dot(gl, lo.forward(zm, t)[0])) / (2 * eps)
    assert np.abs(gz - num).max() < 1e-7
    assert np.all(gz[0] == 0)


def test_gradient_rows_sum_to_zero_and_ignored_rows_are_zero():
    z, t, gl = _problem(20, 33, 13, n_ignore=3)
    gz = lo.backward(gl, z, t)
    np.testing.assert_allclose(gz.sum(1), 0.0, rtol=0, atol=1e-13)
    bad = ~lo.valid_rows(t, 33, -100)
    assert bad.sum() == 4 and np.all(gz[bad] == 0)
    lp, m, ls = lo.forward(z, t)
    assert np.all(lp[bad] == 0)


def test_rows_subset():
    z, t, _ = _problem(30, 17, 17)
    full = lo.forward(z, t)
    rows = [0, 5, 29, 12]
    sub = lo.forward(z, t, rows=rows)
    for a, b in zip(full, sub):
        np.testing.assert_array_equal(a[rows], b[rows])
