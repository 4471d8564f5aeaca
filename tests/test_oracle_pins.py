"""Pins for the FP64 oracle, checked against things other than the oracle itself.

Each test below would fail for a plausible slip in ``oracle/linear_logp.py``
(a dropped bias, the temperature applied to the wrong factor, a transposed
operand in a gradient, a wrong sign in dlogits, an off-by-one target gather,
ignored rows leaking into a reduction):

* the float64 library composition of the docs page's reference semantics
  ("Fused Linear LogP", Reference Semantics), forward and autograd;
* closed forms: normalisation over all V targets, zero weights, V = 1,
  constant bias / logit shifts, the temperature identity;
* central finite differences of sum_n g_n logp_n;
* the zero-sum identities of the gradients (sum_v dz = 0 per row);
* brute-force additivity over rows for duplicate targets;
* the hand-derived worked example in ``tests/golden/``.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(x):
    return None if x is None else x.double().numpy()


def _problem(N, D, V, seed, bias=True, temp=True, n_ignore=1, n_oor=0, scale=1.0):
    inp = workloads.make_inputs(
        N, D, V, seed, hidden_std=1.0, weight_std=scale / math.sqrt(D),
        bias_std=0.3 if bias else None, temperature_range=(0.6, 1.7) if temp else None,
        n_ignore=n_ignore, n_out_of_range=n_oor, grad_std=1.0)
    return inp


def _torch_reference(inp):
    """The docs page's reference semantics in float64 torch ops, with per-row
    temperature; invalid rows are masked out afterwards."""
    h = inp.hidden.double().requires_grad_(True)
    W = inp.weight.double().requires_grad_(True)
    b = None if inp.bias is None else inp.bias.double().requires_grad_(True)
    z = torch.nn.functional.linear(h, W, b)
    if inp.temperature is not None:
        z = z / inp.temperature.double()[:, None]
    lp_all = torch.log_softmax(z, dim=-1)
    lse_all = torch.logsumexp(z, dim=-1)
    V = inp.V
    t = inp.targets
    ok = (t != inp.ignore_index) & (t >= 0) & (t < V)
    tt = torch.where(ok, t, torch.zeros_like(t))
    lp = lp_all.gather(-1, tt[:, None]).squeeze(-1)
    lp = torch.where(ok, lp, torch.zeros_like(lp))
    g = torch.where(ok, inp.grad_logp.double(), torch.zeros_like(inp.grad_logp.double()))
    (lp * g).sum().backward()
    lse = torch.where(ok, lse_all, torch.full_like(lse_all, -math.inf))
    gb = None if b is None else b.grad.numpy()
    return lp.detach().numpy(), lse.detach().numpy(), h.grad.numpy(), W.grad.numpy(), gb


def _oracle(inp):
    a = (_np(inp.hidden), _np(inp.weight), _np(inp.bias), inp.targets.numpy(),
         _np(inp.temperature), inp.ignore_index)
    logp, lse = oracle.forward(*a)
    gh, gw, gb = oracle.backward(_np(inp.grad_logp), *a)
    return logp, lse, gh, gw, gb


@pytest.mark.parametrize("bias,temp", [(True, True), (False, False), (True, False), (False, True)])
def test_matches_library_reference_semantics(bias, temp):
    inp = _problem(9, 16, 13, seed=7, bias=bias, temp=temp, n_ignore=1, n_oor=2)
    lp, lse, gh, gw, gb = _oracle(inp)
    rlp, rlse, rgh, rgw, rgb = _torch_reference(inp)
    np.testing.assert_allclose(lp, rlp, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(rlse))
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse[fin], rlse[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gh, rgh, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gw, rgw, rtol=0, atol=1e-12)
    if bias:
        np.testing.assert_allclose(gb, rgb, rtol=0, atol=1e-12)
    else:
        assert gb is None


def test_tiny_workload_matches_library_reference():
    inp = workloads.tiny()
    lp, lse, gh, gw, gb = _oracle(inp)
    rlp, rlse, rgh, rgw, rgb = _torch_reference(inp)
    np.testing.assert_allclose(lp, rlp, rtol=0, atol=1e-10)
    np.testing.assert_allclose(gh, rgh, rtol=0, atol=1e-10)
    np.testing.assert_allclose(gw, rgw, rtol=0, atol=1e-10)
    np.testing.assert_allclose(gb, rgb, rtol=0, atol=1e-10)
    assert (inp.targets == inp.ignore_index).sum() == 4
    assert np.all(lp[(inp.targets == -100).numpy()] == 0)


def test_normalisation_over_all_targets():
    """sum_t exp(logp(h, t)) = 1 over all V targets of the tiny workload's vocab."""
    inp = workloads.tiny()
    V = inp.V
    rows = [0, 17, 42]
    h = np.repeat(_np(inp.hidden)[rows], V, axis=0)
    t = np.tile(np.arange(V), len(rows))
    temp = np.repeat(np.array([1.0, 0.8, 1.3]), V)
    logp, lse = oracle.forward(h, _np(inp.weight), _np(inp.bias), t, temp)
    tot = np.exp(logp).reshape(len(rows), V).sum(axis=1)
    np.testing.assert_allclose(tot, 1.0, rtol=0, atol=1e-12)
    assert np.all(logp <= 0)
    # lse is one value per row, independent of the target
    l2 = lse.reshape(len(rows), V)
    assert np.all(l2 == l2[:, :1])


def test_single_token_vocab_gives_zero():
    rng = np.random.default_rng(0)
    h = rng.standard_normal((5, 4))
    W = rng.standard_normal((1, 4))
    b = np.array([0.7])
    logp, lse = oracle.forward(h, W, b, np.zeros(5, dtype=np.int64), None)
    assert np.all(logp == 0.0)
    np.testing.assert_allclose(lse, h @ W[0] + 0.7, rtol=0, atol=1e-14)
    gh, gw, gb = oracle.backward(np.ones(5), h, W, b, np.zeros(5, dtype=np.int64), None)
    assert np.all(gh == 0) and np.all(gw == 0) and np.all(gb == 0)


def test_zero_weights_give_uniform_distribution():
    rng = np.random.default_rng(1)
    for V in (1, 2, 7, 4096):
        h = rng.standard_normal((6, 8))
        W = np.zeros((V, 8))
        t = rng.integers(0, V, 6)
        temp = rng.uniform(0.5, 2.0, 6)
        logp, lse = oracle.forward(h, W, None, t, temp)
        np.testing.assert_allclose(logp, -math.log(V), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, math.log(V), rtol=0, atol=1e-13)


def test_constant_bias_shift():
    """b + c leaves logp unchanged and lifts lse by c / tau."""
    inp = _problem(12, 16, 29, seed=3, bias=True, temp=True, n_ignore=0)
    a = [_np(inp.hidden), _np(inp.weight), _np(inp.bias), inp.targets.numpy(), _np(inp.temperature)]
    lp0, lse0 = oracle.forward(*a)
    c = 37.25
    a[2] = a[2] + c
    lp1, lse1 = oracle.forward(*a)
    np.testing.assert_allclose(lp1, lp0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1 - lse0, c / a[4], rtol=0, atol=1e-12)
    # and the gradients do not move either
    g = _np(inp.grad_logp)
    a[2] = a[2] - c
    g0 = oracle.backward(g, *a)
    a[2] = a[2] + c
    g1 = oracle.backward(g, *a)
    for x, y in zip(g0, g1):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_column_shift_of_long_context_row():
    """The long-context stress row: logits shifted by exactly 9984 leave logp unchanged."""
    inp = workloads.long_context(N=130, D=64, V=300, seed=11)
    a = [_np(inp.hidden), _np(inp.weight), None, inp.targets.numpy(), None]
    lp_s, lse_s = oracle.forward(*a)
    a0 = [x.copy() if isinstance(x, np.ndarray) else x for x in a]
    a0[0][0, -1] = 0.0
    lp_0, lse_0 = oracle.forward(*a0)
    np.testing.assert_allclose(lp_s[0], lp_0[0], rtol=0, atol=1e-9)
    np.testing.assert_allclose(lse_s[0] - lse_0[0], workloads.LONG_SHIFT, rtol=0, atol=1e-9)
    np.testing.assert_array_equal(lp_s[1:], lp_0[1:])
    assert torch.equal(inp.targets[64:128], inp.targets[0:64])


def test_temperature_identity():
    """logp(h, b, tau) = logp(h / tau, b / tau, 1) with W shared."""
    inp = _problem(10, 16, 31, seed=5, bias=True, temp=True, n_ignore=0)
    h, W, b, t, tau = _np(inp.hidden), _np(inp.weight), _np(inp.bias), inp.targets.numpy(), _np(inp.temperature)
    lp, lse = oracle.forward(h, W, b, t, tau)
    for n in range(h.shape[0]):
        lp1, lse1 = oracle.forward(h[n:n + 1] / tau[n], W, b / tau[n], t[n:n + 1], None)
        np.testing.assert_allclose(lp1[0], lp[n], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse1[0], lse[n], rtol=0, atol=1e-12)


def test_ignore_rows_and_out_of_range_targets():
    inp = _problem(8, 16, 13, seed=9, bias=True, temp=True, n_ignore=2, n_oor=2)
    t = inp.targets.numpy()
    bad = (t == -100) | (t < 0) | (t >= 13)
    assert bad.sum() == 4
    g = _np(inp.grad_logp)
    g[bad] = np.nan  # must never be read
    a = (_np(inp.hidden), _np(inp.weight), _np(inp.bias), t, _np(inp.temperature))
    lp, lse = oracle.forward(*a)
    assert np.all(lp[bad] == 0) and np.all(np.isneginf(lse[bad]))
    assert np.all(np.isfinite(lse[~bad]))
    gh, gw, gb = oracle.backward(g, *a)
    assert np.all(gh[bad] == 0)
    assert np.all(np.isfinite(gh)) and np.all(np.isfinite(gw)) and np.all(np.isfinite(gb))
    # the valid rows alone give the same weight / bias gradients
    keep = np.nonzero(~bad)[0]
    gh2, gw2, gb2 = oracle.backward(g[keep], a[0][keep], a[1], a[2], t[keep], a[4][keep])
    np.testing.assert_allclose(gw, gw2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(gb, gb2, rtol=0, atol=1e-13)
    # everything ignored: all gradients zero
    t_all = np.full(8, -100)
    gh3, gw3, gb3 = oracle.backward(g, a[0], a[1], a[2], t_all, a[4])
    assert np.all(gh3 == 0) and np.all(gw3 == 0) and np.all(gb3 == 0)
    lp3, lse3 = oracle.forward(a[0], a[1], a[2], t_all, a[4])
    assert np.all(lp3 == 0) and np.all(np.isneginf(lse3))


def test_finite_differences():
    """Central differences of L = sum_n g_n logp_n (FP64, step 1e-6) on N=3, D=8, V=11
    with bias, tau != 1 and one ignored row."""
    rng = np.random.default_rng(2024)
    N, D, V = 3, 8, 11
    h = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.5
    b = rng.standard_normal(V) * 0.3
    tau = np.array([0.7, 1.6, 1.1])
    t = np.array([4, -100, 9])
    g = np.array([1.3, 5.0, -0.8])

    def L(h_, W_, b_):
        lp, _ = oracle.forward(h_, W_, b_, t, tau)
        return float(np.dot(g, lp))

    gh, gw, gb = oracle.backward(g, h, W, b, t, tau)
    eps = 1e-6

    def fd(x, f):
        out = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp = x.copy(); xp[i] += eps
            xm = x.copy(); xm[i] -= eps
            out[i] = (f(xp) - f(xm)) / (2 * eps)
        return out

    fh = fd(h, lambda x: L(x, W, b))
    fw = fd(W, lambda x: L(h, x, b))
    fb = fd(b, lambda x: L(h, W, x))
    for ana, num in ((gh, fh), (gw, fw), (gb, fb)):
        scale = max(1.0, np.abs(num).max())
        assert np.abs(ana - num).max() / scale < 1e-6
    assert np.all(gh[1] == 0)


def test_gradient_zero_sum_identities():
    """sum_v dz[n, v] = 0 per row, hence sum_v grad_b = 0 and sum_v grad_W[v, :] = 0."""
    inp = _problem(16, 24, 37, seed=13, bias=True, temp=True, n_ignore=2)
    a = (_np(inp.hidden), _np(inp.weight), _np(inp.bias), inp.targets.numpy(), _np(inp.temperature))
    gh, gw, gb = oracle.backward(_np(inp.grad_logp), *a)
    assert abs(gb.sum()) < 1e-12
    np.testing.assert_allclose(gw.sum(axis=0), 0.0, rtol=0, atol=1e-12)
    assert np.abs(gb).max() > 1e-3  # not trivially zero


def test_duplicate_targets_are_additive():
    """Rows sharing a target each add their own contribution (brute force, row by row)."""
    rng = np.random.default_rng(5)
    N, D, V = 6, 5, 7
    h = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D))
    b = rng.standard_normal(V)
    tau = rng.uniform(0.7, 1.3, N)
    t = np.array([3, 3, 3, 1, 3, 1])
    g = rng.standard_normal(N)
    gh, gw, gb = oracle.backward(g, h, W, b, t, tau)
    sw = np.zeros_like(gw)
    sb = np.zeros_like(gb)
    for n in range(N):
        _, w1, b1 = oracle.backward(g[n:n + 1], h[n:n + 1], W, b, t[n:n + 1], tau[n:n + 1])
        sw += w1
        sb += b1
    np.testing.assert_allclose(gw, sw, rtol=0, atol=1e-13)
    np.testing.assert_allclose(gb, sb, rtol=0, atol=1e-13)


def test_row_subsets_and_sampled_vocab_rows():
    inp = _problem(40, 16, 50, seed=17, bias=True, temp=True, n_ignore=3)
    a = (_np(inp.hidden), _np(inp.weight), _np(inp.bias), inp.targets.numpy(), _np(inp.temperature))
    g = _np(inp.grad_logp)
    lp, lse = oracle.forward(*a)
    rows = [0, 5, 39, 17]
    lp_r, lse_r = oracle.forward(*a, rows=rows)
    np.testing.assert_array_equal(lp_r[rows], lp[rows])
    gh, gw, gb = oracle.backward(g, *a)
    gh_r, _, _ = oracle.backward(g, *a, rows=rows, need_weight=False)
    np.testing.assert_array_equal(gh_r[rows], gh[rows])
    vr = [0, 3, 49, 22]
    gw_v, gb_v = oracle.grad_weight_rows(g, *a, vocab_rows=vr)
    np.testing.assert_allclose(gw_v, gw[vr], rtol=0, atol=1e-13)
    np.testing.assert_allclose(gb_v, gb[vr], rtol=0, atol=1e-13)


def _eval(expr, env):
    safe = {"exp": math.exp, "log": math.log, "inf": math.inf}
    safe.update(env)
    return float(eval(expr, {"__builtins__": {}}, safe))


def test_hand_derived_worked_example():
    with open(os.path.join(GOLDEN, "worked_example_v3.json")) as f:
        ex = json.load(f)
    i = ex["inputs"]
    h = np.array(i["hidden"], dtype=np.float64)
    W = np.array(i["weight"], dtype=np.float64)
    b = np.array(i["bias"], dtype=np.float64)
    tau = np.array(i["temperature"], dtype=np.float64)
    t = np.array(i["targets"], dtype=np.int64)
    g = np.array(i["grad_logp"], dtype=np.float64)
    env = {}
    for k, e in ex["defs"].items():
        env[k] = _eval(e, env)
    exp = {k: np.array([[_eval(e, env) for e in r] if isinstance(r, list) else _eval(r, env)
                        for r in v]) for k, v in ex["expected"].items()}
    lp, lse = oracle.forward(h, W, b, t, tau, i["ignore_index"])
    gh, gw, gb = oracle.backward(g, h, W, b, t, tau, i["ignore_index"])
    np.testing.assert_allclose(lp, exp["logp"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, exp["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(gh, exp["grad_hidden"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(gw, exp["grad_weight"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(gb, exp["grad_bias"], rtol=0, atol=1e-14)


def test_workloads_are_seeded_and_shaped():
    a = workloads.tiny()
    b = workloads.tiny()
    assert torch.equal(a.hidden, b.hidden) and torch.equal(a.targets, b.targets)
    assert (a.N, a.D, a.V) == (64, 256, 4096)
    assert a.hidden.dtype == torch.bfloat16 and a.weight.dtype == torch.bfloat16
    assert a.bias.dtype == torch.float32 and a.targets.dtype == torch.int64
    r = workloads.rl_scoring(N=2000, D=128, V=5000, seed=3)
    frac_ign = (r.targets == -100).float().mean().item()
    assert 0.02 < frac_ign < 0.09
    lc = workloads.long_context(N=200, D=32, V=100)
    assert lc.hidden[0, -1].item() == workloads.LONG_SHIFT
    assert torch.all(lc.hidden[1:, -1] == 0) and torch.all(lc.weight[:, -1] == 1)
