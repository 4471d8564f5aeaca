"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's source (on the CPU, in
memory: a dropped term, a wrong sign, an off-by-one index, a wrong operand) and
runs a battery of the pins against the copy.  Every mutant must fail at least
one pin, and the unmodified oracle must pass them all.  The pins here restate
``test_oracle_pins.py``'s strongest checks against things outside the oracle:
PyTorch float64 autograd of the reference semantics of the "Fused Linear LogP"
page (log_softmax of F.linear, gathered), central finite differences, the
zero-weight closed form and the ignore / out-of-range rules."""
import importlib.util
import math
import os

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "linear_logp.py")


def _load(source: str, name: str):
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(source, SRC, "exec"), mod.__dict__)
    return mod


def _problem(seed=5, N=6, D=8, V=11):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(N, D))
    w = rng.normal(scale=0.6, size=(V, D))
    b = rng.normal(scale=0.3, size=V)
    tau = rng.uniform(0.7, 1.3, size=N)
    t = rng.integers(0, V, size=N)
    t[1] = -100  # ignored
    t[4] = V     # out of range
    g = rng.normal(size=N)
    return h, w, b, tau, t, g


def _pin_library_reference(orc):
    h, w, b, tau, t, g = _problem()
    ht, wt, bt = (torch.tensor(x, requires_grad=True) for x in (h, w, b))
    z = (ht @ wt.T + bt) / torch.tensor(tau)[:, None]
    ls = torch.log_softmax(z, dim=1)
    ok = (t >= 0) & (t < w.shape[0])
    idx = torch.tensor(np.where(ok, t, 0))
    lp_ref = torch.where(torch.tensor(ok), ls.gather(1, idx[:, None])[:, 0], torch.zeros(()))
    (lp_ref * torch.tensor(np.where(ok, g, 0.0))).sum().backward()
    logp, _ = orc.forward(h, w, b, t, tau)
    gh, gw, gb = orc.backward(g, h, w, b, t, tau)
    return (np.allclose(logp, lp_ref.detach().numpy(), atol=1e-12)
            and np.allclose(gh, ht.grad.numpy(), atol=1e-10)
            and np.allclose(gw, wt.grad.numpy(), atol=1e-10)
            and np.allclose(gb, bt.grad.numpy(), atol=1e-10))


def _pin_finite_differences(orc):
    h, w, b, tau, t, g = _problem(seed=9)
    gh, gw, gb = orc.backward(g, h, w, b, t, tau)

    def f(hh, ww, bb):
        return float(np.dot(g, orc.forward(hh, ww, bb, t, tau)[0]))

    eps = 1e-6
    for arr, grad, args in ((h, gh, lambda x: (x, w, b)), (w, gw, lambda x: (h, x, b)), (b, gb, lambda x: (h, w, x))):
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            up, dn = arr.copy(), arr.copy()
            up[i] += eps
            dn[i] -= eps
            num[i] = (f(*args(up)) - f(*args(dn))) / (2 * eps)
        if not np.allclose(num, grad, rtol=1e-5, atol=1e-7):
            return False
    return True


def _pin_zero_weights(orc):
    h, w, b, tau, t, g = _problem(seed=3)
    V = w.shape[0]
    logp, lse = orc.forward(h, np.zeros_like(w), None, t, tau)
    ok = (t >= 0) & (t < V)
    return np.allclose(logp[ok], -math.log(V), atol=1e-13) and np.allclose(lse[ok], math.log(V), atol=1e-13)


def _pin_invalid_rows(orc):
    h, w, b, tau, t, g = _problem(seed=4)
    t[[0, 3, 5]] = (0, 3, 10)  # real targets
    t[2] = 7  # an ignore index that is also a real token id must still be ignored
    logp, lse = orc.forward(h, w, b, t, tau, ignore_index=7)
    gh, _, _ = orc.backward(g, h, w, b, t, tau, ignore_index=7)
    return (all(logp[i] == 0 and np.isneginf(lse[i]) and not gh[i].any() for i in (1, 2, 4))
            and np.all(logp[[0, 3, 5]] < 0))


PINS = (_pin_library_reference, _pin_finite_differences, _pin_zero_weights, _pin_invalid_rows)


def _passes(orc, pin):
    try:
        return bool(pin(orc))
    except Exception:  # a mutant that crashes on a pin's input has failed it
        return False


MUTATIONS = {
    "bias sign": ("z = z + bias[None, :]", "z = z - bias[None, :]"),
    "temperature multiplies": ("z = z / temperature[rows][:, None]", "z = z * temperature[rows][:, None]"),
    "target index off by one": ("logp[r] = z[np.arange(r.size), t[r]] - l", "logp[r] = z[np.arange(r.size), t[r] - 1] - l"),
    "max dropped from lse": ("l = m + np.log(s)", "l = np.log(s)"),
    "dlogits sign": ("(g * inv_tau)[:, None] * (onehot - p)", "(g * inv_tau)[:, None] * (p - onehot)"),
    "1/tau dropped from dlogits": ("(g * inv_tau)[:, None] * (onehot - p)", "g[:, None] * (onehot - p)"),
    "backward lse without max": ("lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))",
                                 "lse = np.log(np.exp(z - m[:, None]).sum(axis=1))"),
    "tau instead of 1/tau": ("else 1.0 / temperature[r]", "else temperature[r]"),
    "grad_weight rows mispaired": ("gw += dz.T @ hidden[r]", "gw += dz.T @ hidden[r][::-1]"),
    "grad_hidden uses transposed weight rows": ("gh[r] = dz @ weight", "gh[r] = dz @ weight[::-1]"),
    "grad_bias averaged": ("gb += dz.sum(axis=0)", "gb += dz.sum(axis=0) / r.size"),
    "vocab bound off by one": ("& (t < V)", "& (t <= V)"),
    "ignore index not honoured": ("(t != ignore_index) & ", ""),
}


def test_unmodified_oracle_passes_every_pin():
    with open(SRC) as f:
        orc = _load(f.read(), "oracle_control")
    for pin in PINS:
        assert _passes(orc, pin), pin.__name__


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    orc = _load(src.replace(old, new), "oracle_mutant")
    failed = [pin.__name__ for pin in PINS if not _passes(orc, pin)]
    assert failed, f"no pin caught the planted mistake '{name}'"


# ---------------------------------------------------------------------------
# The logits-input oracle ("add backward support for fused logp CUDA kernels"):
# the same check against PyTorch float64 log_softmax + autograd, on logits
# with ignored and out-of-range targets.
# ---------------------------------------------------------------------------
SRC_LOGITS = os.path.join(ROOT, "oracle", "logits_logp.py")


def _pin_logits_library_reference(orc):
    rng = np.random.default_rng(13)
    N, V = 7, 13
    z = rng.normal(scale=3.0, size=(N, V))
    t = rng.integers(0, V, size=N)
    t[2], t[5] = -100, V  # ignored; one past the last token id
    g = rng.normal(size=N)
    zt = torch.tensor(z, requires_grad=True)
    ok = (t >= 0) & (t < V)
    ls = torch.log_softmax(zt, dim=1).gather(1, torch.tensor(np.where(ok, t, 0))[:, None])[:, 0]
    lp_ref = torch.where(torch.tensor(ok), ls, torch.zeros(()))
    (lp_ref * torch.tensor(g)).sum().backward()
    logp, row_max, log_sum = orc.forward(z, t)
    return (np.allclose(logp, lp_ref.detach().numpy(), atol=1e-12)
            and np.allclose((row_max + log_sum)[ok], torch.logsumexp(zt, 1).detach().numpy()[ok], atol=1e-12)
            and np.allclose(orc.backward(g, z, t), zt.grad.numpy(), atol=1e-12))


LOGITS_MUTATIONS = {
    "log-sum sign": ("logp[r] = (z[np.arange(r.size), t[r]] - m) - ls", "logp[r] = (z[np.arange(r.size), t[r]] - m) + ls"),
    "row max kept in the target term": ("logp[r] = (z[np.arange(r.size), t[r]] - m) - ls",
                                        "logp[r] = z[np.arange(r.size), t[r]] - ls"),
    "gradient sign": ("out[r] = g[r][:, None] * (onehot - p)", "out[r] = g[r][:, None] * (p - onehot)"),
    "softmax without the log-sum": ("p = np.exp((z - m[:, None]) - ls[:, None])", "p = np.exp(z - m[:, None])"),
    "vocab bound off by one": ("& (t < V)", "& (t <= V)"),
}


def test_unmodified_logits_oracle_passes():
    with open(SRC_LOGITS) as f:
        assert _passes(_load(f.read(), "logits_control"), _pin_logits_library_reference)


@pytest.mark.parametrize("name", sorted(LOGITS_MUTATIONS))
def test_planted_mistake_in_logits_oracle_fails(name):
    old, new = LOGITS_MUTATIONS[name]
    with open(SRC_LOGITS) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    assert not _passes(_load(src.replace(old, new), "logits_mutant"), _pin_logits_library_reference), name
