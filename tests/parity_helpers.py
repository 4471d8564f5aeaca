"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
(via the thin binding) and the FP64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the contract: forward logp abs 5e-3; grad_hidden atol 1e-2 / rtol 1e-2;
# grad_weight and grad_bias atol 0.1 / rtol 0.02 (the pages' reduction cell,
# "Feat/nemotron h lm head logprob cuda", Tolerance section).
LOGP_ATOL = 5e-3
LSE_ATOL = 5e-3
GH_ATOL, GH_RTOL = 1e-2, 1e-2
GW_ATOL, GW_RTOL = 0.1, 0.02


def np64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def oracle_args(inp):
    return (np64(inp.hidden), np64(inp.weight), np64(inp.bias), inp.targets.numpy(),
            np64(inp.temperature), inp.ignore_index)


def to_device(inp, device="cuda"):
    d = {
        "hidden": inp.hidden.to(device),
        "weight": inp.weight.to(device),
        "bias": None if inp.bias is None else inp.bias.to(device),
        "targets": inp.targets.to(device),
        "temperature": None if inp.temperature is None else inp.temperature.to(device),
        "grad_logp": inp.grad_logp.to(device),
        "ignore_index": inp.ignore_index,
    }
    return d


def gpu_fwd(d):
    import lm_head_selected_gb300 as llp
    logp, lse = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"],
                                    d["ignore_index"])
    return logp, lse


def gpu_bwd(d, lse, need_hidden=True, need_weight=True, need_bias=True, grad=None):
    import lm_head_selected_gb300 as llp
    g = d["grad_logp"] if grad is None else grad
    return llp.linear_logp_bwd(g, lse, d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"],
                               d["ignore_index"], need_hidden, need_weight, need_bias)


def check_device_status():
    import lm_head_selected_gb300 as llp
    code = llp.device_status()
    assert code == 0, f"a kernel gave up on a bounded wait (device status {code})"


def assert_close(name, got, ref, atol, rtol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} / {err.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r} (atol {atol}, rtol {rtol}); "
                             f"max abs err {err.max():.3e}")


def check_forward(inp, logp, lse, rows=None):
    """Compare logp / lse (device tensors) with the oracle on all rows or on `rows`."""
    lp_ref, lse_ref = oracle.forward(*oracle_args(inp), rows=rows)
    lp = np64(logp)
    ls = np64(lse)
    sel = np.arange(inp.N) if rows is None else np.asarray(rows)
    valid = oracle.valid_rows(inp.targets.numpy(), inp.V, inp.ignore_index)
    sv = sel[valid[sel]]
    si = sel[~valid[sel]]
    assert_close("logp", lp[sv], lp_ref[sv], LOGP_ATOL, 0.0)
    assert_close("lse", ls[sv], lse_ref[sv], LSE_ATOL, 0.0)
    assert np.all(lp[si] == 0.0), "ignored rows must give logp == 0"
    assert np.all(np.isneginf(ls[si])), "ignored rows must give lse == -inf"


def check_backward(inp, gh, gw, gb, rows=None):
    """Full oracle backward (rows=None) or grad_hidden on sampled rows."""
    args = oracle_args(inp)
    g = np64(inp.grad_logp)
    if rows is None:
        gh_ref, gw_ref, gb_ref = oracle.backward(g, *args, need_weight=gw is not None)
        if gh is not None:
            assert_close("grad_hidden", np64(gh), gh_ref, GH_ATOL, GH_RTOL)
        if gw is not None:
            assert_close("grad_weight", np64(gw), gw_ref, GW_ATOL, GW_RTOL)
        if gb is not None:
            assert_close("grad_bias", np64(gb), gb_ref, GW_ATOL, GW_RTOL)
    else:
        gh_ref, _, _ = oracle.backward(g, *args, rows=rows, need_weight=False)
        r = np.asarray(rows)
        assert_close("grad_hidden[rows]", np64(gh[torch.as_tensor(r, device=gh.device)]), gh_ref[r],
                     GH_ATOL, GH_RTOL)
