"""Parity at the full workload sizes, in the launch configuration the benchmark
times: every forward row checked for validity, sampled rows against the FP64
oracle, grad_weight / grad_bias of the dense batch itself on sampled vocab rows
(every token contributes; the oracle needs every row's log-sum-exp for that, one
FP64 pass over the logits), grad_weight in full on a batch whose active rows the
oracle can afford (all other rows ignored, so the full-size GEMMs still run over
every token), and bitwise repeatability."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_helpers import (GW_ATOL, GW_RTOL, assert_close, check_backward, check_device_status, check_forward,
                            gpu_bwd, gpu_fwd, np64, oracle_args, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def _sample_rows(N, k, seed, must=()):
    g = torch.Generator().manual_seed(seed)
    rows = set(torch.randperm(N, generator=g)[:k].tolist()) | set(must)
    return sorted(rows)


def _forward_properties(logp, lse, inp):
    valid = torch.as_tensor(oracle.valid_rows(inp.targets.numpy(), inp.V, inp.ignore_index)).cuda()
    assert torch.all(torch.isfinite(logp))
    assert torch.all(logp[valid] <= 5e-3)
    assert torch.all(logp[~valid] == 0)
    assert torch.all(torch.isfinite(lse[valid])) and torch.all(torch.isneginf(lse[~valid]))


def _zero_sum_identities(inp, gw, gb=None):
    """Every valid row's dlogits sums to zero over the vocabulary (g/tau times one
    minus the softmax's total), so at any size sum_v grad_W[v, :] = 0 and
    sum_v grad_b[v] = 0.  Allowed slack: each bf16 element of grad_W carries at
    most 2^-9 relative rounding (so a column sum may stray by that share of the
    column's absolute sum, doubled here), plus 1e-4 of sum_n |g_n / tau_n| |h[n, d]|
    for the fp32 softmax total (1 - sum_v p is about 1e-6 per row) and the fp32
    accumulation.  A dropped term (the one-hot part, a vocab tile, a token
    segment) breaks the identity by far more."""
    valid = torch.as_tensor(oracle.valid_rows(inp.targets.numpy(), inp.V, inp.ignore_index))
    gs = inp.grad_logp.double().abs()
    if inp.temperature is not None:
        gs = gs / inp.temperature.double()
    gs = torch.where(valid, gs, torch.zeros_like(gs))
    s1 = (gs[:, None] * inp.hidden.double().abs()).sum(0).cuda()
    col = gw.double().sum(0)
    mag = gw.double().abs().sum(0)
    bad = col.abs() > 2.0 ** -8 * mag + 1e-4 * s1
    assert not torch.any(bad), f"sum_v grad_W[v, d] != 0 for {int(bad.sum())} columns"
    if gb is not None:
        assert abs(float(gb.double().sum())) <= 1e-4 * float(gs.sum())


def _vocab_rows(inp, k, seed, tile_edges=()):
    """About k vocab rows for a sampled grad_weight check: the targets of several
    valid token rows (their one-hot term lands there), the first and last rows,
    both sides of the given 256-row tile / 128-row CTA edges, and seeded random rows."""
    t = inp.targets
    valid = oracle.valid_rows(t.numpy(), inp.V, inp.ignore_index)
    hit = [int(x) for x in t[torch.as_tensor(valid)][:8].tolist()]
    fixed = {0, 1, inp.V - 1, *hit}
    for e in tile_edges:
        fixed |= {e - 1, e}
    g = torch.Generator().manual_seed(seed)
    rnd = torch.randperm(inp.V, generator=g)[: max(0, k - len(fixed))].tolist()
    return sorted(v for v in fixed | set(rnd) if 0 <= v < inp.V)


def _check_dense_grad_weight_rows(inp, gw, gb, vrows):
    """grad_weight[vrows] (and grad_bias[vrows]) of the dense batch against the
    oracle's sampled-row form, element by element at the reduction tolerance
    ("Feat/nemotron h lm head logprob cuda", Tolerance: atol 0.1 / rtol 0.02)."""
    a = oracle_args(inp)
    gw_ref, gb_ref = oracle.grad_weight_rows(np64(inp.grad_logp), a[0], a[1], a[2], a[3], a[4], vrows,
                                             ignore_index=inp.ignore_index)
    idx = torch.as_tensor(vrows, device=gw.device)
    assert_close("grad_weight[vocab rows]", np64(gw[idx]), gw_ref, GW_ATOL, GW_RTOL)
    if gb is not None:
        assert_close("grad_bias[vocab rows]", np64(gb[idx]), gb_ref, GW_ATOL, GW_RTOL)
    # the check is not vacuous: the sampled rows carry gradients well above the tolerance's floor
    assert float(np.abs(gw_ref).max()) > 2 * GW_ATOL


def _sparse_targets(inp, active, seed):
    """Same inputs, but only `active` rows keep their target; the rest are ignored."""
    g = torch.Generator().manual_seed(seed)
    keep = torch.randperm(inp.N, generator=g)[:active]
    t = torch.full_like(inp.targets, -100)
    t[keep] = inp.targets[keep]
    out = inp.rows(torch.arange(inp.N))
    out.targets = t
    return out


def test_rl_scoring_forward_full_size():
    """N=16384, D=2688, V=131072 (batch 32 x seq 512), high-probability targets."""
    inp = workloads.rl_scoring(seed=1002)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    check_device_status()
    _forward_properties(logp, lse, inp)
    rows = _sample_rows(inp.N, 192, 1, must=(0, inp.N - 1))
    check_forward(inp, logp, lse, rows=rows)
    # the planted targets are high-probability tokens: median logp well above -log V
    valid = torch.as_tensor(oracle.valid_rows(inp.targets.numpy(), inp.V, -100)).cuda()
    assert float(logp[valid].median()) > -4.0
    logp2, lse2 = gpu_fwd(d)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)


def test_rl_head_fwd_bwd_full_size():
    """The benchmark's step (N=16384, D=2688, V=131072, grad_logp ~ N(0,1)): sampled
    grad_hidden rows, sampled grad_weight rows of the dense batch, full grad_weight
    on a batch with 192 active rows."""
    inp = workloads.rl_scoring(seed=1002, grad_std=1.0)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, _ = gpu_bwd(d, lse)
    check_device_status()
    rows = _sample_rows(inp.N, 96, 2, must=(0, inp.N - 1))
    check_backward(inp, gh, None, None, rows=rows)
    gh2, gw2, _ = gpu_bwd(d, lse)
    assert torch.equal(gh, gh2) and torch.equal(gw, gw2)
    _zero_sum_identities(inp, gw)
    _check_dense_grad_weight_rows(inp, gw, None, _vocab_rows(inp, 64, 8, tile_edges=(128, 256, 65536)))
    del gw, gw2, gh2
    sp = _sparse_targets(inp, 192, 3)
    ds = to_device(sp)
    lp_s, lse_s = gpu_fwd(ds)
    _, gw_s, _ = gpu_bwd(ds, lse_s, need_hidden=False)
    check_device_status()
    check_backward(sp, None, gw_s, None)


def test_train_step_full_size():
    """N=16384, D=4096, V=128256 with bias: sampled rows of logp / grad_hidden,
    sampled grad_weight / grad_bias rows of the dense batch (including the last
    256-row vocab tile), grad_weight / grad_bias in full on a batch with 128 active rows."""
    inp = workloads.train()
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    _forward_properties(logp, lse, inp)
    rows = _sample_rows(inp.N, 96, 4, must=(inp.N - 1,))
    check_forward(inp, logp, lse, rows=rows)
    check_backward(inp, gh, None, None, rows=rows)
    assert torch.all(torch.isfinite(gb))
    _zero_sum_identities(inp, gw, gb)
    _check_dense_grad_weight_rows(inp, gw, gb, _vocab_rows(inp, 64, 9, tile_edges=(128, 256, 128000, 128128)))
    del gw, gh
    sp = _sparse_targets(inp, 128, 5)
    ds = to_device(sp)
    lp_s, lse_s = gpu_fwd(ds)
    _, gw_s, gb_s = gpu_bwd(ds, lse_s, need_hidden=False)
    check_device_status()
    check_backward(sp, None, gw_s, gb_s)


def test_long_context_full_size():
    """N=65600 (3 token segments for grad_weight), one row shifted by +9984, duplicate
    targets; two runs bitwise identical; grad_weight in full on 96 active rows."""
    inp = workloads.long_context()
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, _ = gpu_bwd(d, lse)
    check_device_status()
    _forward_properties(logp, lse, inp)
    rows = _sample_rows(inp.N, 96, 6, must=(0, 1, 64, inp.N - 1))
    check_forward(inp, logp, lse, rows=rows)
    check_backward(inp, gh, None, None, rows=rows)
    logp2, lse2 = gpu_fwd(d)
    gh2, gw2, _ = gpu_bwd(d, lse2)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
    assert torch.equal(gh, gh2) and torch.equal(gw, gw2)
    _zero_sum_identities(inp, gw)
    del gw, gw2, gh, gh2
    # the shifted row agrees with its unshifted twin
    twin = inp.rows(torch.tensor([0]))
    twin.hidden[0, -1] = 0
    lp_t, _ = gpu_fwd(to_device(twin))
    assert abs(float(lp_t[0]) - float(logp[0])) < 5e-3
    sp = _sparse_targets(inp, 96, 7)
    ds = to_device(sp)
    lp_s, lse_s = gpu_fwd(ds)
    _, gw_s, _ = gpu_bwd(ds, lse_s, need_hidden=False)
    check_device_status()
    check_backward(sp, None, gw_s, None)
