"""Vocab-parallel shards on one GPU: every shard's device work runs in turn on
the same device (no collectives), the shard triples are merged in rank order,
and the results are checked against the unsharded FP64 oracle.  The
multi-rank orchestration is tested with gloo ranks in tests/test_tp_gloo.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_helpers import (GH_ATOL, GH_RTOL, GW_ATOL, GW_RTOL, LOGP_ATOL, assert_close, check_device_status, np64,
                            oracle_args, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def _bounds(V, R):
    # uneven contiguous shards covering [0, V)
    cuts = [0] + [int(V * (r + 1) / R) - (37 if r % 2 == 0 and r < R - 1 else 0) for r in range(R)]
    cuts[-1] = V
    return list(zip(cuts[:-1], cuts[1:]))


def _run_shards(inp, R):
    from lm_head_selected_gb300 import tp
    d = to_device(inp)
    shards = _bounds(inp.V, R)
    stats = []
    for s, e in shards:
        b = None if d["bias"] is None else d["bias"][s:e].contiguous()
        stats.append(tp.fwd_shard(d["hidden"], d["weight"][s:e].contiguous(), d["targets"], s, b, d["temperature"]))
    logp, lse = tp.merge_shards(torch.stack(stats), d["targets"], inp.V)
    parts, gws, gbs = [], [], []
    for s, e in shards:
        b = None if d["bias"] is None else d["bias"][s:e].contiguous()
        gh, gw, gb = tp.bwd_shard(d["grad_logp"], lse, d["hidden"], d["weight"][s:e].contiguous(), d["targets"], s,
                                  inp.V, b, d["temperature"])
        parts.append(gh)
        gws.append(gw)
        gbs.append(gb)
    gh = tp.sum_partials(torch.stack(parts), d["hidden"].dtype)
    gw = torch.cat(gws)
    gb = None if d["bias"] is None else torch.cat(gbs)
    check_device_status()
    return logp, lse, gh, gw, gb


@pytest.mark.parametrize("R,dtype", [(1, torch.bfloat16), (2, torch.bfloat16), (3, torch.bfloat16),
                                     (2, torch.float16)])
def test_sharded_forward_backward_matches_oracle(R, dtype):
    inp = workloads.make_inputs(200, 264, 5000, seed=31 + R, weight_std=2.0 / math.sqrt(264), bias_std=0.3,
                                temperature_range=(0.7, 1.3), n_ignore=4, n_out_of_range=3, grad_std=1.0, dtype=dtype)
    logp, lse, gh, gw, gb = _run_shards(inp, R)
    assert gh.dtype == dtype and gw.dtype == dtype
    a = oracle_args(inp)
    lp_ref, lse_ref = oracle.forward(*a)
    ok = oracle.valid_rows(inp.targets.numpy(), inp.V, -100)
    assert_close("logp", np64(logp), lp_ref, LOGP_ATOL, 0)
    assert_close("lse", np64(lse)[ok], lse_ref[ok], LOGP_ATOL, 0)
    assert np.all(np.isneginf(np64(lse)[~ok]))
    gh_ref, gw_ref, gb_ref = oracle.backward(np64(inp.grad_logp), *a)
    assert_close("grad_hidden", np64(gh), gh_ref, GH_ATOL, GH_RTOL)
    assert_close("grad_weight", np64(gw), gw_ref, GW_ATOL, GW_RTOL)
    assert_close("grad_bias", np64(gb), gb_ref, GW_ATOL, GW_RTOL)


def test_sharded_matches_unsharded_forward():
    """One shard equals the plain forward bitwise (same splits, same merge)."""
    import lm_head_selected_gb300 as llp
    inp = workloads.make_inputs(100, 128, 3000, seed=5, weight_std=0.1, n_ignore=3)
    d = to_device(inp)
    lp1, lse1, _, _, _ = _run_shards(inp, 1)
    lp0, lse0 = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"])
    assert torch.equal(lp1, lp0) and torch.equal(lse1, lse0)


def test_nemotron_head_two_shards():
    inp = workloads.nemotron_head(N=64, seed=1001)
    inp.grad_logp = torch.randn(64, generator=torch.Generator().manual_seed(2))
    logp, lse, gh, gw, gb = _run_shards(inp, 2)
    rows = list(range(0, 64, 5))
    a = oracle_args(inp)
    lp_ref, _ = oracle.forward(*a, rows=rows)
    assert_close("logp[rows]", np64(logp)[rows], lp_ref[rows], LOGP_ATOL, 0)
    gh_ref, _, _ = oracle.backward(np64(inp.grad_logp), *a, rows=rows, need_weight=False)
    # grad_hidden of a row depends only on that row: compare on the sampled rows
    assert_close("grad_hidden[rows]", np64(gh)[rows], gh_ref[rows], GH_ATOL, GH_RTOL)


def test_entry_point_tp_group_of_one_matches_plain():
    """``linear_logp(..., tp_group=...)`` (the pages' entry point) over a group of
    one rank gives the plain path's logp and gradients bitwise: with one shard the
    merges reduce to the same expressions and roundings."""
    import os
    import socket

    import torch.distributed as dist

    import lm_head_selected_gb300 as llp
    if dist.is_initialized():
        pytest.skip("a process group already exists")
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        inp = workloads.make_inputs(96, 256, 3000, seed=77, weight_std=0.12, bias_std=0.2, n_ignore=3,
                                    grad_std=1.0)
        d = to_device(inp)
        res = []
        for kw in ({}, {"tp_group": dist.group.WORLD}):
            h = d["hidden"].view(2, 48, 256).clone().requires_grad_(True)
            w = d["weight"].clone().requires_grad_(True)
            b = d["bias"].clone().requires_grad_(True)
            out = llp.linear_logp(h, w, d["targets"].view(2, 48), b, **kw)
            (out * d["grad_logp"].view(2, 48)).sum().backward()
            res.append((out.detach(), h.grad, w.grad, b.grad))
        check_device_status()
        for a, c in zip(*res):
            assert torch.equal(a, c)
    finally:
        dist.destroy_process_group()
