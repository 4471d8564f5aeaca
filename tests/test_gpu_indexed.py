"""Row-subset (indexed) variants of the linear op against the plain path and the
FP64 oracle: duplicates count once, out-of-range indices are ignored, the
selected rows' log-probs are bitwise the plain forward's, unselected output
entries are left untouched, and gradients are those of the selected rows only
(grad_hidden zero elsewhere)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_helpers import (GH_ATOL, GH_RTOL, GW_ATOL, GW_RTOL, assert_close, check_device_status, np64,
                            oracle_args, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def _inputs(N=300, D=264, V=5000, seed=21):
    return workloads.make_inputs(N, D, V, seed=seed, weight_std=2.0 / math.sqrt(D), bias_std=0.3,
                                 temperature_range=(0.7, 1.3), n_ignore=5, n_out_of_range=2, grad_std=1.0)


def _selected(idx, N):
    return sorted({int(i) for i in idx if 0 <= int(i) < N})


INDEX_SETS = [
    [3, 17, 17, 299, -1, 300, 5000, 42, 3, 0],  # duplicates, negative, past the end
    list(range(0, 300, 7)) * 2,                 # every 7th row, each twice
    [150],
    [-5, 400],                                  # nothing valid
]


@pytest.mark.parametrize("idx_list", INDEX_SETS)
def test_indexed_forward(idx_list):
    import lm_head_selected_gb300 as llp
    inp = _inputs()
    d = to_device(inp)
    idx = torch.tensor(idx_list, dtype=torch.int64, device="cuda")
    full_lp, full_lse = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"])
    sentinel = 7.25
    lp = torch.full((inp.N,), sentinel, device="cuda")
    lse = torch.full((inp.N,), sentinel, device="cuda")
    llp.linear_logp_fwd_indexed(d["hidden"], d["weight"], d["targets"], idx, d["bias"], d["temperature"],
                                out=(lp, lse))
    check_device_status()
    sel = torch.tensor(_selected(idx_list, inp.N), dtype=torch.int64, device="cuda")
    mask = torch.zeros(inp.N, dtype=torch.bool, device="cuda")
    mask[sel] = True
    assert torch.equal(lp[mask], full_lp[mask]) and torch.equal(lse[mask], full_lse[mask])
    assert torch.all(lp[~mask] == sentinel) and torch.all(lse[~mask] == sentinel)


@pytest.mark.parametrize("idx_list", INDEX_SETS)
def test_indexed_backward(idx_list):
    import lm_head_selected_gb300 as llp
    inp = _inputs()
    d = to_device(inp)
    idx = torch.tensor(idx_list, dtype=torch.int64, device="cuda")
    _, lse = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"])
    gh, gw, gb = llp.linear_logp_bwd_indexed(d["grad_logp"], lse, d["hidden"], d["weight"], d["targets"], idx,
                                             d["bias"], d["temperature"])
    check_device_status()
    rows = _selected(idx_list, inp.N)
    a = oracle_args(inp)
    if rows:
        gh_ref, gw_ref, gb_ref = oracle.backward(np64(inp.grad_logp), *a, rows=rows)
    else:
        gh_ref = np.zeros((inp.N, inp.D))
        gw_ref = np.zeros((inp.V, inp.D))
        gb_ref = np.zeros(inp.V)
    assert_close("grad_hidden", np64(gh), gh_ref, GH_ATOL, GH_RTOL)
    assert_close("grad_weight", np64(gw), gw_ref, GW_ATOL, GW_RTOL)
    assert_close("grad_bias", np64(gb), gb_ref, GW_ATOL, GW_RTOL)
    unsel = np.setdiff1d(np.arange(inp.N), np.array(rows, dtype=np.int64))
    assert np.all(np64(gh)[unsel] == 0)


def test_indexed_empty_index_list():
    import lm_head_selected_gb300 as llp
    inp = _inputs(N=50, D=64, V=300)
    d = to_device(inp)
    idx = torch.empty(0, dtype=torch.int64, device="cuda")
    lp, lse = llp.linear_logp_fwd_indexed(d["hidden"], d["weight"], d["targets"], idx, d["bias"])
    assert torch.all(lp == 0) and torch.all(torch.isneginf(lse))
    _, lse_full = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"])
    gh, gw, gb = llp.linear_logp_bwd_indexed(d["grad_logp"], lse_full, d["hidden"], d["weight"], d["targets"], idx,
                                             d["bias"])
    assert torch.all(gh == 0) and torch.all(gw == 0) and torch.all(gb == 0)


def test_indexed_nemotron_head_subset():
    """Full Nemotron head size, 40 selected rows out of 512 (with repeats)."""
    import lm_head_selected_gb300 as llp
    inp = workloads.nemotron_head(N=512, seed=1001)
    d = to_device(inp)
    g = torch.Generator().manual_seed(4)
    idx_cpu = torch.randint(0, 512, (40,), generator=g)
    idx = torch.cat([idx_cpu, idx_cpu[:10]]).cuda()
    lp, lse = llp.linear_logp_fwd_indexed(d["hidden"], d["weight"], d["targets"], idx, None, d["temperature"])
    rows = _selected(idx.tolist(), 512)
    lp_ref, lse_ref = oracle.forward(*oracle_args(inp), rows=rows)
    assert_close("logp[rows]", np64(lp)[rows], lp_ref[rows], 5e-3, 0)
    full_lp, _ = llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], None, d["temperature"])
    r = torch.tensor(rows, device="cuda")
    assert torch.equal(lp[r], full_lp[r])
