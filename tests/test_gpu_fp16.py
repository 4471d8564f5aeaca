"""fp16 inputs ("Fused Linear LogP", Tensor Contract: hidden and lm_head_weight
may be bf16 or fp16): the fp16 entry points against the FP64 oracle on seeded
fp16 problems (fp16 converts exactly to float64), with the same tolerances as
the bf16 path, plus the autograd op and the dtype checks of the wrapper."""
import math

import pytest
import torch

import workloads
from parity_helpers import (check_backward, check_device_status, check_forward, gpu_bwd, gpu_fwd, np64,
                            to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


SHAPES = [
    # N, D, V, bias, temperature
    (200, 136, 1000, True, True),      # ragged M, K tail, V not a multiple of 8
    (257, 512, 2048, False, True),     # three M tiles, the last with one row
    (96, 2688, 4096, True, False),     # full Nemotron hidden size
    (64, 128, 32832, False, False),    # two vocab K segments of grad_hidden
    (20, 256, 5000, True, True),       # small batch: single-CTA tiles with 32-row hidden boxes
]


@pytest.mark.parametrize("N,D,V,bias,temp", SHAPES)
def test_fp16_forward_backward_match_oracle(N, D, V, bias, temp):
    inp = workloads.make_inputs(N, D, V, seed=700 + N, weight_std=2.0 / math.sqrt(D),
                                bias_std=0.4 if bias else None, temperature_range=(0.7, 1.3) if temp else None,
                                n_ignore=3, n_out_of_range=2, grad_std=1.0, dtype=torch.float16)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    check_device_status()
    check_forward(inp, logp, lse)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    assert gh.dtype == torch.float16 and gw.dtype == torch.float16
    check_backward(inp, gh, gw, gb)


def test_fp16_grad_weight_token_segments():
    """N > 32768: grad_weight sums two fixed token segments into an fp16 result."""
    inp = workloads.make_inputs(32769, 64, 384, seed=77, weight_std=0.25, n_ignore=5, grad_std=1.0,
                                dtype=torch.float16)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    check_forward(inp, logp, lse, rows=list(range(0, inp.N, 997)))
    check_backward(inp, gh, gw, gb)


def test_fp16_matches_bf16_path_on_bf16_exact_values():
    """Values that both formats hold exactly (small integers times powers of two)
    give the same logp through either entry point: only the operand type differs."""
    g = torch.Generator().manual_seed(3)
    N, D, V = 130, 64, 700
    h = (torch.randint(-8, 9, (N, D), generator=g).float() / 8)
    w = (torch.randint(-8, 9, (V, D), generator=g).float() / 64)
    t = torch.randint(0, V, (N,), generator=g)
    import lm_head_selected_gb300 as llp
    lp16, lse16 = llp.linear_logp_fwd(h.half().cuda(), w.half().cuda(), t.cuda())
    lpbf, lsebf = llp.linear_logp_fwd(h.bfloat16().cuda(), w.bfloat16().cuda(), t.cuda())
    assert torch.equal(lp16, lpbf) and torch.equal(lse16, lsebf)


def test_fp16_autograd_op():
    import lm_head_selected_gb300 as llp
    inp = workloads.make_inputs(300, 128, 1000, seed=9, weight_std=0.2, bias_std=0.2, n_ignore=5, grad_std=1.0,
                                dtype=torch.float16)
    d = to_device(inp)
    h = d["hidden"].view(3, 100, 128).clone().requires_grad_(True)
    w = d["weight"].clone().requires_grad_(True)
    b = d["bias"].clone().requires_grad_(True)
    out = llp.linear_logp(h, w, d["targets"].view(3, 100), b)
    (out * d["grad_logp"].view(3, 100)).sum().backward()
    assert h.grad.dtype == torch.float16 and w.grad.dtype == torch.float16 and b.grad.dtype == torch.float32
    check_forward(inp, out.detach().reshape(-1), gpu_fwd(d)[1])
    check_backward(inp, h.grad.reshape(300, 128), w.grad, b.grad)


def test_mixed_or_fp32_inputs_are_refused():
    import lm_head_selected_gb300 as llp
    h = torch.zeros(4, 64, device="cuda", dtype=torch.float16)
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(TypeError):
        llp.linear_logp_fwd(h, torch.zeros(10, 64, device="cuda", dtype=torch.bfloat16), t)
    with pytest.raises(TypeError):
        llp.linear_logp_fwd(h.float(), torch.zeros(10, 64, device="cuda"), t)
    with pytest.raises(TypeError):  # the no-allocation forward stays bf16-only
        llp.ops.linear_logp_fwd_noalloc(h, torch.zeros(10, 64, device="cuda", dtype=torch.float16), t)


def test_fp16_row_subsets():
    """fp16 row-subset forward gives the plain fp16 forward's values on the selected
    rows; its backward matches the oracle restricted to those rows."""
    import numpy as np

    import lm_head_selected_gb300 as llp
    import oracle
    from parity_helpers import GH_ATOL, GH_RTOL, GW_ATOL, GW_RTOL, assert_close, oracle_args
    inp = workloads.make_inputs(300, 192, 1500, seed=23, weight_std=0.15, bias_std=0.3, n_ignore=4, grad_std=1.0,
                                dtype=torch.float16)
    d = to_device(inp)
    idx = torch.tensor([5, 17, 17, 250, 299, 0, 1000, -3], dtype=torch.int64, device="cuda")
    rows = sorted({5, 17, 250, 299, 0})
    lp_all, lse_all = gpu_fwd(d)
    lp, lse = llp.linear_logp_fwd_indexed(d["hidden"], d["weight"], d["targets"], idx, d["bias"])
    r = torch.tensor(rows, device="cuda")
    assert torch.equal(lp[r], lp_all[r]) and torch.equal(lse[r], lse_all[r])
    gh, gw, gb = llp.linear_logp_bwd_indexed(d["grad_logp"], lse_all, d["hidden"], d["weight"], d["targets"], idx,
                                             d["bias"])
    check_device_status()
    assert gh.dtype == torch.float16 and gw.dtype == torch.float16
    sub = inp.rows(torch.tensor(rows))
    gh_ref, gw_ref, gb_ref = oracle.backward(np64(sub.grad_logp), *oracle_args(sub))
    assert_close("grad_hidden[rows]", np64(gh)[rows], gh_ref, GH_ATOL, GH_RTOL)
    others = np.setdiff1d(np.arange(inp.N), rows)
    assert np.all(np64(gh)[others] == 0)
    assert_close("grad_weight", np64(gw), gw_ref, GW_ATOL, GW_RTOL)
    assert_close("grad_bias", np64(gb), gb_ref, GW_ATOL, GW_RTOL)
