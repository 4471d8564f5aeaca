"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle,
element by element, on seeded inputs that span several tiles and ragged tails
in every dimension, plus the degenerate and invalid-target cases."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_helpers import (assert_close, check_backward, check_device_status, check_forward, gpu_bwd, gpu_fwd,
                            np64, oracle_args, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()
    torch.cuda.init()


def _roundtrip(inp, bwd=True, check_bwd=True):
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    check_device_status()
    check_forward(inp, logp, lse)
    if bwd:
        gh, gw, gb = gpu_bwd(d, lse)
        check_device_status()
        if check_bwd:
            check_backward(inp, gh, gw, gb)
        return logp, lse, gh, gw, gb
    return logp, lse


def test_tiny_forward_backward():
    _roundtrip(workloads.tiny())


SHAPES = [
    # N, D, V, bias, temperature, n_ignore, n_out_of_range
    (200, 136, 1000, True, True, 3, 2),   # ragged M, K tail (136 = 2*64 + 8), V not a multiple of 8
    (129, 64, 257, False, True, 1, 0),    # one row / one column past a tile
    (1, 8, 1, True, False, 0, 0),         # single token, minimal D, single-token vocab
    (300, 256, 50257, True, False, 5, 0),  # GPT-2 vocab (odd)
    (64, 128, 32832, False, False, 0, 0),  # two vocab K segments [32768, 64]
    (96, 2688, 4096, True, True, 2, 1),   # full Nemotron hidden size, 42 k-blocks
    (257, 512, 2048, False, True, 0, 0),  # three M tiles, the last with one row
    (33, 64, 131073, False, True, 1, 0),  # 257 vocab splits: the split merge takes a second round of one split
    (40, 64, 200000, True, False, 2, 1),  # 391 vocab splits, ragged last split
    # >= 1024 tokens: grad_weight takes two k-blocks per stage; D = 3 x 64 is an odd number of 64-column
    # chunks, so a copy's second chunk of hidden runs past D (read as zeros)
    (16, 2688, 33000, True, True, 2, 1),  # small batch: single-CTA tiles with 32-row hidden boxes
    (1100, 192, 3000, True, True, 3, 1),
    (1030, 200, 2500, False, True, 2, 0),  # D not a multiple of 64: every GEMM on one k-block per stage, 2-D maps
]


@pytest.mark.parametrize("N,D,V,bias,temp,n_ign,n_oor", SHAPES)
def test_ragged_shapes(N, D, V, bias, temp, n_ign, n_oor):
    inp = workloads.make_inputs(N, D, V, seed=N * 7 + V, hidden_std=1.0, weight_std=2.0 / math.sqrt(D),
                                bias_std=0.5 if bias else None,
                                temperature_range=(0.7, 1.3) if temp else None,
                                n_ignore=n_ign, n_out_of_range=n_oor, grad_std=1.0)
    _roundtrip(inp)


def test_nemotron_head_n32():
    """Batch 2 x seq 16 on the Nemotron head: D=2688, V=131072, per-row temperature."""
    _roundtrip(workloads.nemotron_head(N=32))


@pytest.mark.parametrize("N,segments", [(32768, 1), (32769, 2), (65600, 3)])
def test_grad_weight_token_segments(N, segments):
    """grad_weight reduces over tokens in fixed 32768-token segments ([32768],
    [32768, 1], [32768, 32768, 64]), the cases of "Feat/nemotron h lm head
    logprob cuda" (det-GEMM split verification)."""
    assert math.ceil(N / 32768) == segments
    inp = workloads.make_inputs(N, 64, 320, seed=N, hidden_std=1.0, weight_std=0.25, bias_std=0.1,
                                n_ignore=17, grad_std=1.0)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, gb = gpu_bwd(d, lse, need_hidden=False)
    check_device_status()
    check_forward(inp, logp, lse)
    check_backward(inp, None, gw, gb)
    # bitwise reproducible across two runs
    gh2, gw2, gb2 = gpu_bwd(d, lse, need_hidden=False)
    assert torch.equal(gw, gw2) and torch.equal(gb, gb2)


def test_all_rows_ignored():
    inp = workloads.make_inputs(70, 64, 300, seed=3, bias_std=0.3, grad_std=1.0)
    inp.targets[:] = -100
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    assert torch.all(logp == 0) and torch.all(torch.isneginf(lse))
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    assert torch.all(gh == 0) and torch.all(gw == 0) and torch.all(gb == 0)


def test_nan_upstream_gradient_on_ignored_rows_does_not_leak():
    inp = workloads.make_inputs(50, 64, 300, seed=4, bias_std=0.3, n_ignore=6, n_out_of_range=4, grad_std=1.0)
    bad = ~torch.as_tensor(oracle.valid_rows(inp.targets.numpy(), inp.V, -100))
    inp.grad_logp[bad] = float("nan")
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    assert torch.all(torch.isfinite(gh.float())) and torch.all(torch.isfinite(gw.float()))
    assert torch.all(gh[bad.cuda()] == 0)
    inp.grad_logp[bad] = 0.0
    check_backward(inp, gh, gw, gb)


def test_empty_batch():
    inp = workloads.make_inputs(0, 64, 300, seed=5, bias_std=0.3, grad_std=1.0)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    assert logp.numel() == 0 and lse.numel() == 0
    gh, gw, gb = gpu_bwd(d, lse)
    assert gh.numel() == 0
    assert torch.all(gw == 0) and torch.all(gb == 0)


def test_constant_logit_shift_row():
    """Row 0's logits lifted by exactly 9984 (the long-context stress row) at small size."""
    inp = workloads.long_context(N=130, D=64, V=300, seed=11)
    inp.grad_logp = torch.randn(inp.N, generator=torch.Generator().manual_seed(1))
    logp, lse, gh, gw, gb = _roundtrip(inp)
    ref = inp.rows(torch.arange(inp.N))
    ref.hidden[0, -1] = 0.0
    d0 = to_device(ref)
    logp0, _ = gpu_fwd(d0)
    assert abs(float(logp[0]) - float(logp0[0])) < 5e-3


def test_autograd_leading_shape():
    """The leading-shape interface: [3, 100] tokens, gradients into hidden, weight, bias."""
    import lm_head_selected_gb300 as llp
    inp = workloads.make_inputs(300, 128, 1000, seed=9, weight_std=0.2, bias_std=0.2, n_ignore=5, grad_std=1.0)
    d = to_device(inp)
    h = d["hidden"].view(3, 100, 128).clone().requires_grad_(True)
    w = d["weight"].clone().requires_grad_(True)
    b = d["bias"].clone().requires_grad_(True)
    t = d["targets"].view(3, 100)
    out = llp.linear_logp(h, w, t, b)
    assert out.shape == (3, 100) and out.dtype == torch.float32
    (out * d["grad_logp"].view(3, 100)).sum().backward()
    logp, lse = gpu_fwd(d)
    assert torch.equal(out.detach().reshape(-1), logp)
    gh, gw, gb = gpu_bwd(d, lse)
    assert torch.equal(h.grad.reshape(300, 128), gh)
    assert torch.equal(w.grad, gw)
    assert torch.equal(b.grad, gb)


def test_bias_at_unaligned_offset():
    """A bias that starts one float into its buffer (a vocab shard's slice): scalar bias loads, same results."""
    inp = workloads.make_inputs(150, 128, 1300, seed=21, weight_std=0.2, bias_std=0.4, n_ignore=2, grad_std=1.0)
    d = to_device(inp)
    buf = torch.zeros(inp.V + 1, dtype=torch.float32, device=d["bias"].device)
    buf[1:] = d["bias"]
    d["bias"] = buf[1:]
    assert d["bias"].data_ptr() % 16 != 0
    logp, lse = gpu_fwd(d)
    check_device_status()
    check_forward(inp, logp, lse)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    check_backward(inp, gh, gw, gb)


def test_call_from_a_fresh_thread():
    """A thread whose first CUDA work is this library's call (no context bound on
    it yet; an autograd worker whose tensors come from the allocator's cache is one)
    gets the same results as the main thread."""
    import threading

    import lm_head_selected_gb300 as llp
    inp = workloads.make_inputs(64, 256, 4096, seed=3, weight_std=0.125, bias_std=0.1, n_ignore=4, grad_std=1.0)
    d = to_device(inp)
    logp0, lse0 = gpu_fwd(d)
    gh0, gw0, gb0 = gpu_bwd(d, lse0)
    logp = torch.empty_like(logp0)
    lse = torch.empty_like(lse0)
    ws_f = torch.empty(llp.fwd_workspace_bytes(inp.N, inp.D, inp.V), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(llp.bwd_workspace_bytes(inp.N, inp.D, inp.V, True), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    out, err = {}, []

    def work():
        try:
            llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], None, workspace=ws_f, out=(logp, lse))
            out["g"] = llp.linear_logp_bwd(d["grad_logp"], lse, d["hidden"], d["weight"], d["targets"], d["bias"],
                                           workspace=ws_b)
            torch.cuda.synchronize()
        except Exception as e:  # reported in the main thread
            err.append(e)

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert not err, err
    check_device_status()
    gh, gw, gb = out["g"]
    assert torch.equal(logp, logp0) and torch.equal(lse, lse0)
    assert torch.equal(gh, gh0) and torch.equal(gw, gw0) and torch.equal(gb, gb0)


def test_concurrent_threads_on_their_own_streams():
    """Four host threads, each with its own CUDA stream and its own problem, run
    forward + backward at the same time; each gets exactly what it gets alone (the
    entry points share no per-call state)."""
    import threading

    import lm_head_selected_gb300 as llp
    shapes = [(300, 256, 5000, 11), (64, 512, 4096, 12), (129, 136, 1000, 13), (32, 2688, 131072, 14)]
    probs, alone = [], []
    for N, D, V, seed in shapes:
        inp = workloads.make_inputs(N, D, V, seed=seed, weight_std=2.0 / math.sqrt(D), bias_std=0.2,
                                    temperature_range=(0.8, 1.2), n_ignore=2, grad_std=1.0)
        d = to_device(inp)
        lp, ls = gpu_fwd(d)
        alone.append((lp, ls) + tuple(gpu_bwd(d, ls)))
        probs.append(d)
    torch.cuda.synchronize()
    results, errors = [None] * len(probs), []
    start = threading.Barrier(len(probs))

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                start.wait()
                for _ in range(3):
                    lp, ls = gpu_fwd(probs[i])
                    out = (lp, ls) + tuple(gpu_bwd(probs[i], ls))
            s.synchronize()
            results[i] = out
        except Exception as e:  # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(probs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    check_device_status()
    for got, ref in zip(results, alone):
        for a, b in zip(got, ref):
            assert (a is None and b is None) or torch.equal(a, b)
