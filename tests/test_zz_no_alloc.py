"""The forward entry point that allocates nothing (linear_logp_fwd_noalloc).

It is meant for callers that cannot allocate device memory themselves, such as
a plugin inside a host program that owns every byte of device memory, or a
loop where cudaMalloc is not allowed.  Its scratch is a fixed 16 MiB array
inside the library, shared by every call.  These tests call it through the C
ABI and check that two calls in a row give bitwise the results of the regular
forward (which takes a caller workspace: the same kernels with the same
parameters, so nothing may differ), that sampled rows match the FP64 oracle,
that a problem too large for the array is refused before anything runs, and
that the array's leftover contents from a previous call do not leak into the
next one.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process too.
"""
import ctypes
import math

import pytest
import torch

import workloads
from parity_helpers import check_device_status, check_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from lm_head_selected_gb300 import _lib, build
    build.build()
    return _lib.load()


def _noalloc(lib, d, N, D, V):
    dev = d["hidden"].device
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.linear_logp_fwd_noalloc(p(d["hidden"]), p(d["weight"]), p(d["bias"]), p(d["targets"]),
                                     p(d["temperature"]), N, D, V, d["ignore_index"], p(logp), p(lse),
                                     ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    return st, logp, lse


def _regular(d):
    import lm_head_selected_gb300 as llp
    return llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"],
                               d["ignore_index"])


CASES = [
    # (N, D, V, bias, temperature): the Nemotron head near the scratch limit, then
    # smaller problems, so each call runs on the previous call's leftovers; the
    # last one a batch small enough for single-CTA tiles with 32-row hidden boxes.
    (4000, 2688, 131072, False, True),
    (333, 264, 50257, True, False),
    (20, 2688, 131072, True, True),
]


def test_two_calls_in_a_row_match_the_workspace_forward(lib):
    for i, (N, D, V, bias, temp) in enumerate(CASES):
        inp = workloads.make_inputs(N, D, V, seed=500 + i, weight_std=2.0 / math.sqrt(D),
                                    bias_std=0.3 if bias else None,
                                    temperature_range=(0.7, 1.3) if temp else None, n_ignore=7, n_out_of_range=3)
        d = to_device(inp)
        st, logp, lse = _noalloc(lib, d, N, D, V)
        assert st == 0, lib.linear_logp_status_string(st)
        ref_logp, ref_lse = _regular(d)
        check_device_status()
        # same kernels, same tiling, same fixed-order merge: bitwise equal, the
        # 0 / -inf of invalid rows included
        assert torch.equal(logp, ref_logp)
        assert torch.equal(lse, ref_lse)
        # and right, not merely consistent: sampled rows (ignored and out-of-range
        # ones among them) against the FP64 oracle
        bad = [int(r) for r in torch.nonzero(~torch.isfinite(ref_lse)).flatten()[:4].cpu()]
        g = torch.Generator().manual_seed(700 + i)
        rows = sorted(set(torch.randperm(N, generator=g)[:24].tolist()) | {0, N - 1} | set(bad))
        check_forward(inp, logp, lse, rows=rows)


def test_refuses_problems_beyond_the_scratch_limit(lib):
    from lm_head_selected_gb300 import _lib
    N, D, V = 9000, 2688, 131072  # needs about 18.5 MB > 16 MiB
    inp = workloads.make_inputs(N, D, 1024, seed=3)  # small weight: only the sizes matter here
    d = to_device(inp)
    w = torch.empty((V, D), dtype=torch.bfloat16, device="cuda")
    d["weight"] = w
    st, logp, lse = _noalloc(lib, d, N, D, V)
    assert st == _lib.LLP_ERR_SCRATCH_LIMIT
    assert torch.all(torch.isnan(logp)) and torch.all(torch.isnan(lse))  # nothing ran
