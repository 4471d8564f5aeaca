"""The CUDA path under CUDA graph capture.

Every entry point only enqueues work on the caller's stream: no host
synchronisation and no allocation inside the library, with the workspace passed
in.  A forward + backward step can therefore be captured into a CUDA graph and
replayed.  A replay must give the eager path's results bitwise, also after the
step's inputs are overwritten in place with another batch."""
import dataclasses
import math

import pytest
import torch

import workloads
from parity_helpers import check_device_status, gpu_bwd, gpu_fwd, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def _batches(N, D, V, bias, temp):
    kw = dict(weight_std=2.0 / math.sqrt(D), bias_std=0.2 if bias else None,
              temperature_range=(0.8, 1.2) if temp else None, n_ignore=3, n_out_of_range=1, grad_std=1.0)
    a = workloads.make_inputs(N, D, V, seed=4100 + N, **kw)
    b = workloads.make_inputs(N, D, V, seed=4200 + N, **kw)
    # the same head: a second batch of tokens through the first batch's weight and bias
    return a, dataclasses.replace(b, weight=a.weight, bias=a.bias)


@pytest.mark.parametrize("N,D,V,bias,temp", [(300, 256, 5000, True, True),    # CTA-pair tiles
                                             (32, 2688, 131072, False, True)])  # single-CTA tiles
def test_graph_replay_matches_eager(N, D, V, bias, temp):
    import lm_head_selected_gb300 as llp
    first, second = _batches(N, D, V, bias, temp)
    d = to_device(first)
    ws_f = torch.empty(llp.fwd_workspace_bytes(N, D, V), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(llp.bwd_workspace_bytes(N, D, V, bias), dtype=torch.uint8, device="cuda")
    logp = torch.empty(N, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")

    def step():
        llp.linear_logp_fwd(d["hidden"], d["weight"], d["targets"], d["bias"], d["temperature"],
                            d["ignore_index"], workspace=ws_f, out=(logp, lse))
        return llp.linear_logp_bwd(d["grad_logp"], lse, d["hidden"], d["weight"], d["targets"], d["bias"],
                                   d["temperature"], d["ignore_index"], workspace=ws_b)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # first call outside the capture: one-time device set-up
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gh, gw, gb = step()

    for batch in (second, first):
        ref = to_device(batch)
        for k in ("hidden", "targets", "temperature", "grad_logp"):
            if d[k] is not None:
                d[k].copy_(ref[k])
        graph.replay()
        torch.cuda.synchronize()
        lp_e, lse_e = gpu_fwd(ref)
        gh_e, gw_e, gb_e = gpu_bwd(ref, lse_e)
        assert torch.equal(logp, lp_e) and torch.equal(lse, lse_e)
        assert torch.equal(gh, gh_e) and torch.equal(gw, gw_e)
        assert (gb is None and gb_e is None) or torch.equal(gb, gb_e)
    check_device_status()
