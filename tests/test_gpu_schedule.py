"""The work schedule never changes a result: the gradient GEMMs' in-order unit
claiming (used when units span >= 128 k-blocks) and round-robin assignment
(forced with LINEAR_LOGP_SCHEDULE=static, read once per process, so that run
happens in a child process) give bitwise identical outputs."""
import os
import subprocess
import sys

import pytest
import torch

import workloads
from parity_helpers import check_device_status, gpu_bwd, gpu_fwd, to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# N = 8192 tokens and V = 16384: both gradient GEMMs have 128+ k-block units
CASE = dict(N=8192, D=128, V=16384, seed=41)

CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import workloads
from parity_helpers import check_device_status, gpu_bwd, gpu_fwd, to_device
inp = workloads.make_inputs({N}, {D}, {V}, seed={seed}, weight_std=0.1, bias_std=0.2, n_ignore=9, grad_std=1.0)
d = to_device(inp)
logp, lse = gpu_fwd(d)
gh, gw, gb = gpu_bwd(d, lse)
check_device_status()
torch.save({{"logp": logp.cpu(), "gh": gh.cpu(), "gw": gw.cpu(), "gb": gb.cpu()}}, {out!r})
"""


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def test_in_order_and_round_robin_schedules_agree_bitwise(tmp_path):
    out = str(tmp_path / "static.pt")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), out=out, **CASE)
    env = dict(os.environ, LINEAR_LOGP_SCHEDULE="static")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    ref = torch.load(out)

    inp = workloads.make_inputs(CASE["N"], CASE["D"], CASE["V"], seed=CASE["seed"], weight_std=0.1, bias_std=0.2,
                                n_ignore=9, grad_std=1.0)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, gw, gb = gpu_bwd(d, lse)
    check_device_status()
    assert os.environ.get("LINEAR_LOGP_SCHEDULE") != "static"
    assert torch.equal(logp.cpu(), ref["logp"])
    assert torch.equal(gh.cpu(), ref["gh"]), "grad_hidden depends on the schedule"
    assert torch.equal(gw.cpu(), ref["gw"]), "grad_weight depends on the schedule"
    assert torch.equal(gb.cpu(), ref["gb"])


# grad_hidden of batches of at most 96 rows runs on the swapped-operand kernel
# (hidden on the MMA's M side, tokens on N); LINEAR_LOGP_SMALL_GRAD_HIDDEN=0 (read
# once per process) sends them through the CTA-pair GEMM.  Both accumulate every
# element over the same 16-wide vocab slices in the same order.
SMALL_CASES = [
    # (N, D, V, bias, temperature, fp16)
    (32, 2688, 131072, False, True, False),   # the Nemotron head at batch 2 x seq 16
    (17, 264, 50257, True, True, False),      # D not a multiple of 128, V not a multiple of 64
    (96, 512, 33000, False, False, False),    # the largest batch the kernel takes (two dz slots, two weight stages)
    (128, 512, 33000, False, False, False),   # above it: both processes run the CTA-pair GEMM
    (100, 256, 40000, True, False, True),     # fp16 inputs
    (1, 128, 70000, False, False, False),     # a single token, three vocab segments
]

SMALL_CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import workloads
from parity_helpers import check_device_status, gpu_bwd, gpu_fwd, to_device
from lm_head_selected_gb300 import tp
out = {{}}
for i, (N, D, V, bias, temp, f16) in enumerate({cases!r}):
    inp = workloads.make_inputs(N, D, V, seed=300 + i, weight_std=0.05, bias_std=0.2 if bias else None,
                                temperature_range=(0.7, 1.3) if temp else None, n_ignore=min(3, N - 1),
                                grad_std=1.0, dtype=torch.float16 if f16 else torch.bfloat16)
    d = to_device(inp)
    logp, lse = gpu_fwd(d)
    gh, _, _ = gpu_bwd(d, lse, need_weight=False)
    out["gh%d" % i] = gh.cpu()
    if i == 2:  # a vocab shard's fp32 contribution (the first half of the vocabulary)
        part, _, _ = tp.bwd_shard(d["grad_logp"], lse, d["hidden"], d["weight"][: V // 2], d["targets"], 0, V,
                                  None, d["temperature"], need_weight=False)
        out["part"] = part.cpu()
check_device_status()
torch.save(out, {out_path!r})
"""


def test_small_batch_grad_hidden_kernel_matches_pair_gemm_bitwise(tmp_path):
    out_path = str(tmp_path / "pair.pt")
    code = SMALL_CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), cases=SMALL_CASES, out_path=out_path)
    env = dict(os.environ, LINEAR_LOGP_SMALL_GRAD_HIDDEN="0")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    ref = torch.load(out_path)
    # this process runs the swapped-operand kernel (the default)
    assert os.environ.get("LINEAR_LOGP_SMALL_GRAD_HIDDEN") != "0"
    out_path2 = str(tmp_path / "small.pt")
    code2 = SMALL_CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), cases=SMALL_CASES, out_path=out_path2)
    r2 = subprocess.run([sys.executable, "-c", code2], capture_output=True, text=True, timeout=600,
                        env={k: v for k, v in os.environ.items() if k != "LINEAR_LOGP_SMALL_GRAD_HIDDEN"})
    assert r2.returncode == 0, r2.stderr[-3000:]
    got = torch.load(out_path2)
    assert set(got) == set(ref)
    for k in sorted(ref):
        assert torch.equal(got[k], ref[k]), f"{k}: the two grad_hidden forms differ"
        assert torch.isfinite(got[k].float()).all()
