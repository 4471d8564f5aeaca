"""GPU parity of the logits-input fused log-prob (include/fused_logp.h) against
its FP64 oracle, for bf16 and fp32 logits: ragged vocab sizes (vectorised and
scalar paths, split tails), invalid targets, a +1e4 shifted row, batch
invariance, repeatability and the autograd wrapper."""
import math

import numpy as np
import pytest
import torch

from oracle import logits_logp as lo

pytestmark = pytest.mark.gpu

LOGP_ATOL = 5e-3
# grad atol, rtol (16-bit types: one output rounding)
TOL = {torch.float32: (1e-5, 1e-4), torch.bfloat16: (1e-3, 1e-2), torch.float16: (1e-4, 2e-3)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lm_head_selected_gb300 import build
    build.build()


def _problem(N, V, dtype, seed, shift_row=None):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(N, V, generator=g) * 3.0
    if shift_row is not None and N > shift_row:
        z[shift_row] += 1e4
    z = z.to(dtype)
    t = torch.randint(0, V, (N,), generator=g)
    if N >= 4:
        t[1] = -100
        t[3] = V + 7
    gl = torch.randn(N, generator=g)
    return z, t, gl


def _close(name, got, ref, atol, rtol):
    got = got.double().cpu().numpy()
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{name}: {bad.sum()} bad, max err {err.max():.3e}"


def _check(z, t, gl):
    import lm_head_selected_gb300 as llp
    zd, td, gd = z.cuda(), t.cuda(), gl.cuda()
    logp, m, ls = llp.fused_logp_fwd(zd, td)
    grad = llp.fused_logp_bwd(gd, m, ls, zd, td)
    torch.cuda.synchronize()
    zn = z.double().numpy()
    lp_ref, m_ref, ls_ref = lo.forward(zn, t.numpy())
    ok = lo.valid_rows(t.numpy(), z.shape[1], -100)
    _close("logp", logp, lp_ref, LOGP_ATOL, 0)
    assert np.array_equal(m.cpu().double().numpy()[ok], m_ref[ok])  # the max of the given values is exact
    _close("log_sum", ls[torch.as_tensor(ok).cuda()], ls_ref[ok], 1e-4, 0)
    assert torch.all(torch.isneginf(m[torch.as_tensor(~ok).cuda()]))
    assert torch.all(logp[torch.as_tensor(~ok).cuda()] == 0)
    atol, rtol = TOL[z.dtype]
    g_ref = lo.backward(gl.double().numpy(), zn, t.numpy())
    _close("grad_logits", grad, g_ref, atol, rtol)
    assert grad.dtype == z.dtype
    return logp, m, ls, grad


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("N,V", [(64, 4096), (37, 50257), (5, 131072), (300, 16385), (1, 1), (130, 32768)])
def test_parity(dtype, N, V):
    z, t, gl = _problem(N, V, dtype, seed=N + V, shift_row=0 if dtype == torch.float32 else None)
    _check(z, t, gl)


def test_shifted_row_bf16():
    """A bf16 row lifted by about 1e4 (the values themselves round to bf16's spacing
    of 64 there): parity with the oracle on those exact inputs, and row_max near 1e4."""
    z, t, gl = _problem(8, 3000, torch.float32, seed=3)
    zs = z.clone()
    zs[2] += 1e4
    zs = zs.to(torch.bfloat16)
    import lm_head_selected_gb300 as llp
    _, m, _ = llp.fused_logp_fwd(zs.cuda(), t.cuda())
    _check(zs, t, gl)
    assert 9900 < float(m[2]) < 10100


def test_batch_invariance_and_repeatability():
    import lm_head_selected_gb300 as llp
    z, t, gl = _problem(257, 131072, torch.bfloat16, seed=11)
    zd, td = z.cuda(), t.cuda()
    lp, m, ls = llp.fused_logp_fwd(zd, td)
    for size in (1, 7, 64):
        idx = torch.randperm(257, generator=torch.Generator().manual_seed(size))[:size]
        lps, ms, lss = llp.fused_logp_fwd(zd[idx.cuda()].contiguous(), td[idx.cuda()].contiguous())
        assert torch.equal(lps, lp[idx.cuda()]) and torch.equal(lss, ls[idx.cuda()])
    lp2, m2, ls2 = llp.fused_logp_fwd(zd, td)
    assert torch.equal(lp, lp2) and torch.equal(ls, ls2)
    g1 = llp.fused_logp_bwd(gl.cuda(), m, ls, zd, td)
    g2 = llp.fused_logp_bwd(gl.cuda(), m, ls, zd, td)
    assert torch.equal(g1, g2)


def test_autograd_leading_shape():
    import lm_head_selected_gb300 as llp
    z, t, gl = _problem(60, 1000, torch.float32, seed=5)
    zd = z.cuda().view(3, 20, 1000).clone().requires_grad_(True)
    out = llp.fused_logp(zd, t.cuda().view(3, 20))
    assert out.shape == (3, 20)
    (out * gl.cuda().view(3, 20)).sum().backward()
    g_ref = lo.backward(gl.double().numpy(), z.double().numpy(), t.numpy())
    _close("grad via autograd", zd.grad.reshape(60, 1000), g_ref, 1e-5, 1e-4)
    assert math.isfinite(float(out.detach().sum()))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_indexed_rows(dtype):
    """Row subsets ("recursive deterministic LogP autograd on B200", Indexed semantics):
    selected rows equal the dense op bitwise, other outputs stay untouched, and the
    gradient rows not selected are zero."""
    import lm_head_selected_gb300 as llp
    z, t, gl = _problem(70, 20000, dtype, seed=21)
    zd, td, gd = z.cuda(), t.cuda(), gl.cuda()
    lp0, m0, ls0 = llp.fused_logp_fwd(zd, td)
    g0 = llp.fused_logp_bwd(gd, m0, ls0, zd, td)
    idx = torch.tensor([3, 9, 9, 69, 0, 70, -1, 1], dtype=torch.int64, device="cuda")
    rows = sorted({3, 9, 69, 0, 1})
    sentinel = torch.full((70,), 123.0, device="cuda")
    out = (sentinel.clone(), sentinel.clone(), sentinel.clone())
    lp, m, ls = llp.fused_logp_fwd_indexed(zd, td, idx, out=out)
    r = torch.tensor(rows, device="cuda")
    assert torch.equal(lp[r], lp0[r]) and torch.equal(m[r], m0[r]) and torch.equal(ls[r], ls0[r])
    others = torch.tensor(sorted(set(range(70)) - set(rows)), device="cuda")
    assert torch.all(lp[others] == 123.0) and torch.all(m[others] == 123.0)
    g = llp.fused_logp_bwd_indexed(gd, m0, ls0, zd, td, idx)
    assert torch.equal(g[r], g0[r])
    assert torch.all(g[others] == 0)
    g_none = llp.fused_logp_bwd_indexed(gd, m0, ls0, zd, td, idx[:0])
    assert torch.all(g_none == 0)


def test_full_size_benchmark_problem():
    """The benchmark's problem and launch configuration (N=16384, V=131072, bf16
    logits drawn as ``bench.py --op fused_logp`` draws them, plus ignored rows):
    every row valid, sampled rows against the oracle, bitwise repeatable."""
    import lm_head_selected_gb300 as llp
    N, V = 16384, 131072
    g = torch.Generator().manual_seed(1005)
    z = (torch.randn(N, V, generator=g) * 3.0).to(torch.bfloat16)
    t = torch.randint(0, V, (N,), generator=g)
    gl = torch.randn(N, generator=g)
    t[::97] = -100
    zd, td, gd = z.cuda(), t.cuda(), gl.cuda()
    logp, m, ls = llp.fused_logp_fwd(zd, td)
    grad = llp.fused_logp_bwd(gd, m, ls, zd, td)
    ok = torch.as_tensor(lo.valid_rows(t.numpy(), V, -100)).cuda()
    assert torch.all(torch.isfinite(logp)) and torch.all(logp[ok] <= 0) and torch.all(logp[~ok] == 0)
    assert torch.all(torch.isfinite(ls[ok])) and torch.all(torch.isneginf(m[~ok]))
    assert torch.all(grad[~ok] == 0)
    rows = sorted(set(torch.randperm(N, generator=torch.Generator().manual_seed(9))[:64].tolist()) | {0, 97, N - 1})
    r = torch.tensor(rows)
    zr, tr = z[r].double().numpy(), t[r].numpy()
    lp_ref, m_ref, ls_ref = lo.forward(zr, tr)
    okr = lo.valid_rows(tr, V, -100)
    rd = r.cuda()
    _close("logp[rows]", logp[rd], lp_ref, LOGP_ATOL, 0)
    assert np.array_equal(m[rd].cpu().double().numpy()[okr], m_ref[okr])
    _close("log_sum[rows]", ls[rd][torch.as_tensor(okr).cuda()], ls_ref[okr], 1e-4, 0)
    _close("grad_logits[rows]", grad[rd], lo.backward(gl[r].double().numpy(), zr, tr), *TOL[torch.bfloat16])
    logp2, m2, ls2 = llp.fused_logp_fwd(zd, td)
    assert torch.equal(logp, logp2) and torch.equal(m, m2) and torch.equal(ls, ls2)
    assert torch.equal(grad, llp.fused_logp_bwd(gd, m, ls, zd, td))
