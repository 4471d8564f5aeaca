"""Vocab-parallel orchestration across ranks, on CPU with gloo (world size 2 and 3).

``lm_head_selected_gb300.tp.linear_logp_vocab_parallel`` all-gathers the shard
triples and merges them in rank order, and sums the grad_hidden contributions
in rank order, either by a hand-made reduce-scatter (all_to_all of row blocks,
ordered sum, all_gather) or by all-gathering every contribution; the device
work is injected here as small float64 CPU functions of the same contract (a
shard's max / sum of exp / target logit; the rank-ordered merge; the shard's
dlogits contractions), so the collective logic, the rank order and the
autograd wiring are checked without a GPU, against the unsharded oracle, and
the two grad_hidden exchanges are checked to give the same bits."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _cpu_ops():
    from lm_head_selected_gb300.tp import ShardOps

    def logits(hidden, w, b, tau):
        z = hidden.double() @ w.double().T
        if b is not None:
            z = z + b.double()
        if tau is not None:
            z = z / tau.double()[:, None]
        return z

    def fwd_shard(hidden, w, targets, start, b, tau, ignore):
        z = logits(hidden, w, b, tau)
        m = z.max(1).values
        se = torch.exp(z - m[:, None]).sum(1)
        tl = targets - start
        local = (targets != ignore) & (tl >= 0) & (tl < w.shape[0])
        zt = torch.where(local, z.gather(1, tl.clamp(0, w.shape[0] - 1)[:, None]).squeeze(1),
                         torch.full_like(m, -math.inf))
        return torch.stack([m, se, zt])

    def merge(g, targets, global_v, ignore):
        m, se, zt = g[:, 0], g[:, 1], g[:, 2]
        M = m.max(0).values
        S = torch.zeros_like(M)
        for r in range(g.shape[0]):  # ascending rank order
            S = S + se[r] * torch.exp(m[r] - M)
        ZT = zt.max(0).values
        ok = (targets != ignore) & (targets >= 0) & (targets < global_v)
        lse = torch.where(ok, M + torch.log(S), torch.full_like(M, -math.inf))
        logp = torch.where(ok, ZT - M - torch.log(S), torch.zeros_like(M))
        return logp, lse

    def bwd_shard(g, lse, hidden, w, targets, start, global_v, b, tau, ignore, need_w, need_b):
        z = logits(hidden, w, b, tau)
        ok = (targets != ignore) & (targets >= 0) & (targets < global_v)
        inv_tau = torch.ones_like(lse) if tau is None else 1.0 / tau.double()
        p = torch.exp(z - torch.where(ok, lse, torch.zeros_like(lse))[:, None])
        tl = targets - start
        onehot = (tl[:, None] == torch.arange(w.shape[0])[None, :]).double()
        dz = torch.where(ok[:, None], (g.double() * inv_tau)[:, None] * (onehot - p), torch.zeros_like(p))
        return dz @ w.double(), dz.T @ hidden.double(), (dz.sum(0) if b is not None else None)

    def sum_partials(parts, dtype=None):  # kept in float64 here; dtype names the device path's rounding
        out = torch.zeros_like(parts[0])
        for r in range(parts.shape[0]):
            out = out + parts[r]
        return out

    return ShardOps(fwd_shard=fwd_shard, merge_shards=merge, bwd_shard=bwd_shard, sum_partials=sum_partials)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import workloads
    from lm_head_selected_gb300.tp import linear_logp_vocab_parallel
    inp = workloads.make_inputs(40, 16, 97, seed=9, weight_std=0.5, bias_std=0.3, temperature_range=(0.7, 1.3),
                                n_ignore=3, n_out_of_range=2, grad_std=1.0)
    V = inp.V
    cuts = [0, 30, 61, 97] if world == 3 else [0, 45, 97]
    s, e = cuts[rank], cuts[rank + 1]
    tau = inp.temperature.double()
    grads = {}
    for exchange in ("reduce_scatter", "gather"):
        h = inp.hidden.double().requires_grad_(True)
        w = inp.weight.double()[s:e].clone().requires_grad_(True)
        b = inp.bias.double()[s:e].clone().requires_grad_(True)
        logp = linear_logp_vocab_parallel(h, w, inp.targets, b, tau, vocab_start=s, global_vocab_size=V,
                                          ops=_cpu_ops(), grad_hidden_exchange=exchange)
        (logp * inp.grad_logp.double()).sum().backward()
        grads[exchange] = (logp.detach(), h.grad, w.grad, b.grad)
    same = all(torch.equal(x, y) for x, y in zip(grads["reduce_scatter"], grads["gather"]))
    a = (inp.hidden.double().numpy(), inp.weight.double().numpy(), inp.bias.double().numpy(), inp.targets.numpy(),
         inp.temperature.double().numpy(), -100)
    lp_ref, _ = oracle.forward(*a)
    gh_ref, gw_ref, gb_ref = oracle.backward(inp.grad_logp.double().numpy(), *a)
    err = max(np.abs(logp.detach().numpy() - lp_ref).max(), np.abs(h.grad.numpy() - gh_ref).max(),
              np.abs(w.grad.numpy() - gw_ref[s:e]).max(), np.abs(b.grad.numpy() - gb_ref[s:e]).max())
    dist.destroy_process_group()
    q.put((rank, float(err), same))


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_orchestration_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _, _ in res] == list(range(world))
    assert all(err < 1e-10 for _, err, _ in res), res
    # the reduce-scatter and the all-gather exchange give bitwise the same gradients
    assert all(same for _, _, same in res), res


def _sum_worker(rank, world, port, q):
    """rank_ordered_sum on fp32 contributions with the device path's rounding
    (fp32 sum in ascending rank order, one rounding to bf16), N not a multiple of
    the world size: both exchanges and a local recomputation agree bitwise."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from lm_head_selected_gb300.tp import ShardOps, rank_ordered_sum

    def sum_partials(parts, dtype):
        acc = parts[0].clone()
        for r in range(1, parts.shape[0]):
            acc = acc + parts[r]
        return acc.to(dtype)

    ops = ShardOps(sum_partials=sum_partials)
    N, D = 41, 24
    every = [torch.randn(N, D, generator=torch.Generator().manual_seed(50 + r)) * (10.0 ** r) for r in range(world)]
    out_rs = rank_ordered_sum(every[rank], None, torch.bfloat16, ops, "reduce_scatter")
    out_g = rank_ordered_sum(every[rank], None, torch.bfloat16, ops, "gather")
    local = sum_partials(torch.stack(every), torch.bfloat16)
    ok = (out_rs.dtype == torch.bfloat16 and out_rs.shape == (N, D) and torch.equal(out_rs, out_g)
          and torch.equal(out_rs, local))
    dist.destroy_process_group()
    q.put((rank, ok))


@pytest.mark.parametrize("world", [2, 3])
def test_rank_ordered_sum_exchanges_agree_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sum_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(r, True) for r in range(world)], res
