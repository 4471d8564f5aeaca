"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The path runs as independent replicas (one per GPU, no exchange): the only
cross-rank steps are the barriers around the timed region and the max over
ranks of the elapsed time.  These run here with the gloo backend."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist.barrier()
    mx = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx))


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(r, 10.0 + 5.0 * (world - 1)) for r in range(world)]


def test_reference_arm_skips_non_zero_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
