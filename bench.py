#!/usr/bin/env python
"""Benchmark of the fused linear selected-token log-probability on GB300.

One step = one pass of the whole hot path over one batch: the forward (vocab
split partials + fixed-order merge) and the backward (dlogits recompute,
grad_hidden, grad_weight and their fixed-order segment sums) through the C ABI.

Default workload: the RL-scoring / training head of the pages' Nemotron-3-Nano
shape, N=16384 tokens (batch 32 x seq 512), D=2688, V=131072, bf16, no bias,
tau = 1, grad_logp ~ N(0,1), inputs resident in HBM.  W (704.6 MB) is larger
than the 129 MB L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (launched with torch.distributed.run) every rank runs an independent
replica of the same workload on its own GPU (the path needs no exchange) and
the value is the total tokens of all ranks over the slowest rank's time.
``--impl reference`` times the FP64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd+bwd tokens/s and % bf16 tensor peak at D=2688 V=131072 (1 GB300)"
UNIT = "tokens/s"
WORKLOADS = {
    # name: (N, D, V, description)
    "rl_head_fwd_bwd": (16384, 2688, 131072,
                        "Nemotron-3-Nano LM head, N=16384 (32x512), D=2688, V=131072, no bias, tau=1, "
                        "85% planted high-probability / 10% uniform / 5% ignored targets, grad_logp~N(0,1)"),
    # smaller token count of the same head, for profiler captures (weight still > L2)
    "rl_head_small": (2048, 2688, 131072,
                      "same head and distributions with N=2048 (for profiler captures)"),
}
# The pages' number for this metric and workload: strict fused fwd+bwd, 16384 tokens,
# D=2688, V=131072, 351.2 ms on an H100 PCIe ("Feat/nemotron h lm head logprob cuda",
# Benchmark table, cuBLASLt strict column) -> 16384 / 0.3512 s.
PAGES_TOKENS_PER_S = 16384 / 0.3512
PAGES_CONTEXT = "H100 PCIe, strict cuBLASLt fwd+bwd 351.2 ms at 16384 tokens (context: other hardware)"

# DRAM traffic per launch of the dominant kernel from one ncu capture, valid only
# while the kernel sources are unchanged (checked by hash).  None until captured.
NCU_TRAFFIC = None  # e.g. {"kernel": "grad_hidden", "bytes_per_launch": ..., "sources_sha": "..."}

GEMM_KERNELS = ("fwd_partials", "dlogits", "grad_hidden", "grad_weight")


def sources_sha() -> str:
    csrc = os.path.join(ROOT, "lm_head_selected_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (a no-op for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_cores_used() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample_seconds(inp, rows: int) -> float:
    """Time the FP64 oracle's forward + backward on the first `rows` tokens."""
    import oracle
    sub = inp.rows(list(range(rows)))
    a = (sub.hidden.double().numpy(), sub.weight.double().numpy(), None, sub.targets.numpy(), None, -100)
    g = sub.grad_logp.double().numpy()
    t0 = time.perf_counter()
    oracle.forward(*a)
    oracle.backward(g, *a)
    return time.perf_counter() - t0


def make_workload(name):
    import workloads
    N, D, V, desc = WORKLOADS[name]
    inp = workloads.rl_scoring(N=N, D=D, V=V, seed=1002, grad_std=1.0)
    return inp, desc


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp, desc = make_workload(args.workload)
    rows = args.reference_rows
    for _ in range(args.warmup):
        oracle_sample_seconds(inp, rows)
    times = [oracle_sample_seconds(inp, rows) for _ in range(args.steps)]
    mean_s = sum(times) / len(times)
    value = rows / mean_s
    cores = cpu_cores_used()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "N": inp.N, "D": inp.D, "V": inp.V, "description": desc,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} of {inp.N} tokens per step, full D and V, FP64 forward+backward"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from lm_head_selected_gb300 import _lib, build
    build.build()
    import lm_head_selected_gb300 as llp

    inp, desc = make_workload(args.workload)
    N, D, V = inp.N, inp.D, inp.V
    h = inp.hidden.to(dev)
    w = inp.weight.to(dev)
    t = inp.targets.to(dev)
    g = inp.grad_logp.to(dev)
    ws_f = torch.empty(llp.fwd_workspace_bytes(N, D, V), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(llp.bwd_workspace_bytes(N, D, V, False), dtype=torch.uint8, device=dev)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)

    def step():
        llp.linear_logp_fwd(h, w, t, workspace=ws_f, out=(logp, lse))
        return llp.linear_logp_bwd(g, lse, h, w, t, workspace=ws_b)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
            torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step()
    if llp.device_status() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait during warm-up")
    barrier()

    cap = args.steps * 8
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    _lib.profile_start(cap)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    launches = _lib.profile_stop(cap)
    clk = clocks.stop() if clocks else None
    if llp.device_status() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait during the timed region")
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    value = world * N / (ms_step * 1e-3)

    # per-kernel device time from the launch recorder (same stream, same timed region)
    per = {}
    for name, ms in launches:
        d = per.setdefault(name, {"launches": 0, "ms_total": 0.0})
        d["launches"] += 1
        d["ms_total"] += ms
    kernels = {}
    for name, d in per.items():
        avg = d["ms_total"] / d["launches"]
        kernels[name] = {"launches_per_step": d["launches"] / args.steps, "ms_per_launch": avg,
                         "share": d["ms_total"] / max(sum(x["ms_total"] for x in per.values()), 1e-9)}
        if name in GEMM_KERNELS:
            kernels[name]["tflops"] = 2.0 * N * V * D / (avg * 1e-3) / 1e12

    peaks = load_peaks()
    flops_counted = 6.0 * N * V * D
    step_tflops = flops_counted / (ms_step * 1e-3) / 1e12
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches_per_step"])
    dk = kernels[dom]
    if dom in GEMM_KERNELS:
        achieved = dk["tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops_sustained"], "kernel": dom,
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "peak_kind": f"bf16 sustained ({peaks['source']}); kernel timed inside back-to-back steps",
                "algorithmic_per_launch": f"2*N*V*D = {2.0 * N * V * D:.4e} flop"}
    else:
        roof = {"bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": None,
                "kernel": dom}
    roof["traffic"] = None
    if NCU_TRAFFIC and NCU_TRAFFIC.get("kernel") == dom and NCU_TRAFFIC.get("sources_sha") == sources_sha():
        roof["traffic"] = NCU_TRAFFIC["bytes_per_launch"]

    # forward-only throughput (same inputs), for context
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        llp.linear_logp_fwd(h, w, t, workspace=ws_f, out=(logp, lse))
    f1.record(stream)
    barrier()
    fwd_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.steps

    # end to end through the public autograd API with pinned host inputs and a
    # device-to-host read of the per-token log-probs every step
    h_host = inp.hidden.pin_memory()
    t_host = inp.targets.pin_memory()
    g_host = inp.grad_logp.pin_memory()
    out_host = torch.empty(N, dtype=torch.float32).pin_memory()
    w_param = w.detach().clone().requires_grad_(True)

    def e2e_step():
        hd = h_host.to(dev, non_blocking=True).requires_grad_(True)
        td = t_host.to(dev, non_blocking=True)
        gd = g_host.to(dev, non_blocking=True)
        w_param.grad = None
        lp = llp.linear_logp(hd, w_param, td)
        lp.backward(gd)
        out_host.copy_(lp.detach(), non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    t1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    h2d = h_host.numel() * 2 + t_host.numel() * 8 + g_host.numel() * 4
    d2h = out_host.numel() * 4

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = args.cpu_rows
        secs = oracle_sample_seconds(inp, rows)
        cpu = {"value": rows / secs, "unit": UNIT, "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"first {rows} of {N} tokens, full D={D} and V={V}, FP64 forward+backward, "
                         f"{secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGES_TOKENS_PER_S, "vs_baseline_context": PAGES_CONTEXT,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "N": N, "D": D, "V": V, "bias": False, "temperature": False,
                       "description": desc, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (weight 704.6 MB > 129 MB), no flush"},
            "tensor_peak_frac": step_tflops / peaks["bf16_tflops_sustained"],
            "tensor_peak_frac_of_burst": step_tflops / peaks["bf16_tflops"],
            "step_tflops_counted": step_tflops,
            "flops_counted_per_step": "6*N*V*D", "flops_executed_per_step": "8*N*V*D (logit tiles recomputed)",
            "roofline": roof,
            "kernels": kernels,
            "gpu_launches": len(launches),
            "fwd_only": {"value": world * N / (fwd_ms * 1e-3), "unit": UNIT, "ms_per_step": fwd_ms,
                         "tensor_peak_frac": 2.0 * N * V * D / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"]},
            "e2e": {"value": world * N / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "lm_head_selected_gb300.linear_logp autograd, pinned host inputs"},
            "cpu_baseline": cpu,
            "clocks": clk,
            "peaks": peaks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOADS), default="rl_head_fwd_bwd")
    ap.add_argument("--cpu-rows", type=int, default=512, help="token rows in the timed oracle sample")
    ap.add_argument("--reference-rows", type=int, default=64, help="token rows per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
