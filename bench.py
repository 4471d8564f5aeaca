#!/usr/bin/env python
"""Benchmark of the fused linear selected-token log-probability on GB300.

One step = one pass of the whole hot path over one batch: the forward (vocab
split partials + fixed-order merge) and the backward (dlogits recompute,
grad_hidden, grad_weight and their fixed-order segment sums) through the C ABI.

Default workload: the RL-scoring / training head of the pages' Nemotron-3-Nano
shape, N=16384 tokens (batch 32 x seq 512), D=2688, V=131072, bf16, no bias,
tau = 1, grad_logp ~ N(0,1), inputs resident in HBM.  W (704.6 MB) is larger
than the 129 MB L2, so no L2 flush is needed between steps; workloads whose
working set fits in L2 (``--workload tiny``) write a buffer twice the L2 size
between steps instead.

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
import re
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
    # batch 2 x seq 16 on the same head: the weight stream bounds every kernel (HBM roofline)
    "nemotron_n32": (32, 2688, 131072,
                     "Nemotron-3-Nano LM head, N=32 (2x16), D=2688, V=131072, no bias, per-row tau~U[0.7,1.3], "
                     "uniform targets, grad_logp=1"),
    # batch 1 x seq 16 on the same head
    "nemotron_n16": (16, 2688, 131072,
                     "Nemotron-3-Nano LM head, N=16 (1x16), D=2688, V=131072, no bias, per-row tau~U[0.7,1.3], "
                     "uniform targets, grad_logp=1"),
    # the tiny correctness configuration (quick runs of the bench's own code paths)
    "tiny": (64, 256, 4096,
             "tiny correctness case, N=64, D=256, V=4096, bias~N(0,0.1^2), 4 ignored rows, grad_logp=1"),
    # the training-step and long-context parity configurations, timed for reference
    "train_d4096": (16384, 4096, 128256,
                    "training step, N=16384, D=4096, V=128256, bf16, bias~N(0,0.1^2), grad_logp~N(0,1), "
                    "uniform targets"),
    "long_context": (65600, 2688, 131072,
                     "long-context stress, N=65600, D=2688, V=131072, no bias, one row shifted by +9984, "
                     "duplicate targets; grad_weight reduced over three 32768-token segments"),
}
# The pages' number for this metric and workload: strict fused fwd+bwd, 16384 tokens,
# D=2688, V=131072, 351.2 ms on an H100 PCIe ("Feat/nemotron h lm head logprob cuda",
# Benchmark table, cuBLASLt strict column) -> 16384 / 0.3512 s.
PAGES_TOKENS_PER_S = 16384 / 0.3512
PAGES_CONTEXT = "H100 PCIe, strict cuBLASLt fwd+bwd 351.2 ms at 16384 tokens (context: other hardware)"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# tcgen05 GEMM kernel from one single-pass ncu capture of the default workload,
# valid only while the kernel sources are unchanged (checked by sources_sha).
NCU_TRAFFIC = {
    "workload": "rl_head_fwd_bwd",
    "sources_sha": "78e648d649a7c836",
    "how": ("dram__bytes_read.sum + dram__bytes_write.sum of one launch per kernel (ncu -k one kernel, -c 1, "
            "1 pass), full-size workload, one box; box-to-box spread for the same build is large"),
    "bytes_per_launch": {"fwd_partials": 4217778000 + 36973056, "dlogits": 6445659000 + 4277988000,
                         "grad_hidden": 26158636000 + 696774400, "grad_weight": 11885443000 + 705190400},
}

GEMM_KERNELS = ("fwd_partials", "dlogits", "grad_hidden", "grad_weight")


def sources_sha(csrc=None) -> str:
    """Hash of the CUDA / C++ sources with comments and blank space removed, so a
    comment edit keeps the recorded traffic valid and a code edit does not."""
    csrc = csrc or os.path.join(ROOT, "lm_head_selected_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            text = " ".join(text.split())
            h.update(f.encode())
            h.update(text.encode())
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
    sub = inp.rows(list(range(min(rows, inp.N))))
    a = (sub.hidden.double().numpy(), sub.weight.double().numpy(),
         None if sub.bias is None else sub.bias.double().numpy(), sub.targets.numpy(),
         None if sub.temperature is None else sub.temperature.double().numpy(), sub.ignore_index)
    g = sub.grad_logp.double().numpy()
    t0 = time.perf_counter()
    oracle.forward(*a)
    oracle.backward(g, *a)
    return time.perf_counter() - t0


def make_workload(name):
    import workloads
    N, D, V, desc = WORKLOADS[name]
    if name in ("nemotron_n32", "nemotron_n16"):
        inp = workloads.nemotron_head(N=N, seed=1001)
    elif name == "tiny":
        inp = workloads.tiny()
    elif name == "train_d4096":
        inp = workloads.train(N=N, seed=1003)
    elif name == "long_context":
        inp = workloads.long_context(N=N, seed=1004)
        import torch
        inp.grad_logp = torch.randn(N, generator=torch.Generator().manual_seed(1004))
    else:
        inp = workloads.rl_scoring(N=N, D=D, V=V, seed=1002, grad_std=1.0)
    return inp, desc


def kernel_model(name, N, D, V, has_bias, has_tau):
    """Algorithmic (flop, byte) count of one launch of each kernel of the path:
    every operand read once, every result written once."""
    S = -(-V // 512)
    Vp = -(-V // 64) * 64
    nseg_v = -(-V // 32768)
    nseg_n = -(-N // 32768)
    W = 2.0 * V * D
    H = 2.0 * N * D
    row_in = 8.0 * N + (4.0 * N if has_tau else 0.0) + (4.0 * V if has_bias else 0.0)
    gemm = 2.0 * N * V * D
    if name == "fwd_partials":
        return gemm, W + H + row_in + 8.0 * S * N + 4.0 * N
    if name == "fwd_merge":
        return 0.0, 8.0 * S * N + 4.0 * N + 8.0 * N + 8.0 * N
    if name == "dlogits":
        return gemm, W + H + row_in + 8.0 * N + 2.0 * N * Vp + (4.0 * V * (-(-N // 32)) if has_bias else 0.0)
    if name == "grad_hidden":
        return gemm, 2.0 * N * V + W + (4.0 * nseg_v * N * D if nseg_v > 1 else 2.0 * N * D)
    if name == "segment_sum_hidden":
        return 0.0, 4.0 * nseg_v * N * D + 2.0 * N * D
    if name == "grad_weight":
        return gemm, 2.0 * N * V + H + (4.0 * nseg_n * V * D if nseg_n > 1 else W)
    if name == "segment_sum_weight":
        return 0.0, 4.0 * nseg_n * V * D + W
    if name == "bias_sum":
        return 0.0, 4.0 * V * (-(-N // 32)) + 4.0 * V
    return 0.0, 0.0


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp, desc = make_workload(args.workload)
    rows = min(args.reference_rows, inp.N)
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
    if args.dtype == "fp16":  # the same values rounded to fp16 (exact for these ranges)
        inp.hidden = inp.hidden.to(torch.float16)
        inp.weight = inp.weight.to(torch.float16)
        desc += "; hidden / weight in fp16"
    N, D, V = inp.N, inp.D, inp.V
    h = inp.hidden.to(dev)
    w = inp.weight.to(dev)
    t = inp.targets.to(dev)
    g = inp.grad_logp.to(dev)
    b = None if inp.bias is None else inp.bias.to(dev)
    tau = None if inp.temperature is None else inp.temperature.to(dev)
    ws_f = torch.empty(llp.fwd_workspace_bytes(N, D, V), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(llp.bwd_workspace_bytes(N, D, V, b is not None), dtype=torch.uint8, device=dev)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)

    # A working set that fits in L2 is flushed between timed steps by writing a
    # buffer twice the L2 size (inside the timed region); larger ones need no flush.
    l2_bytes = 129e6
    small = (2.0 * V * D + 2.0 * N * D) < 2 * l2_bytes
    flush_buf = torch.empty(int(2 * l2_bytes), dtype=torch.uint8, device=dev) if small else None
    if small:
        l2_note = f"working set {(2.0 * V * D + 2.0 * N * D) / 1e6:.1f} MB fits in L2: a 258 MB buffer is " \
                  "written between steps, inside the timed region"
    else:
        l2_note = f"inputs larger than L2 (weight {2.0 * V * D / 1e6:.1f} MB > 129 MB), no flush"

    def flush():
        if flush_buf is not None:
            flush_buf.zero_()

    def step():
        flush()
        llp.linear_logp_fwd(h, w, t, b, tau, workspace=ws_f, out=(logp, lse))
        return llp.linear_logp_bwd(g, lse, h, w, t, b, tau, workspace=ws_b)

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

    cap = args.steps * 12  # at most 9 launches per fwd+bwd step
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
    peaks = load_peaks()
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    kernels = {}
    for name, d in per.items():
        avg = d["ms_total"] / d["launches"]
        fl, by = kernel_model(name, N, D, V, b is not None, tau is not None)
        kernels[name] = {"launches_per_step": d["launches"] / args.steps, "ms_per_launch": avg,
                         "share": d["ms_total"] / max(sum(x["ms_total"] for x in per.values()), 1e-9),
                         "algorithmic_gb": by / 1e9, "gbs": by / (avg * 1e-3) / 1e9,
                         "bound": "tensor" if fl > ridge * by else "hbm"}
        if fl > 0:
            kernels[name]["tflops"] = fl / (avg * 1e-3) / 1e12

    flops_counted = 6.0 * N * V * D
    step_tflops = flops_counted / (ms_step * 1e-3) / 1e12
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches_per_step"])
    dk = kernels[dom]
    if dk["bound"] == "tensor":
        achieved = dk["tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops_sustained"], "kernel": dom,
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "peak_kind": f"bf16 sustained ({peaks['source']}); kernel timed inside back-to-back steps",
                "algorithmic_per_launch": f"2*N*V*D = {2.0 * N * V * D:.4e} flop"}
    else:
        achieved = dk["gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": dom,
                "peak_kind": f"HBM copy bandwidth ({peaks['source']})",
                "algorithmic_per_launch": f"{dk['algorithmic_gb'] * 1e9:.4e} bytes (every operand read once, "
                                          f"every result written once)"}
    roof["traffic"] = None
    roof["traffic_source"] = "none recorded for this build and workload"
    if (NCU_TRAFFIC and args.dtype == "bf16" and NCU_TRAFFIC["workload"] == args.workload
            and NCU_TRAFFIC["sources_sha"] == sources_sha()
            and dom in NCU_TRAFFIC["bytes_per_launch"]):
        roof["traffic"] = NCU_TRAFFIC["bytes_per_launch"][dom]
        roof["traffic_source"] = ("recorded ncu capture, not measured in this run: " + NCU_TRAFFIC["how"] +
                                  f"; sources sha {NCU_TRAFFIC['sources_sha']}")
        for k, v in NCU_TRAFFIC["bytes_per_launch"].items():
            if k in kernels:
                kernels[k]["dram_gb_ncu"] = v / 1e9

    # forward-only throughput (same inputs), for context
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        flush()
        llp.linear_logp_fwd(h, w, t, b, tau, workspace=ws_f, out=(logp, lse))
    f1.record(stream)
    barrier()
    fwd_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.steps

    # end to end through the public autograd API with pinned host inputs and a
    # device-to-host read of the per-token log-probs every step.  As in a training
    # input pipeline, the next step's inputs are copied on a second stream while
    # the current step computes: K steps time K host-to-device copies (the first
    # step's before the timed region, one for a step after it inside).
    h_host = inp.hidden.pin_memory()
    t_host = inp.targets.pin_memory()
    g_host = inp.grad_logp.pin_memory()
    tau_host = None if inp.temperature is None else inp.temperature.pin_memory()
    out_host = torch.empty(N, dtype=torch.float32).pin_memory()
    w_param = w.detach().clone().requires_grad_(True)
    b_param = None if b is None else b.detach().clone().requires_grad_(True)
    copy_stream = torch.cuda.Stream(dev)

    def prefetch():
        with torch.cuda.stream(copy_stream):
            bufs = (h_host.to(dev, non_blocking=True), t_host.to(dev, non_blocking=True),
                    g_host.to(dev, non_blocking=True),
                    None if tau_host is None else tau_host.to(dev, non_blocking=True))
        ready = torch.cuda.Event()
        ready.record(copy_stream)
        return bufs, ready

    def e2e_step(staged):
        bufs, ready = staged
        stream.wait_event(ready)
        for x in bufs:
            if x is not None:
                x.record_stream(stream)
        nxt = prefetch()
        flush()
        hd, td, gd, taud = bufs
        hd.requires_grad_(True)
        w_param.grad = None
        if b_param is not None:
            b_param.grad = None
        lp = llp.linear_logp(hd, w_param, td, b_param, taud)
        lp.backward(gd)
        out_host.copy_(lp.detach(), non_blocking=True)
        return nxt

    staged = prefetch()
    for _ in range(3):
        staged = e2e_step(staged)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        staged = e2e_step(staged)
    t1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    h2d = h_host.numel() * 2 + t_host.numel() * 8 + g_host.numel() * 4 + (0 if tau_host is None else 4 * N)
    d2h = out_host.numel() * 4

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = min(args.cpu_rows, N)
        secs = oracle_sample_seconds(inp, rows)
        cpu = {"value": rows / secs, "unit": UNIT, "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"first {rows} of {N} tokens, full D={D} and V={V}, FP64 forward+backward, "
                         f"{secs:.1f} s"}

    # the pages' number is for the bf16 N=16384, D=2688, V=131072 step only
    same_as_pages = args.workload == "rl_head_fwd_bwd" and args.dtype == "bf16"
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGES_TOKENS_PER_S if same_as_pages else None,
            "vs_baseline_context": PAGES_CONTEXT if same_as_pages else "the pages quote no number for this workload",
            "dtype": "f16" if args.dtype == "fp16" else "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "N": N, "D": D, "V": V, "bias": b is not None, "temperature": tau is not None,
                       "description": desc, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": l2_note},
            "tensor_peak_frac": step_tflops / peaks["bf16_tflops_sustained"],
            "tensor_peak_frac_of_burst": step_tflops / peaks["bf16_tflops"],
            "step_tflops_counted": step_tflops,
            "flops_counted_per_step": "6*N*V*D", "flops_executed_per_step": "8*N*V*D (logit tiles recomputed)",
            "roofline": roof,
            "kernels": kernels,
            "gpu_launches": len(launches),
            # a short loop of forwards alone: quoted against the burst peak first
            "fwd_only": {"value": world * N / (fwd_ms * 1e-3), "unit": UNIT, "ms_per_step": fwd_ms,
                         "tensor_peak_frac": 2.0 * N * V * D / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                         "tensor_peak_frac_of_sustained":
                             2.0 * N * V * D / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                         "peak_kind": "bf16 burst (the loop is short); sustained beside it"},
            "e2e": {"value": world * N / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "lm_head_selected_gb300.linear_logp autograd, pinned host inputs",
                    "copies": "next step's inputs copied on a second stream during the current step"},
            "cpu_baseline": cpu,
            "clocks": clk,
            "peaks": peaks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_fused(args):
    """Logits-input fused log-prob: forward (row statistics + target gather) and
    backward (grad_logits from the saved statistics) over bf16 logits [N, V];
    bound by HBM bandwidth (forward reads every logit once; backward reads every
    logit and writes every gradient once)."""
    import torch

    from lm_head_selected_gb300 import build
    build.build()
    import lm_head_selected_gb300 as llp

    N, V = args.fused_n, args.fused_v
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(1005)
    z = (torch.randn(N, V, generator=g) * 3.0).to(torch.bfloat16).to(dev)
    t = torch.randint(0, V, (N,), generator=g).to(dev)
    gl = torch.randn(N, generator=g).to(dev)
    from lm_head_selected_gb300 import _lib
    ws = torch.empty(_lib.load().fused_logp_workspace_bytes(N, V), dtype=torch.uint8, device=dev)
    grad = torch.empty_like(z)

    def fwd():
        return llp.fused_logp_fwd(z, t, workspace=ws)

    _, m, ls = fwd()

    def bwd():
        llp.fused_logp_bwd(gl, m, ls, z, t, out=grad)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(0)
    clocks.start()
    f_ms = timed(fwd)
    b_ms = timed(bwd)
    clk = clocks.stop()
    peaks = load_peaks()
    S = -(-V // 16384)
    f_bytes = 2.0 * N * V + 8.0 * N * S + 8.0 * N + 12.0 * N
    b_bytes = 2.0 * N * V * 2 + 8.0 * N + 12.0 * N
    f_gbs = f_bytes / (f_ms * 1e-3) / 1e9
    b_gbs = b_bytes / (b_ms * 1e-3) / 1e9
    dom_name, dom_gbs, dom_bytes = ("fused_grad", b_gbs, b_bytes) if b_ms >= f_ms else ("fused_split", f_gbs, f_bytes)
    line = {
        "metric": "logits-input fused logp fwd+bwd tokens/s (HBM-bound)", "value": N / ((f_ms + b_ms) * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": f_ms + b_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"fused_logp N={N} V={V} bf16 logits", "N": N, "V": V,
                   "l2": f"inputs larger than L2 ({2.0 * N * V / 1e9:.2f} GB of logits)"},
        "fwd": {"ms": f_ms, "gbs": f_gbs, "frac_of_hbm": f_gbs / peaks["hbm_gbs"]},
        "bwd": {"ms": b_ms, "gbs": b_gbs, "frac_of_hbm": b_gbs / peaks["hbm_gbs"]},
        "roofline": {"bound": "hbm", "achieved": dom_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dom_gbs / peaks["hbm_gbs"], "kernel": dom_name, "traffic": None,
                     "algorithmic_per_launch": f"{dom_bytes:.4e} bytes"},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_indexed(args):
    """Row-subset variant (linear_logp_fwd_indexed / _bwd_indexed) on a seeded
    subset of round(select_frac * N) rows of the workload, timed against the plain
    path on the same rows compacted into a K-row problem: the difference is the
    cost of selecting, compacting and scattering back."""
    import torch

    from lm_head_selected_gb300 import build
    build.build()
    import lm_head_selected_gb300 as llp

    inp, desc = make_workload(args.workload)
    N, D, V = inp.N, inp.D, inp.V
    dev = torch.device("cuda", 0)
    h, w, t, g = inp.hidden.to(dev), inp.weight.to(dev), inp.targets.to(dev), inp.grad_logp.to(dev)
    b = None if inp.bias is None else inp.bias.to(dev)
    tau = None if inp.temperature is None else inp.temperature.to(dev)
    K = max(1, min(N, int(round(args.select_frac * N))))
    idx = torch.randperm(N, generator=torch.Generator().manual_seed(1006))[:K].sort().values.to(dev)
    logp = torch.zeros(N, dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("-inf"), dtype=torch.float32, device=dev)

    def indexed():
        llp.ops.linear_logp_fwd_indexed(h, w, t, idx, b, tau, out=(logp, lse))
        llp.ops.linear_logp_bwd_indexed(g, lse, h, w, t, idx, b, tau)

    hk, tk, gk = h[idx].contiguous(), t[idx].contiguous(), g[idx].contiguous()
    tauk = None if tau is None else tau[idx].contiguous()
    ws_f = torch.empty(llp.fwd_workspace_bytes(K, D, V), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(llp.bwd_workspace_bytes(K, D, V, b is not None), dtype=torch.uint8, device=dev)
    lpk = torch.empty(K, dtype=torch.float32, device=dev)
    lsek = torch.empty(K, dtype=torch.float32, device=dev)

    def plain():
        llp.linear_logp_fwd(hk, w, tk, b, tauk, workspace=ws_f, out=(lpk, lsek))
        llp.linear_logp_bwd(gk, lsek, hk, w, tk, b, tauk, workspace=ws_b)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    # alternate the two (A B B A) so that neither gets the cooler, faster clock
    clocks = ClockSampler(0)
    clocks.start()
    i_ms = timed(indexed)
    p_ms = timed(plain)
    p_ms = (p_ms + timed(plain)) / 2
    i_ms = (i_ms + timed(indexed)) / 2
    clk = clocks.stop()
    if llp.device_status() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")
    peaks = load_peaks()
    tflops = 6.0 * K * V * D / (i_ms * 1e-3) / 1e12
    line = {
        "metric": "row-subset fwd+bwd selected tokens/s", "value": K / (i_ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": i_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if h.dtype == torch.float16 else "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}, indexed: {K} of {N} rows", "N": N, "K": K, "D": D, "V": V,
                   "description": desc},
        "tensor_peak_frac": tflops / peaks["bf16_tflops_sustained"],
        "plain_same_rows_ms": p_ms,
        "selection_overhead": i_ms / p_ms - 1.0,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_shards(args):
    """Vocab-parallel device work of one rank on one GPU: the workload's head cut
    into R equal contiguous vocab shards; rank 0's step is its shard forward, the
    merge of the R gathered (max, sum, target logit) triples, its shard backward
    and the rank-ordered sum of the R fp32 grad_hidden contributions.  The other
    ranks' triples and contributions are computed once beforehand, standing in for
    the all-gathers (not timed: one GPU, no interconnect).  Timed against the
    unsharded step on the same GPU."""
    import torch

    from lm_head_selected_gb300 import build, tp
    build.build()
    import lm_head_selected_gb300 as llp

    inp, desc = make_workload(args.workload)
    N, D, V = inp.N, inp.D, inp.V
    R = args.shards
    if V % R:
        raise ValueError("--shards must divide the vocabulary size")
    Vl = V // R
    dev = torch.device("cuda", 0)
    h, w, t, g = inp.hidden.to(dev), inp.weight.to(dev), inp.targets.to(dev), inp.grad_logp.to(dev)
    b = None if inp.bias is None else inp.bias.to(dev)
    tau = None if inp.temperature is None else inp.temperature.to(dev)
    shard = [(w[r * Vl:(r + 1) * Vl], None if b is None else b[r * Vl:(r + 1) * Vl]) for r in range(R)]
    gathered = torch.stack([tp.fwd_shard(h, ws_, t, r * Vl, bs_, tau) for r, (ws_, bs_) in enumerate(shard)])
    _, lse0 = tp.merge_shards(gathered, t, V)
    parts = torch.stack([tp.bwd_shard(g, lse0, h, ws_, t, r * Vl, V, bs_, tau)[0]
                         for r, (ws_, bs_) in enumerate(shard)])

    def rank0():
        gathered[0] = tp.fwd_shard(h, shard[0][0], t, 0, shard[0][1], tau)
        _, lse = tp.merge_shards(gathered, t, V)
        parts[0] = tp.bwd_shard(g, lse, h, shard[0][0], t, 0, V, shard[0][1], tau)[0]
        tp.sum_partials(parts, h.dtype)

    ws_f = torch.empty(llp.fwd_workspace_bytes(N, D, V), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(llp.bwd_workspace_bytes(N, D, V, b is not None), dtype=torch.uint8, device=dev)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)

    def whole():
        llp.linear_logp_fwd(h, w, t, b, tau, workspace=ws_f, out=(logp, lse))
        llp.linear_logp_bwd(g, lse, h, w, t, b, tau, workspace=ws_b)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(0)
    clocks.start()
    s_ms = timed(rank0)
    u_ms = timed(whole)
    u_ms = (u_ms + timed(whole)) / 2
    s_ms = (s_ms + timed(rank0)) / 2
    clk = clocks.stop()
    if llp.device_status() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait")
    line = {
        "metric": "vocab-parallel fwd+bwd device time of one rank", "value": s_ms, "unit": "ms",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": s_ms,
        "higher_is_better": False, "scaling": "strong", "vs_baseline": None,
        "dtype": "f16" if h.dtype == torch.float16 else "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}, {R} vocab shards of {Vl}", "N": N, "D": D, "V": V, "shards": R,
                   "description": desc, "exchange": "not timed (one GPU): the all-gathers of the triples and "
                                                    "of the fp32 grad_hidden contributions"},
        "unsharded_ms": u_ms,
        "rank_share_of_unsharded": s_ms / u_ms,
        "ideal_share": 1.0 / R,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
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
    ap.add_argument("--dtype", choices=("bf16", "fp16"), default="bf16", help="hidden / weight type")
    ap.add_argument("--op", choices=("linear_logp", "fused_logp", "indexed", "shards"), default="linear_logp",
                    help="linear_logp: the fused LM-head path (default); fused_logp: the logits-input op; "
                         "indexed: the row-subset variant on --select-frac of the workload's rows; "
                         "shards: one rank's device work of the vocab-parallel path with --shards shards")
    ap.add_argument("--select-frac", type=float, default=0.5)
    ap.add_argument("--shards", type=int, default=2)
    ap.add_argument("--fused-n", type=int, default=16384)
    ap.add_argument("--fused-v", type=int, default=131072)
    args = ap.parse_args(argv)
    if args.op == "fused_logp":
        return run_fused(args)
    if args.op == "indexed":
        return run_indexed(args)
    if args.op == "shards":
        return run_shards(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
