"""Throughput of the GPT-2-small forward pass + mean next-token cross-entropy on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full forward + loss (embedding, 12 blocks, ln_f, tied head with
the fused cross-entropy, mean) over a batch of B x T synthetic tokens of the
GPT-2-small workload (V=50257, C=768, H=12, L=12; B=16, T=1024, Zipf(1.1) ids,
seed 4; random-init weights of that architecture, bf16 with fp32 accumulation).
Prints one JSON line on rank 0. Under torchrun each rank runs an independent
replica on its own GPU (the path has no exchange step): value = all ranks'
tokens / max-over-ranks time ("weak" scaling).

--impl reference times the fp64 oracle on the host cores, one bounded sample
(one sequence prefix) per step, in the same metric and unit.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPT-2 small fwd+CE tokens/sec on 1 GB300; % of BF16 tensor-core peak"
WORKLOAD = "gpt2_small_b16_t1024"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def step_flops(cfg, B, T):
    """2 * unique params * tokens + causal attention 2*L*C*T*(T+1)*B (the stated convention)."""
    from decoder_only_transformer_gpt_gb300 import binding
    n = binding.param_count(cfg)
    return 2.0 * n * B * T + 2.0 * cfg.L * cfg.C * T * (T + 1) * B


class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(wl, w, ids, tg, budget_s: float = 12.0):
    """The fp64 oracle, as it stands, on a bounded sample: the first row's prefix."""
    import oracle
    T = 128
    best = None
    while True:
        t0 = time.perf_counter()
        oracle.forward(wl.cfg, w, ids[:1, :T], tg[:1, :T])
        dt = time.perf_counter() - t0
        best = (T, dt)
        if dt * 2.2 > budget_s or T >= ids.shape[1]:
            break
        T = min(ids.shape[1], T * 2)
    T, dt = best
    return {"value": T / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"1 sequence x {T} tokens of the same workload (prefix of row 0), numpy float64",
            "seconds": dt}


def run_reference(args, rank, world):
    """--impl reference: the oracle timed on host cores (rank 0 only)."""
    if rank != 0:
        return
    from workloads import workload
    from workloads.generate import generate
    import oracle
    wl = workload("gpt2_sweep")
    w, ids, tg = generate(wl, B=16, T=1024)
    T = 128
    for _ in range(args.warmup):
        oracle.forward(wl.cfg, w, ids[:1, :T], tg[:1, :T])
    t0 = time.perf_counter()
    for k in range(args.steps):
        r = k % ids.shape[0]
        oracle.forward(wl.cfg, w, ids[r:r + 1, :T], tg[r:r + 1, :T])
    dt = time.perf_counter() - t0
    value = args.steps * T / dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "B": 16, "T": 1024, "sample_per_step": f"1 x {T} tokens"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"1 sequence x {T} tokens per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import workload
    from workloads.generate import generate

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workload("gpt2_sweep")
    B, T = args.batch, args.seq
    w, ids_np, tg_np = generate(wl, B=B, T=T)
    cfg = wl.cfg
    model = binding.GPTModel(cfg, w, B * T)
    lib = model.lib
    ids = torch.from_numpy(ids_np).to(dev)
    tg = torch.from_numpy(tg_np).to(dev)
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up (also checks the device status once)
    for _ in range(args.warmup):
        model.forward(ids, tg, loss, None, check=False)
    model.status()
    launches_per_step = lib.gpt_last_launch_count(model.handle)

    # timed region: K steps, the head launch of each step bracketed by events
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in ev0 + ev1:
        e.record(stream)          # torch creates the CUDA event on first record; the library re-records it
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for k in range(args.steps):
        lib.gpt_time_step(model.handle, 8, -1, ev0[k].cuda_event, ev1[k].cuda_event)   # GPT_STEP_HEAD
        model.forward(ids, tg, loss, None, check=False)
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    model.status()
    ms = start.elapsed_time(stop)
    head_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    tokens = B * T * args.steps * world
    value = tokens / (ms_max / 1e3)

    # e2e: the host-buffer C-ABI call (H2D of ids and targets, D2H of the loss and
    # the status word inside every step), timed on the host clock
    pin_ids = torch.from_numpy(ids_np).pin_memory()
    pin_tg = torch.from_numpy(tg_np).pin_memory()
    pin_loss = torch.zeros(1, dtype=torch.float32).pin_memory()
    for _ in range(2):
        model.forward_host_ptrs(pin_ids.data_ptr(), pin_tg.data_ptr(), B, T, pin_loss.data_ptr())
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        model.forward_host_ptrs(pin_ids.data_ptr(), pin_tg.data_ptr(), B, T, pin_loss.data_ptr())
    e2e_s = time.perf_counter() - t0
    te = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(te, op=dist.ReduceOp.MAX)
    e2e_value = tokens / float(te.item())

    if rank != 0:
        model.close()
        return
    pk, pk_src = peaks()
    flops = step_flops(cfg, B, T)
    head_flops = 2.0 * B * T * cfg.V * cfg.C
    head_avg = statistics.mean(head_ms)
    achieved = head_flops / (head_avg / 1e3) / 1e12
    peak = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")))
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, w, ids_np, tg_np)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD if (B, T) == (16, 1024) else f"gpt2_small_b{B}_t{T}", "B": B, "T": T,
                   "V": cfg.V, "C": cfg.C, "H": cfg.H, "L": cfg.L, "ids": "zipf(1.1) seed 4",
                   "l2": "inputs larger than L2 (weights 249 MB + activations per step > 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "tflops": flops * args.steps * world / (ms_max / 1e3) / 1e12,
        "frac_of_peak": flops / (ms_max / args.steps / 1e3) / 1e12 / float(pk["bf16_tflops"]),
        "peak_source": f"{pk_src} bf16 {pk['bf16_tflops']} TFLOP/s burst",
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * B * T * 4,
                "d2h_bytes_per_step": 8},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": "gemm_tc_kernel<EPI_CE> (tied LM head + cross-entropy partials)",
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{pk_src} bf16 sustained", "avg_launch_ms": head_avg},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    model.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--seq", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from decoder_only_transformer_gpt_gb300 import build
    build.build()
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
