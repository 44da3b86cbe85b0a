"""Throughput of the GPT-2-small forward pass + mean next-token cross-entropy on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--model gpt2_small|gpt2_xl]

One step = one full forward + loss (embedding, 12 blocks, ln_f, tied head with
the fused cross-entropy, mean) over a batch of B x T synthetic tokens of the
GPT-2-small workload (V=50257, C=768, H=12, L=12; B=16, T=1024, Zipf(1.1) ids,
seed 4; random-init weights of that architecture, bf16 with fp32 accumulation).
Prints one JSON line on rank 0. Under torchrun each rank runs an independent
replica on its own GPU (the path has no exchange step): value = all ranks'
tokens / max-over-ranks time ("weak" scaling).

--impl reference times the fp64 oracle on the host cores, one bounded sample
(one sequence prefix) per step, in the same metric and unit.

--model gpt2_xl runs the same path at the GPT-2 XL shape (48 blocks, C = 1600,
25 heads, FFN 6400; 1.56 B parameters) as a second workload; the default is
GPT-2 small, the configuration the throughput target is stated on.
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
MODELS = {   # --model: (workload, metric, workload name at B=16, T=1024)
    "gpt2_small": ("gpt2_sweep", METRIC, WORKLOAD),
    "gpt2_xl": ("gpt2_xl", "GPT-2 XL fwd+CE tokens/sec on 1 GB300; % of BF16 tensor-core peak",
                "gpt2_xl_b16_t1024"),
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# The steps of one forward pass, as numbered by the library's GPT_STEP_* probe
# ids: (name, probe id, launched once per block).
STEP_KINDS = [("embed", 0, False), ("c_attn", 1, True), ("attention", 2, True), ("c_proj", 3, True),
              ("ln_mid", 4, True), ("c_fc", 5, True), ("mlp_proj", 6, True), ("ln_out", 7, True),
              ("head", 8, False), ("ce_combine", 9, False), ("mean", 10, False)]

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of the same
# launch configuration, valid only while the kernel's sources hash to the digest recorded with it.
NCU_TRAFFIC = {
    "attention": {"bytes": 76.483840e6 + 3.919360e6, "profile": "profiles/attention_b16_t1024_h12_d64.md",
                  "sources": ["decoder_only_transformer_gpt_gb300/csrc/k_attn_tc.cu",
                              "decoder_only_transformer_gpt_gb300/csrc/common.cuh"],
                  "digest": "1458438068a7e65286a8c275768f49580badcdc5"},
    "head": {"bytes": 102.692096e6 + 17.542656e6, "profile": "profiles/head_ce_gemm_m16384_v50257_c768.md",
             "sources": ["decoder_only_transformer_gpt_gb300/csrc/k_gemm_tc.cu",
                         "decoder_only_transformer_gpt_gb300/csrc/common.cuh"],
             "digest": "f178bf16f28b49e4bd9873c0482bfb5e717633a7"},
    "mlp_proj": {"bytes": 173.873408e6 + 28.476928e6, "profile": "profiles/mlp_proj_gemm_m16384_n768_k3072.md",
                 "sources": ["decoder_only_transformer_gpt_gb300/csrc/k_gemm_tc.cu",
                             "decoder_only_transformer_gpt_gb300/csrc/common.cuh"],
                 "digest": "f178bf16f28b49e4bd9873c0482bfb5e717633a7"},
}

# The same for the training step's dominant step at B = 16, T = 1024: the attention derivative (Dsum,
# the derivative, the dQ conversion: dram__bytes_read.sum + dram__bytes_write.sum of each, one ncu
# capture at the full size) plus the 50.3 MB its memset of the fp32 dQ accumulator writes (not a kernel:
# counted, not captured).
TRAIN_NCU_TRAFFIC = {
    "b_attn": {"bytes": 291.41e6 + 123.16e6, "profile": "profiles/attention_bwd_b16_t1024_h12_d64.md",
               "sources": ["decoder_only_transformer_gpt_gb300/csrc/k_attn_bwd_tc.cu",
                           "decoder_only_transformer_gpt_gb300/csrc/common.cuh"],
               "digest": "29353750e4990b451a3948b707dec65cfdc0bab0"},
}


KERNEL_OF_STEP = {
    "embed": "embed_kernel (token + position rows, fused first LayerNorm)",
    "c_attn": "gemm_pair_kernel<EPI_BIAS_OUT, 0, 4> (fused QKV projection, CTA pairs)",
    "attention": "attn_fwd_tc_kernel<64> (causal attention, online softmax)",
    "c_proj": "gemm_tc_kernel<EPI_BIAS_RESID> (attention output projection + residual)",
    "ln_mid": "layernorm_kernel (ln_2)",
    "c_fc": "gemm_pair_kernel<EPI_BIAS_GELU_OUT, 0, 8> (MLP up-projection + GELU, CTA pairs, eight epilogue warps)",
    "mlp_proj": "gemm_pair_kernel<EPI_BIAS_RESID, 1, 4, 0> (MLP down-projection + residual, CTA pairs, stream-K)",
    "ln_out": "layernorm_kernel (next ln_1 / ln_f)",
    "head": "gemm_tc_kernel<EPI_CE> (tied LM head + cross-entropy partials)",
    "ce_combine": "ce_combine_kernel",
    "mean": "mean_kernel",
}


def source_digest(files):
    import hashlib
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def step_work(name, cfg, B, T):
    """Algorithmic work of one launch of a step: (amount, bound, unit of the rate).

    Contractions count 2 flops per multiply-add of the unique products (the causal
    half of QK^T and PV for attention); row-wise steps count the bytes they must
    move once: fp32 residual read + bf16 output for a LayerNorm, token rows of wte
    and wpe + fp32 x + bf16 LN output for the embedding, the head's partials for
    the combine.
    """
    M, C, F, V = B * T, cfg.C, cfg.ffn, cfg.V
    nb = (V + 255) // 256
    if name == "c_attn":
        return 2.0 * M * 3 * C * C, "tensor"
    if name == "attention":
        return 2.0 * B * C * T * (T + 1), "tensor"
    if name == "c_proj":
        return 2.0 * M * C * C, "tensor"
    if name in ("c_fc", "mlp_proj"):
        return 2.0 * M * C * F, "tensor"
    if name == "head":
        return 2.0 * M * V * C, "tensor"
    if name in ("ln_mid", "ln_out"):
        return M * C * (4.0 + 2.0), "hbm"
    if name == "embed":
        return M * 4.0 + M * C * 2.0 + T * C * 2.0 + M * C * (4.0 + 2.0), "hbm"
    if name == "ce_combine":
        return 2.0 * nb * M * 4 + 3.0 * M * 4, "hbm"
    return M * 4.0, "hbm"


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
    """The fp64 oracle, as it stands, on a bounded sample of the workload.

    Sequence prefixes of row 0 double in length until one costs a sizeable part
    of the budget (or the whole row is reached); then whole rows 1, 2, ... are
    added until about `budget_s` seconds of oracle time have been spent.
    """
    import oracle
    T = 128
    while True:
        t0 = time.perf_counter()
        oracle.forward(wl.cfg, w, ids[:1, :T], tg[:1, :T])
        dt = time.perf_counter() - t0
        if dt * 2.2 > budget_s or T >= ids.shape[1]:
            break
        T = min(ids.shape[1], T * 2)
    rows, tokens, spent = 1, T, dt
    while T == ids.shape[1] and spent + dt < budget_s and rows < ids.shape[0]:
        t0 = time.perf_counter()
        oracle.forward(wl.cfg, w, ids[rows:rows + 1, :T], tg[rows:rows + 1, :T])
        spent += time.perf_counter() - t0
        tokens += T
        rows += 1
    return {"value": tokens / spent, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows} sequence(s) x {T} tokens of the same workload (rows 0..{rows - 1}), numpy float64",
            "seconds": spent}


class RuntimeEvents:
    """CUDA events from the CUDA runtime library itself (ctypes), for the timing probe of the timed
    region: the library replays one captured forward per step and points its two event-record nodes
    at each step's events, which the driver accepts for these events (not for torch's)."""

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.rt = None
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                self.rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.rt is None:
            raise RuntimeError("libcudart not found for the timing events")

    def create(self) -> int:
        h = self.ct.c_void_p()
        if self.rt.cudaEventCreate(self.ct.byref(h)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        return h.value

    def elapsed_ms(self, a: int, b: int) -> float:
        ms = self.ct.c_float()
        rc = self.rt.cudaEventElapsedTime(self.ct.byref(ms), self.ct.c_void_p(a), self.ct.c_void_p(b))
        if rc != 0:
            raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
        return float(ms.value)

    def destroy(self, h: int) -> None:
        self.rt.cudaEventDestroy(self.ct.c_void_p(h))


def replica_rate(ms_local: float, units_local: float, world: int, device):
    """Independent replicas (weak scaling): the job's time is the slowest rank's, and its rate is
    every rank's units over that time. Collective: every rank must call it."""
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, units_local * world / (ms_max / 1e3)


def run_reference(args, rank, world):
    """--impl reference: the oracle timed on host cores (rank 0 only)."""
    if rank != 0:
        return
    from workloads import workload
    from workloads.generate import generate
    import oracle
    wl_name, metric, wl_label = MODELS[args.model]
    wl = workload(wl_name)
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
    line = {"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": wl_label, "B": 16, "T": 1024, "sample_per_step": f"1 x {T} tokens"},
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
    wl_name, metric, wl_label = MODELS[args.model]
    wl = workload(wl_name)
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

    # per-step breakdown (untimed): every launch of one forward bracketed by events, one probe per forward
    rte = RuntimeEvents()
    pa, pb = rte.create(), rte.create()
    breakdown = {}
    for name, sid, per_block in STEP_KINDS:
        times = []
        for layer in (range(cfg.L) if per_block else [-1]):
            lib.gpt_time_step(model.handle, sid, layer, pa, pb)
            model.forward(ids, tg, loss, None, check=False)
            torch.cuda.synchronize()
            if lib.gpt_last_probe_hits(model.handle) == 1:
                times.append(rte.elapsed_ms(pa, pb))
        if not times:                 # the step did not run in this configuration
            continue
        work, bound = step_work(name, cfg, B, T)
        breakdown[name] = {"launches_per_step": len(times), "avg_ms": statistics.mean(times),
                           "ms_per_step": sum(times), "work": work, "bound": bound}
    lib.gpt_time_step(model.handle, -1, -1, None, None)
    dom = max(breakdown, key=lambda k: breakdown[k]["ms_per_step"])
    dom_sid, dom_per_block = next((sid, pb_) for n, sid, pb_ in STEP_KINDS if n == dom)

    # timed region: K steps, one launch of the dominant step in each bracketed by events (the same
    # block's launch every step, so the library replays one captured graph whose two event-record
    # nodes it points at each step's events)
    ev0 = [rte.create() for _ in range(args.steps)]
    ev1 = [rte.create() for _ in range(args.steps)]
    dom_layer = (cfg.L // 2) if dom_per_block else -1
    for k in range(2):                # untimed: capture (and replay once) the probed forward
        lib.gpt_time_step(model.handle, dom_sid, dom_layer, ev0[k], ev1[k])
        model.forward(ids, tg, loss, None, check=False)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for k in range(args.steps):
        lib.gpt_time_step(model.handle, dom_sid, dom_layer, ev0[k], ev1[k])
        model.forward(ids, tg, loss, None, check=False)
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    model.status()
    ms = start.elapsed_time(stop)
    lib.gpt_time_step(model.handle, -1, -1, None, None)
    dom_ms = [rte.elapsed_ms(a, b) for a, b in zip(ev0, ev1)]
    for h in ev0 + ev1 + [pa, pb]:
        rte.destroy(h)
    ms_max, value = replica_rate(ms, B * T * args.steps, world, dev)

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
    _, e2e_value = replica_rate(1e3 * e2e_s, B * T * args.steps, world, dev)

    if rank != 0:
        model.close()
        return
    pk, pk_src = peaks()
    flops = step_flops(cfg, B, T)
    # every kernel here runs inside a step of a few ms, not a seconds-long loop under the power cap,
    # so the burst figure is its denominator; the sustained one is reported beside it
    peak_t = float(pk["bf16_tflops"])
    peak_ts = float(pk.get("bf16_tflops_sustained", peak_t))
    peak_b = float(pk.get("hbm_gbs"))

    def rate(work, bound, ms):
        if bound == "tensor":
            a = work / (ms / 1e3) / 1e12
            return a, peak_t, "TFLOP/s"
        a = work / (ms / 1e3) / 1e9
        return a, peak_b, "GB/s"

    # The breakdown brackets each launch with events, which stops it from overlapping its neighbours
    # (programmatic dependent launch): the bracketed times add up to more than a step. ms_per_step_scaled
    # shares the measured step time out in proportion to them.
    total_ms = sum(v["ms_per_step"] for v in breakdown.values())
    step_ms = ms_max / args.steps
    kernels = []
    for name, v in sorted(breakdown.items(), key=lambda kv: -kv[1]["ms_per_step"]):
        a, p, u = rate(v["work"], v["bound"], v["avg_ms"])
        kernels.append({"step": name, "launches_per_step": v["launches_per_step"], "avg_ms": v["avg_ms"],
                        "ms_per_step_scaled": v["ms_per_step"] * step_ms / total_ms,
                        "share": v["ms_per_step"] / total_ms, "bound": v["bound"], "achieved": a, "unit": u,
                        "frac": a / p})
    dom_avg = statistics.mean(dom_ms)
    achieved, peak, unit = rate(breakdown[dom]["work"], breakdown[dom]["bound"], dom_avg)
    traffic = None
    tr = NCU_TRAFFIC.get(dom)
    if (tr is not None and tr["bytes"] is not None and args.model == "gpt2_small" and (B, T) == (16, 1024)
            and source_digest(tr["sources"]) == tr["digest"]):
        traffic = tr["bytes"]
    n_params = cfg.L * (12 * cfg.C * cfg.C + 13 * cfg.C) + (cfg.V + cfg.ctx + 2) * cfg.C   # ffn = 4C
    weight_mb = 2e-6 * n_params                                                          # bf16
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, w, ids_np, tg_np)
    line = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl_label if (B, T) == (16, 1024) else f"{args.model}_b{B}_t{T}", "B": B, "T": T,
                   "V": cfg.V, "C": cfg.C, "H": cfg.H, "L": cfg.L, "ids": "zipf(1.1) seed 4",
                   "l2": f"inputs larger than L2 (weights {weight_mb:.0f} MB + activations per step > 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "tflops": flops * args.steps * world / (ms_max / 1e3) / 1e12,
        "frac_of_peak": flops / (ms_max / args.steps / 1e3) / 1e12 / float(pk["bf16_tflops"]),
        "peak_source": f"{pk_src} bf16 {pk['bf16_tflops']} TFLOP/s burst",
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * B * T * 4,
                "d2h_bytes_per_step": 8},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": KERNEL_OF_STEP[dom], "step": dom, "bound": breakdown[dom]["bound"],
                     "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": traffic,
                     "algorithmic": breakdown[dom]["work"],
                     "peak_source": f"{pk_src} " + ("bf16 burst" if unit == "TFLOP/s" else "HBM copy"),
                     "frac_of_sustained": (achieved / peak_ts) if unit == "TFLOP/s" else None,
                     "avg_launch_ms": dom_avg, "launches_timed": len(dom_ms)},
        "kernels": kernels,
        "kernels_note": ("avg_ms: each launch bracketed by events outside the timed region (no overlap with "
                         "its neighbours); sum of bracketed times per step %.3f ms against %.3f ms measured; "
                         "ms_per_step_scaled rescales them to the step" % (total_ms, step_ms)),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    model.close()


def run_decode(args, rank, world, local_rank):
    """--decode: tokens/s of incremental decoding with the key/value cache (a second measurement,
    not the default line). B sequences are prefilled with a prompt of --prompt tokens; then --steps
    decode steps (one new token per sequence each) are timed with CUDA events. Decode streams
    every weight and each sequence's cached keys and values once per step, so the roofline is
    HBM bandwidth: algorithmic bytes per step = weights (bf16) + B x L x (pos + 1) x 2C x 2 bytes
    of cache + the B x V fp32 logits written, averaged over the timed positions."""
    import torch
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import workload
    from workloads.generate import generate

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl_name, _, wl_label = MODELS[args.model]
    wl = workload(wl_name)
    cfg = wl.cfg
    B, T0 = args.batch, args.prompt
    n_new = args.warmup + args.steps
    if T0 + n_new > cfg.ctx:
        raise SystemExit(f"--prompt {T0} + {n_new} decode steps exceed ctx {cfg.ctx}")
    w, ids_np, _ = generate(wl, B=B, T=T0 + n_new)
    model = binding.GPTModel(cfg, w, B * T0)
    model.kv_reserve(B)
    ids = torch.from_numpy(ids_np).to(dev)
    cols = [ids[:, t].contiguous() for t in range(T0 + n_new)]
    logits = torch.empty((B, cfg.V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    model.prefill(ids[:, :T0].contiguous(), logits)
    for k in range(args.warmup):
        model.decode_step(cols[T0 + k], T0 + k, logits)
    model.status()
    launches = model.lib.gpt_last_launch_count(model.handle)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    torch.cuda.synchronize()
    start.record(stream)
    p0 = T0 + args.warmup
    for k in range(args.steps):
        model.decode_step(cols[p0 + k], p0 + k, logits)
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    model.status()
    ms = start.elapsed_time(stop)
    n_params = cfg.L * (12 * cfg.C * cfg.C + 13 * cfg.C) + (cfg.V + cfg.ctx + 2) * cfg.C
    mean_pos = p0 + (args.steps - 1) / 2.0
    step_bytes = 2.0 * n_params + B * cfg.L * (mean_pos + 1) * 2 * cfg.C * 2 + B * cfg.V * 4
    pk, pk_src = peaks()
    achieved = step_bytes * args.steps / (ms / 1e3) / 1e9
    line = {
        "metric": f"{wl_label.split('_b')[0]} decode tokens/sec (KV cache) on 1 GB300", "value": B * args.steps / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.model}_decode_b{B}_prompt{T0}", "B": B, "prompt": T0,
                   "positions": [p0, p0 + args.steps - 1],
                   "l2": f"weights {2e-6 * n_params:.0f} MB read per step, larger than L2"},
        "clocks": clk, "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                     "frac": achieved / float(pk["hbm_gbs"]), "traffic": None, "algorithmic_bytes_per_step": step_bytes,
                     "peak_source": f"{pk_src} HBM copy"},
    }
    print(json.dumps(line), flush=True)
    model.close()


# backward steps that gpt_backward can bracket with the probe: (name, step id, per block, kernel)
TRAIN_STEP_KINDS = [
    ("b_dz", 16, False, "gemm_tc_kernel<EPI_CE_GRAD> (recomputed logits -> cross-entropy gradient dz)"),
    ("b_dh", 17, False, "gemm_pair_kernel<EPI_BIAS_RESID> split-K (dh = dz E, CTA pairs)"),
    ("b_de", 18, False, "gemm_pair_kernel<EPI_BIAS_RESID, MN> (head share of the table gradient, dz^T h, CTA pairs)"),
    ("b_mp_w", 19, True, "gemm_pair_kernel<EPI_BIAS_RESID, MN> split-K (MLP down-projection weight gradient, CTA pairs)"),
    ("b_dg", 20, True, "gemm_tc_kernel<EPI_GELU_GRAD> (du = (dx W_mp) gelu'(u))"),
    ("b_fc_w", 21, True, "gemm_pair_kernel<EPI_BIAS_RESID, MN> split-K (MLP up-projection weight gradient, CTA pairs)"),
    ("b_da2", 22, True, "gemm_pair_kernel<EPI_F32_OUT> (du W_fc, CTA pairs)"),
    ("b_proj_w", 23, True, "gemm_pair_kernel<EPI_BIAS_RESID, MN> split-K (attention output projection weight gradient, CTA pairs)"),
    ("b_dy", 24, True, "gemm_tc_kernel<EPI_BIAS_OUT> (dy = ds1 W_proj)"),
    ("b_attn", 25, True, "attn_bwd_tc_kernel<64> + attn_bwd_dsum_kernel<64> + attn_bwd_dq_convert_kernel + memset "
                         "(causal attention derivative on tcgen05)"),
    ("b_attn_w", 26, True, "gemm_pair_kernel<EPI_BIAS_RESID, MN> split-K (QKV projection weight gradient, CTA pairs)"),
    ("b_da1", 27, True, "gemm_pair_kernel<EPI_F32_OUT> (dqkv W_attn, CTA pairs)"),
]


def train_work(name, cfg, B, T):
    """Algorithmic FLOPs of one launch of a backward step (2 per multiply-add; attention's
    derivative: the four products dP = dY U^T, dU = A^T dY, dQ = dS K, dK = dS^T Q over the
    causal pairs, 8 D per pair and head; recomputed scores are not counted)."""
    M, C, F, V = B * T, cfg.C, cfg.ffn, cfg.V
    return {"b_dz": 2.0 * M * V * C, "b_dh": 2.0 * M * V * C, "b_de": 2.0 * M * V * C,
            "b_mp_w": 2.0 * M * C * F, "b_dg": 2.0 * M * C * F, "b_fc_w": 2.0 * M * C * F, "b_da2": 2.0 * M * C * F,
            "b_proj_w": 2.0 * M * C * C, "b_dy": 2.0 * M * C * C, "b_attn": 4.0 * B * C * T * (T + 1),
            "b_attn_w": 6.0 * M * C * C, "b_da1": 6.0 * M * C * C}[name]


def train_cpu_baseline(wl, w, ids, tg, budget_s: float = 20.0):
    """The fp64 gradient oracle, as it stands, on whole sequences of the workload until about
    budget_s seconds have been spent (at least one)."""
    import oracle
    rows, spent, T = 0, 0.0, ids.shape[1]
    while rows < ids.shape[0] and (rows == 0 or spent * (rows + 1) / rows < budget_s):
        t0 = time.perf_counter()
        oracle.backward(wl.cfg, w, ids[rows:rows + 1], tg[rows:rows + 1])
        spent += time.perf_counter() - t0
        rows += 1
    return {"value": rows * T / spent, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows} sequence(s) x {T} tokens of the same workload, loss and gradients, numpy float64",
            "seconds": spent}


def run_train(args, rank, world, local_rank):
    """--train: tokens/s of a whole training step, a second measurement beside the forward line: the
    forward and loss, the gradient of every parameter (gpt_backward) and one AdamW update of every
    weight (gpt_adamw_step, lr 1e-4). FLOPs per step = 3 x the forward's (the forward, then twice its
    products for the input and weight gradients); recomputed logits and scores and the optimiser's
    elementwise work are not counted. The dominant probed step's launches are timed inside the timed
    region for the roofline."""
    import torch
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import workload
    from workloads.generate import generate

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl_name, _, wl_label = MODELS[args.model]
    wl = workload(wl_name)
    cfg = wl.cfg
    B, T = args.batch, args.seq
    w, ids_np, tg_np = generate(wl, B=B, T=T)
    model = binding.GPTModel(cfg, w, B * T)
    lib = model.lib
    ids = torch.from_numpy(ids_np).to(dev)
    tg = torch.from_numpy(tg_np).to(dev)
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    def train_step():
        model.backward(ids, tg, loss, check=False)
        n = lib.gpt_last_launch_count(model.handle)
        model.adamw_step(1e-4, 0.9, 0.95, 1e-8, 0.1)
        return n + lib.gpt_last_launch_count(model.handle)

    for _ in range(args.warmup):
        launches_per_step = train_step()
    model.status()
    rte = RuntimeEvents()
    pa, pb = rte.create(), rte.create()
    breakdown = {}
    for name, sid, per_block, _ in TRAIN_STEP_KINDS:
        times = []
        for layer in (range(cfg.L) if per_block else [-1]):
            lib.gpt_time_step(model.handle, sid, layer, pa, pb)
            model.backward(ids, tg, loss, check=False)
            hits = lib.gpt_last_probe_hits(model.handle)
            model.adamw_step(1e-4, 0.9, 0.95, 1e-8, 0.1)
            torch.cuda.synchronize()
            if hits == 1:
                times.append(rte.elapsed_ms(pa, pb))
        if times:
            breakdown[name] = {"launches_per_step": len(times), "avg_ms": statistics.mean(times),
                               "ms_per_step": sum(times), "work": train_work(name, cfg, B, T)}
    lib.gpt_time_step(model.handle, -1, -1, None, None)
    dom = max(breakdown, key=lambda k: breakdown[k]["ms_per_step"])
    dom_sid, dom_pb, dom_kernel = next((sid, p_, k_) for n, sid, p_, k_ in TRAIN_STEP_KINDS if n == dom)
    dom_layer = cfg.L // 2 if dom_pb else -1

    # timed region: K steps, the dominant step's launch in block dom_layer bracketed in each
    ev0 = [rte.create() for _ in range(args.steps)]
    ev1 = [rte.create() for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for k in range(args.steps):
        lib.gpt_time_step(model.handle, dom_sid, dom_layer, ev0[k], ev1[k])
        train_step()
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    model.status()
    ms = start.elapsed_time(stop)
    dom_ms = [rte.elapsed_ms(a, b) for a, b in zip(ev0, ev1)]
    for h in ev0 + ev1 + [pa, pb]:
        rte.destroy(h)
    ms_max, value = replica_rate(ms, B * T * args.steps, world, dev)

    # e2e: ids and targets copied from pinned host memory and the loss read back inside every step
    pin_ids = torch.from_numpy(ids_np).pin_memory()
    pin_tg = torch.from_numpy(tg_np).pin_memory()
    pin_loss = torch.zeros(1, dtype=torch.float32).pin_memory()
    d_ids, d_tg = torch.empty_like(ids), torch.empty_like(tg)

    def host_step():
        d_ids.copy_(pin_ids, non_blocking=True)
        d_tg.copy_(pin_tg, non_blocking=True)
        model.backward(d_ids, d_tg, loss, check=False)
        model.adamw_step(1e-4, 0.9, 0.95, 1e-8, 0.1)
        pin_loss.copy_(loss, non_blocking=True)
        torch.cuda.synchronize()

    host_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        host_step()
    _, e2e_value = replica_rate(1e3 * (time.perf_counter() - t0), B * T * args.steps, world, dev)
    if rank != 0:
        model.close()
        return
    pk, pk_src = peaks()
    peak_t = float(pk["bf16_tflops"])          # a step of tens of ms: the burst figure
    peak_ts = float(pk.get("bf16_tflops_sustained", peak_t))
    flops = 3.0 * step_flops(cfg, B, T)
    total_ms = ms / args.steps
    kernels = []
    for name, v in sorted(breakdown.items(), key=lambda kv: -kv[1]["ms_per_step"]):
        a = v["work"] / (v["avg_ms"] / 1e3) / 1e12
        kernels.append({"step": name, "launches_per_step": v["launches_per_step"], "avg_ms": v["avg_ms"],
                        "share_of_step": v["ms_per_step"] / total_ms, "bound": "tensor", "achieved": a,
                        "unit": "TFLOP/s", "frac": a / peak_t})
    dom_avg = statistics.mean(dom_ms)
    achieved = breakdown[dom]["work"] / (dom_avg / 1e3) / 1e12
    traffic = None
    tr = TRAIN_NCU_TRAFFIC.get(dom)
    if (tr is not None and tr["bytes"] is not None and args.model == "gpt2_small" and (B, T) == (16, 1024)
            and source_digest(tr["sources"]) == tr["digest"]):
        traffic = tr["bytes"]
    cpu = None if (args.no_cpu_baseline or world > 1) else train_cpu_baseline(wl, w, ids_np, tg_np)
    line = {
        "metric": f"{wl_label.split('_b')[0]} training forward+backward tokens/sec on 1 GB300", "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.model}_train_b{B}_t{T}", "B": B, "T": T, "V": cfg.V, "C": cfg.C, "H": cfg.H,
                   "L": cfg.L, "ids": "zipf(1.1) seed 4", "l2": "inputs larger than L2 (weights and activations)",
                   "step": "forward + loss + gradient of every parameter + AdamW update",
                   "parallelism": f"replicas x{world}"},
        "tflops": flops * args.steps * world / (ms_max / 1e3) / 1e12,
        "frac_of_peak": flops / (ms_max / args.steps / 1e3) / 1e12 / float(pk["bf16_tflops"]),
        "peak_source": f"{pk_src} bf16 {pk['bf16_tflops']} TFLOP/s burst",
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * B * T * 4, "d2h_bytes_per_step": 4},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": dom_kernel, "step": dom, "bound": "tensor", "achieved": achieved, "peak": peak_t,
                     "unit": "TFLOP/s", "frac": achieved / peak_t, "traffic": traffic,
                     "algorithmic": breakdown[dom]["work"], "peak_source": f"{pk_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_ts,
                     "avg_launch_ms": dom_avg, "launches_timed": len(dom_ms)},
        "kernels": kernels,
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
    ap.add_argument("--model", choices=sorted(MODELS), default="gpt2_small")
    ap.add_argument("--decode", action="store_true", help="time incremental decoding instead of the forward")
    ap.add_argument("--train", action="store_true", help="time forward + backward (gpt_backward) instead")
    ap.add_argument("--prompt", type=int, default=512, help="--decode: prompt length before the timed steps")
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
    if args.decode:
        if rank == 0:
            run_decode(args, rank, world, local_rank)
    elif args.train:
        run_train(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
