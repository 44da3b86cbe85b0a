"""Time one step kernel of the library in isolation (CUDA events, warm-up, mean of N).

    python kbench.py attention --B 16 --T 1024 --H 12 --D 64
    python kbench.py attention_bwd --B 16 --T 1024 --H 12 --D 64
    python kbench.py gemm --M 16384 --N 768 --K 768 --epi 2
    python kbench.py gemm --M 16384 --N 768 --K 3072 --pair
    python kbench.py head --M 16384 --V 50257 --C 768
    python kbench.py layernorm --M 16384 --C 768
    python kbench.py train --B 16 --T 1024
    python kbench.py forward --B 16 --T 1024

(`train`: one gpt_backward call, forward + loss + every gradient, of GPT-2 small on
seeded synthetic tokens; `forward`: one gpt_forward call, forward + loss, on the same. `attention_bwd`: one gptk_attention_bwd call, the attention
derivative's memset and three kernels, after one gptk_attention_lse for its inputs.)

Inputs are random device tensors; the figure printed is algorithmic TFLOP/s
(or GB/s for the row-wise kernels) over the mean launch time.
"""
import argparse
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from decoder_only_transformer_gpt_gb300 import binding  # noqa: E402


def _time(fn, warmup, iters):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    binding.status()
    return sum(a.elapsed_time(b) for a, b in evs) / iters


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["attention", "attention_bwd", "gemm", "head", "layernorm", "train", "forward"])
    ap.add_argument("--B", type=int, default=16)
    ap.add_argument("--T", type=int, default=1024)
    ap.add_argument("--H", type=int, default=12)
    ap.add_argument("--D", type=int, default=64)
    ap.add_argument("--M", type=int, default=16384)
    ap.add_argument("--N", type=int, default=768)
    ap.add_argument("--K", type=int, default=768)
    ap.add_argument("--V", type=int, default=50257)
    ap.add_argument("--C", type=int, default=768)
    ap.add_argument("--epi", type=int, default=0)
    ap.add_argument("--pair", action="store_true", help="gemm: the residual product on CTA pairs (gptk_gemm_pair)")
    ap.add_argument("--ksplit", type=int, default=0, help="gemm --pair: K slices (no bias when > 1)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--iters", type=int, default=10)
    a = ap.parse_args()
    binding.load()
    torch.manual_seed(0)
    dev = "cuda"
    if a.kernel == "attention":
        C = a.H * a.D
        qkv = torch.randn(a.B, a.T, 3 * C, device=dev).to(torch.bfloat16)
        y = torch.empty(a.B, a.T, C, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda: binding.attention(qkv, y, a.H), a.warmup, a.iters)
        flop = 2.0 * C * a.T * (a.T + 1) * a.B
        out = {"kernel": "attention", "shape": [a.B, a.T, a.H, a.D], "ms": ms, "tflops": flop / ms / 1e9}
    elif a.kernel == "attention_bwd":
        C = a.H * a.D
        qkv = torch.randn(a.B, a.T, 3 * C, device=dev).to(torch.bfloat16)
        dy = (0.25 * torch.randn(a.B, a.T, C, device=dev)).to(torch.bfloat16)
        y = torch.empty(a.B, a.T, C, device=dev, dtype=torch.bfloat16)
        lse2 = torch.empty(a.B * a.H * a.T, device=dev)
        binding.attention_lse(qkv, y, lse2, a.H)
        dqkv = torch.empty(a.B, a.T, 3 * C, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda: binding.attention_bwd(qkv, y, dy, lse2, dqkv, a.H), a.warmup, a.iters)
        flop = 4.0 * C * a.T * (a.T + 1) * a.B         # dP, dU, dK, dQ over the causal half
        out = {"kernel": "attention_bwd", "shape": [a.B, a.T, a.H, a.D], "ms": ms, "tflops": flop / ms / 1e9}
    elif a.kernel == "gemm":
        A = torch.randn(a.M, a.K, device=dev).to(torch.bfloat16)
        W = (0.05 * torch.randn(a.N, a.K, device=dev)).to(torch.bfloat16)
        bias = torch.randn(a.N, device=dev)
        odt = torch.bfloat16 if a.epi in (0, 1) else torch.float32
        out_t = torch.zeros(a.M, a.N, device=dev, dtype=odt)
        if a.pair:
            out_t = torch.zeros(a.M, a.N, device=dev, dtype=torch.float32)
            pb = bias if a.ksplit <= 1 else None
            pe = binding.EPI_F32 if a.epi == binding.EPI_F32 else binding.EPI_BIAS_RESID
            ms = _time(lambda: binding.gemm_pair(A, W, pb, out_t, a.ksplit, pe), a.warmup, a.iters)
        else:
            ms = _time(lambda: binding.gemm(A, W, bias, out_t, a.epi), a.warmup, a.iters)
        flop = 2.0 * a.M * a.N * a.K
        name = f"gemm_pair_epi{a.epi}_ks{a.ksplit}" if a.pair else f"gemm_epi{a.epi}"
        out = {"kernel": name, "shape": [a.M, a.N, a.K], "ms": ms, "tflops": flop / ms / 1e9}
    elif a.kernel == "head":
        h = torch.randn(a.M, a.C, device=dev).to(torch.bfloat16)
        E = (0.02 * torch.randn(a.V, a.C, device=dev)).to(torch.bfloat16)
        tg = torch.randint(0, a.V, (a.M,), device=dev, dtype=torch.int32)
        nll = torch.empty(a.M, device=dev)
        ms = _time(lambda: binding.lmhead_ce(h, E, tg, nll), a.warmup, a.iters)
        flop = 2.0 * a.M * a.V * a.C
        out = {"kernel": "head_ce", "shape": [a.M, a.V, a.C], "ms": ms, "tflops": flop / ms / 1e9}
    elif a.kernel in ("train", "forward"):
        from workloads import workload
        from workloads.generate import generate
        wl = workload("gpt2_small")
        w, ids, tg = generate(wl, B=a.B, T=a.T)
        m = binding.GPTModel(wl.cfg, w, a.B * a.T)
        d_ids, d_tg = torch.from_numpy(ids).to(dev), torch.from_numpy(tg).to(dev)
        loss = torch.zeros(1, device=dev)
        if a.kernel == "train":
            ms = _time(lambda: m.backward(d_ids, d_tg, loss, check=False), a.warmup, a.iters)
        else:
            ms = _time(lambda: m.forward(d_ids, d_tg, loss, None, check=False), a.warmup, a.iters)
        m.status()
        out = {"kernel": a.kernel, "shape": [a.B, a.T], "ms": ms, "tokens_per_s": a.B * a.T / ms * 1e3,
               "launches_per_call": m.lib.gpt_last_launch_count(m.handle)}
        m.close()
    else:
        x = torch.randn(a.M, a.C, device=dev)
        g = torch.ones(a.C, device=dev)
        b = torch.zeros(a.C, device=dev)
        o = torch.empty(a.M, a.C, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda: binding.layernorm(x, g, b, o), a.warmup, a.iters)
        byts = a.M * a.C * (4 + 2)
        out = {"kernel": "layernorm", "shape": [a.M, a.C], "ms": ms, "gbs": byts / ms / 1e6}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
