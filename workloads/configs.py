"""Model configurations and the five named workloads.

Field names follow the notation of the pages: V vocabulary size, C hidden
width, H heads (D = C/H per head), L blocks, ctx the position-table length,
ffn the MLP hidden width (4C on every workload here).

Sources:
  * "第 25 章 从小 GPT 到 GPT-2" §25.1 (GPT-2 small: L=12, C=768, H=12, ctx=1024,
    V=50257) and §25.4 (the V=17, C=16, ctx 12, 2-block toy);
  * "Day 16 从零组装 MiniGPT" §三 (MiniGPT: V=5000, max_seq 128, C=128, H=4,
    L=4, FFN 512);
  * "GPT-1 学习笔记" §3.1-3.2 (post-norm block, no final LayerNorm) and §4.1
    (context 512, 40000 BPE merges).
"""
from dataclasses import dataclass, field, replace
from typing import List, Tuple

PRE_NORM = 0
POST_NORM = 1
GELU_TANH = 0
GELU_ERF = 1
DT_FP32 = 0
DT_BF16 = 1


@dataclass(frozen=True)
class GPTConfig:
    V: int
    C: int
    H: int
    L: int
    ctx: int
    ffn: int
    norm_mode: int = PRE_NORM
    final_ln: int = 1
    gelu: int = GELU_TANH
    dtype: int = DT_BF16
    ln_eps: float = 1e-5
    untied_head: int = 0          # 1: the head has its own [V, C] matrix instead of reusing E

    @property
    def D(self) -> int:
        return self.C // self.H


@dataclass(frozen=True)
class Workload:
    """A configuration plus the batch shape and the seeded input recipe."""
    name: str
    cfg: GPTConfig
    B: int
    T: int
    seed: int
    ids: str                      # "uniform" or "zipf"
    targets: str                  # "shifted" or "uniform"
    scale_cproj: bool = False     # residual-branch projections x 1/sqrt(2L)
    zipf_s: float = 1.1
    extra_shapes: Tuple[Tuple[int, int], ...] = field(default=())

    def with_shape(self, B: int, T: int) -> "Workload":
        return replace(self, B=B, T=T)


GPT2_SMALL = GPTConfig(V=50257, C=768, H=12, L=12, ctx=1024, ffn=3072)
GPT2_XL = GPTConfig(V=50257, C=1600, H=25, L=48, ctx=1024, ffn=6400)

WORKLOADS = {
    # toy GPT-2 from the chapter-25 experiment; fp32 parity mode
    "toy": Workload("toy", GPTConfig(V=17, C=16, H=2, L=2, ctx=12, ffn=64, dtype=DT_FP32),
                    B=2, T=12, seed=0, ids="uniform", targets="uniform"),
    "minigpt": Workload("minigpt", GPTConfig(V=5000, C=128, H=4, L=4, ctx=128, ffn=512),
                        B=4, T=64, seed=1, ids="uniform", targets="shifted"),
    "gpt2_small": Workload("gpt2_small", GPT2_SMALL, B=8, T=1024, seed=2, ids="zipf",
                           targets="shifted", scale_cproj=True),
    "gpt1_postnorm": Workload("gpt1_postnorm",
                              GPTConfig(V=40000, C=768, H=12, L=12, ctx=512, ffn=3072,
                                        norm_mode=POST_NORM, final_ln=0),
                              B=16, T=512, seed=3, ids="uniform", targets="shifted"),
    "gpt2_sweep": Workload("gpt2_sweep", GPT2_SMALL, B=16, T=1024, seed=4, ids="zipf",
                           targets="shifted", scale_cproj=True,
                           extra_shapes=((1, 1024), (16, 1024), (32, 1024), (16, 777))),
    # the same path at the GPT-2 XL shape (48 blocks, C = 1600, 25 heads of 64)
    "gpt2_xl": Workload("gpt2_xl", GPT2_XL, B=16, T=1024, seed=6, ids="zipf", targets="shifted",
                        scale_cproj=True),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def layer_shapes(cfg: GPTConfig) -> List[Tuple[str, Tuple[int, ...]]]:
    """Per-block parameter names and shapes (nn.Linear orientation [out, in])."""
    C, F = cfg.C, cfg.ffn
    return [
        ("ln1_g", (C,)), ("ln1_b", (C,)),
        ("attn_w", (3 * C, C)), ("attn_b", (3 * C,)),
        ("proj_w", (C, C)), ("proj_b", (C,)),
        ("ln2_g", (C,)), ("ln2_b", (C,)),
        ("fc_w", (F, C)), ("fc_b", (F,)),
        ("mp_w", (C, F)), ("mp_b", (C,)),
    ]
