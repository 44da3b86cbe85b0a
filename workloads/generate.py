"""Seeded weight and token generators.

Init recipe ("第 25 章 从小 GPT 到 GPT-2" §25.6; "预训练一个 Mini GPT" 第1步):
N(0, 0.02) for the token table, the position table and every linear weight,
biases 0, LayerNorm gain 1 and shift 0; on the GPT-2-small workloads the two
residual-branch projections (attention c_proj and MLP c_proj) are scaled by
1/sqrt(2L). §25.6 notes that the order of draws changes the values, so the
order here is fixed and ours: wte, wpe, then per block ln1, attn_w, attn_b,
proj_w, proj_b, ln2, fc_w, fc_b, mp_w, mp_b, then ln_f, then token ids.
Tensors that are constant at init (biases, LayerNorm) draw nothing unless
``affine="random"`` asks for random biases and LayerNorm parameters, which the
tests use so that a dropped bias or gain cannot go unnoticed.

Samples are drawn in fp32 from numpy.random.Generator(PCG64(seed)); on bf16
workloads every weight is then rounded to the nearest bf16 (ties to even) and
kept as fp32, so the oracle and the GPU consume identical values.
"""
import math
from typing import Dict, Optional, Tuple

import numpy as np

from .configs import GPTConfig, Workload, DT_BF16, layer_shapes

WEIGHT_ORDER = ("wte", "wpe", "layers", "lnf")


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    a = np.array(a, dtype=np.float32, copy=True, order="C")
    assert np.isfinite(a).all()
    u = a.view(np.uint32)          # finite inputs: the sums below stay under 2**32
    lsb = u >> 16
    lsb &= 1
    u += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return a


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def make_weights(cfg: GPTConfig, rng: np.random.Generator, scale_cproj: bool = False,
                 affine: str = "init", wstd: float = 0.02) -> Dict[str, object]:
    """Draw a full weight set. Returns {'wte','wpe','layers':[{...}],'lnf_g','lnf_b'} (+ 'head' when untied)."""
    V, C, L, ctx = cfg.V, cfg.C, cfg.L, cfg.ctx
    w: Dict[str, object] = {}
    w["wte"] = _normal(rng, (V, C), wstd)
    w["wpe"] = _normal(rng, (ctx, C), wstd)
    proj_std = wstd / math.sqrt(2 * L) if (scale_cproj and L > 0) else wstd
    layers = []
    for _ in range(L):
        p = {}
        for name, shape in layer_shapes(cfg):
            if name.endswith("_w"):
                std = proj_std if name in ("proj_w", "mp_w") else wstd
                p[name] = _normal(rng, shape, std)
            elif name in ("ln1_g", "ln2_g"):
                p[name] = (np.ones(shape, np.float32) if affine == "init"
                           else (1.0 + _normal(rng, shape, 0.1)).astype(np.float32))
            else:  # biases and LayerNorm shifts
                p[name] = (np.zeros(shape, np.float32) if affine == "init"
                           else _normal(rng, shape, 0.02))
        layers.append(p)
    w["layers"] = layers
    if affine == "init":
        w["lnf_g"] = np.ones((C,), np.float32)
        w["lnf_b"] = np.zeros((C,), np.float32)
    else:
        w["lnf_g"] = (1.0 + _normal(rng, (C,), 0.1)).astype(np.float32)
        w["lnf_b"] = _normal(rng, (C,), 0.02)
    if cfg.untied_head:                      # drawn last, so tied models' draws are unchanged
        w["head"] = _normal(rng, (V, C), wstd)
    if cfg.dtype == DT_BF16:
        w["wte"] = round_to_bf16(w["wte"])
        w["wpe"] = round_to_bf16(w["wpe"])
        if cfg.untied_head:
            w["head"] = round_to_bf16(w["head"])
        for p in layers:
            for k in ("attn_w", "proj_w", "fc_w", "mp_w"):
                p[k] = round_to_bf16(p[k])
    return w


def make_tokens(V: int, B: int, T: int, rng: np.random.Generator, ids: str = "uniform",
                targets: str = "shifted", zipf_s: float = 1.1) -> Tuple[np.ndarray, np.ndarray]:
    """Token ids [B,T] and next-token targets [B,T], int32.

    "shifted": one stream of T+1 ids per row, inputs s[:T] and targets s[1:]
    ("第 25 章" §25.7: x=[0,1,2,3], y=[1,2,3,4]); "uniform": independent draws.
    Zipf ids: k ~ Zipf(s) (k >= 1), id = min(k-1, V-1), so id 0 is the commonest.
    """
    n = T + 1 if targets == "shifted" else T

    def draw(shape):
        if ids == "zipf":
            k = rng.zipf(zipf_s, size=shape)
            return np.minimum(k - 1, V - 1).astype(np.int32)
        return rng.integers(0, V, size=shape, dtype=np.int64).astype(np.int32)

    s = draw((B, n))
    if targets == "shifted":
        return np.ascontiguousarray(s[:, :T]), np.ascontiguousarray(s[:, 1:])
    return s, draw((B, T))


def generate(wl: Workload, B: Optional[int] = None, T: Optional[int] = None,
             affine: str = "init", seed: Optional[int] = None, wstd: float = 0.02):
    """Weights, ids and targets of a workload, all from one seeded generator."""
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    w = make_weights(wl.cfg, rng, wl.scale_cproj, affine=affine, wstd=wstd)
    ids, tg = make_tokens(wl.cfg.V, B, T, rng, wl.ids, wl.targets, wl.zipf_s)
    return w, ids, tg
