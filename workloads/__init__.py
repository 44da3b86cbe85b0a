"""Seeded synthetic workloads: model configurations, weights and token ids.

This module is shared by the fp64 oracle and by the CUDA path. It holds no
arithmetic of the forward pass itself: it only draws numbers (normal weights,
uniform or Zipf token ids) and, for bf16 workloads, rounds the drawn fp32
weights to the nearest bf16 value so that both sides consume bit-identical
parameters.
"""
from .configs import GPTConfig, WORKLOADS, workload, PRE_NORM, POST_NORM, GELU_TANH, GELU_ERF, DT_FP32, DT_BF16
from .generate import make_weights, make_tokens, round_to_bf16, generate, WEIGHT_ORDER

__all__ = [
    "GPTConfig", "WORKLOADS", "workload", "PRE_NORM", "POST_NORM", "GELU_TANH",
    "GELU_ERF", "DT_FP32", "DT_BF16", "make_weights", "make_tokens",
    "round_to_bf16", "generate", "WEIGHT_ORDER",
]
