"""fp64 CPU oracle of the GPT forward pass, next-token cross-entropy and its gradient.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(the CUDA library and its Python binding) never calls it, and it shares no
code with the CUDA path: the two meet only in the seeded input generators of
the ``workloads`` package.
"""
from .gpt_oracle import (
    param_count, linear, layernorm, gelu, embed, attention_probs,
    causal_self_attention, block_pre_norm, block_post_norm, forward_hidden,
    lm_head, cross_entropy_rows, cross_entropy, forward, sample_next,
)
from .gpt_grad import (
    linear_backward, layernorm_backward, gelu_backward, attention_backward,
    causal_self_attention_backward, cross_entropy_backward, embed_backward, backward, adamw_step,
)

__all__ = [
    "param_count", "linear", "layernorm", "gelu", "embed", "attention_probs",
    "causal_self_attention", "block_pre_norm", "block_post_norm", "forward_hidden",
    "lm_head", "cross_entropy_rows", "cross_entropy", "forward", "sample_next",
    "linear_backward", "layernorm_backward", "gelu_backward", "attention_backward",
    "causal_self_attention_backward", "cross_entropy_backward", "embed_backward", "backward", "adamw_step",
]
