"""Host-side bookkeeping of bench.py (no GPU): the backward step ids it arms match the library's
header, and its algorithmic FLOP counts follow from the forward's (each backward product is one
forward product's shape; the attention derivative has twice the forward attention's products)."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import workload  # noqa: E402


def _header_enum():
    text = open(os.path.join(ROOT, "include", "gpt.h")).read()
    return {k: int(v) for k, v in re.findall(r"\b(GPT_STEP_\w+)\s*=\s*(\d+)", text)}


def test_train_step_ids_match_the_header():
    enum = _header_enum()
    for name, sid, _, _ in bench.TRAIN_STEP_KINDS:
        key = "GPT_STEP_" + name.upper()
        assert enum[key] == sid, (name, sid, enum.get(key))
    fwd_names = {"embed": "EMBED", "c_attn": "C_ATTN", "attention": "ATTN", "c_proj": "C_PROJ", "ln_mid": "LN_MID",
                 "c_fc": "C_FC", "mlp_proj": "MLP_PROJ", "ln_out": "LN_OUT", "head": "HEAD", "ce_combine": "CE",
                 "mean": "MEAN"}
    for name, sid, _ in bench.STEP_KINDS:
        assert enum["GPT_STEP_" + fwd_names[name]] == sid, name


@pytest.mark.parametrize("B,T", [(16, 1024), (2, 77)])
def test_backward_flops_are_twice_the_forward_products(B, T):
    cfg = workload("gpt2_small").cfg
    fwd = lambda n: bench.step_work(n, cfg, B, T)[0]
    bwd = lambda n: bench.train_work(n, cfg, B, T)
    block_fwd = fwd("c_attn") + fwd("c_proj") + fwd("c_fc") + fwd("mlp_proj")
    block_bwd = sum(bwd(n) for n in ("b_attn_w", "b_da1", "b_proj_w", "b_dy", "b_fc_w", "b_da2", "b_mp_w", "b_dg"))
    assert block_bwd == pytest.approx(2 * block_fwd, rel=1e-12)
    assert bwd("b_attn") == pytest.approx(2 * fwd("attention"), rel=1e-12)
    assert bwd("b_dh") + bwd("b_de") == pytest.approx(2 * fwd("head"), rel=1e-12)
