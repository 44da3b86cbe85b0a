"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each test ties an oracle function to something other than itself: a value the
pages print (tests/golden/pages_pins.json), a closed form, an invariant, brute
force on tiny inputs, or an independent library routine (torch, scipy, math).
The planted-mistake tests at the end check that plausible errors in the oracle
would be caught by these pins.
"""
import itertools
import json
import math
import os
import statistics

import numpy as np
import pytest

import oracle
from oracle import gpt_oracle as go
from workloads import GPTConfig, generate, workload, POST_NORM, GELU_ERF, DT_FP32
from workloads.generate import make_weights, make_tokens

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_pins.json")))


def _cfg(**kw):
    base = dict(V=17, C=16, H=2, L=2, ctx=12, ffn=64, dtype=DT_FP32)
    base.update(kw)
    return GPTConfig(**base)


def _rand_model(cfg, seed=0, affine="random", wstd=0.02):
    rng = np.random.Generator(np.random.PCG64(seed))
    return make_weights(cfg, rng, affine=affine, wstd=wstd), rng


# ---------------------------------------------------------------- parameter count

@pytest.mark.parametrize("case", GOLDEN["param_counts"], ids=lambda c: str(c["value"]))
def test_param_count_printed(case):
    cfg = GPTConfig(V=case["V"], C=case["C"], H=case["H"], L=case["L"], ctx=case["ctx"], ffn=case["ffn"])
    assert go.param_count(cfg) == case["value"], case["cite"]


def test_untied_head_extra():
    g = GOLDEN["untied_extra"]
    cfg = GPTConfig(V=g["V"], C=g["C"], H=12, L=12, ctx=1024, ffn=3072)
    assert go.param_count(cfg, tied=False) - go.param_count(cfg) == g["value"], g["cite"]


def test_param_count_closed_form():
    # per block (4C^2+4C) + (8C^2+5C) + 4C = 12C^2+13C; plus VC + ctx*C + 2C
    pb = GOLDEN["per_block"]
    for V, C, L, ctx in [(50257, 768, 12, 1024), (17, 16, 2, 12), (5000, 128, 4, 128), (31, 40, 3, 7)]:
        cfg = GPTConfig(V=V, C=C, H=4, L=L, ctx=ctx, ffn=4 * C)
        per_block = (pb["attn_quad"] + pb["mlp_quad"]) * C * C + (pb["attn_lin"] + pb["mlp_lin"] + pb["ln_lin"]) * C
        assert go.param_count(cfg) == L * per_block + V * C + ctx * C + 2 * C


def test_param_count_gpt1_about_117m():
    g = GOLDEN["gpt1_post_norm_params_approx"]
    cfg = workload("gpt1_postnorm").cfg
    n = go.param_count(cfg)
    assert n == 116_167_680
    assert abs(n / 1e6 - g["value_millions"]) / g["value_millions"] < 0.01, g["cite"]


def test_param_count_gpt2_xl_about_1_5b():
    # the page rounds 1,557,611,200 (tied head, ctx 1024) to "1.5B"; its FFN width is 4C
    g = GOLDEN["gpt2_xl_shape"]
    cfg = workload("gpt2_xl").cfg
    assert (cfg.V, cfg.C, cfg.H, cfg.L, cfg.ffn) == (g["V"], g["C"], g["H"], g["L"], g["ffn"]), g["cite"]
    assert cfg.ffn == 4 * cfg.C and cfg.C // cfg.H == 64
    n = go.param_count(cfg)
    assert n == 48 * (12 * 1600 ** 2 + 13 * 1600) + 50257 * 1600 + 1024 * 1600 + 2 * 1600 == 1_557_611_200
    assert abs(n / 1e9 - g["value_billions"]) / g["value_billions"] < 0.05, g["cite"]
    e = GOLDEN["gpt2_xl_embedding_params_approx"]
    assert abs(e["V"] * e["C"] / 1e6 - e["value_millions"]) / e["value_millions"] < 0.01, e["cite"]


def test_kv_values_per_token():
    g = GOLDEN["kv_values_per_token"]
    assert 2 * g["L"] * g["H"] * g["D"] == g["value"]


# ---------------------------------------------------------------- shape walks

@pytest.mark.parametrize("walk", GOLDEN["shape_walks"], ids=lambda w: w["cite"][:12])
def test_shape_walk(walk):
    B, T, C, H = walk["B"], walk["T"], walk["C"], walk["H"]
    D = C // H
    rng = np.random.default_rng(0)
    a = rng.standard_normal((B, T, C))
    qkv = go.linear(a, rng.standard_normal((3 * C, C)), np.zeros(3 * C))
    if "c_attn" in walk:
        assert list(qkv.shape) == walk["c_attn"]
        assert list(qkv[..., :C].shape) == walk["split"]
    q = qkv[..., :C].reshape(B, T, H, D).transpose(0, 2, 1, 3)
    k = qkv[..., C:2 * C].reshape(B, T, H, D).transpose(0, 2, 1, 3)
    if "heads" in walk:
        assert list(q.shape) == walk["heads"]
    assert list(go.attention_probs(q, k).shape) == walk["scores"]
    y = go.causal_self_attention(qkv, H)
    assert list(y.shape) == [B, T, C]
    if "logits" in walk:
        cfg = GPTConfig(V=walk["V"], C=C, H=H, L=walk["L"], ctx=128, ffn=4 * C, dtype=DT_FP32)
        w, _ = _rand_model(cfg, affine="init")
        ids = rng.integers(0, walk["V"], size=walk["ids"])
        assert list(go.embed(w["wte"], w["wpe"], ids).shape) == walk["embed"]
        _, logits = go.forward(cfg, w, ids)
        assert list(logits.shape) == walk["logits"]


# ---------------------------------------------------------------- loss special cases

@pytest.mark.parametrize("V", [17, 5000, 50257, 40000])
def test_zero_weights_give_ln_v(V):
    cfg = GPTConfig(V=V, C=16, H=2, L=2, ctx=8, ffn=64, dtype=DT_FP32)
    w, rng = _rand_model(cfg, affine="init")
    w["wte"][:] = 0
    w["wpe"][:] = 0
    for p in w["layers"]:
        for k in ("attn_w", "proj_w", "fc_w", "mp_w"):
            p[k][:] = 0
    ids = rng.integers(0, V, size=(2, 8))
    tg = rng.integers(0, V, size=(2, 8))
    loss, logits = go.forward(cfg, w, ids, tg)
    assert np.all(logits == 0.0)
    assert abs(loss - math.log(V)) < 1e-12


def test_initial_loss_near_ln_v_printed():
    g = GOLDEN["initial_loss"]
    cfg = GPTConfig(V=g["V"], C=128, H=4, L=4, ctx=64, ffn=512, dtype=DT_FP32)
    w, rng = _rand_model(cfg, affine="init")
    ids, tg = make_tokens(cfg.V, 2, 64, rng)
    loss, _ = go.forward(cfg, w, ids, tg)
    assert abs(loss - g["value"]) < 0.1, g["cite"]
    assert abs(math.log(g["V"]) - g["value"]) < g["tol"]


@pytest.mark.parametrize("name", ["toy", "minigpt"])
def test_workload_initial_loss_near_ln_v(name):
    wl = workload(name)
    w, ids, tg = generate(wl)
    loss, _ = go.forward(wl.cfg, w, ids, tg)
    assert abs(loss - math.log(wl.cfg.V)) < 0.05


def test_cross_entropy_vs_scipy():
    from scipy.special import logsumexp
    rng = np.random.default_rng(3)
    z = rng.standard_normal((7, 33)) * 5
    y = rng.integers(0, 33, size=7)
    ref = np.mean([logsumexp(z[i]) - z[i, y[i]] for i in range(7)])
    assert abs(go.cross_entropy(z, y) - ref) < 1e-12
    with pytest.raises(ValueError):
        go.cross_entropy(z, np.full(7, 33))


def test_cross_entropy_uniform_and_peaked():
    z = np.zeros((3, 11))
    assert abs(go.cross_entropy(z, np.array([0, 5, 10])) - math.log(11)) < 1e-14
    z = np.full((1, 4), -1000.0)
    z[0, 2] = 1000.0
    assert go.cross_entropy(z, np.array([2])) == 0.0


# ---------------------------------------------------------------- LayerNorm and GELU

def test_layernorm_constant_row_gives_beta():
    g = np.array([1.5, -2.0, 0.3, 4.0])
    b = np.array([0.1, 0.2, -0.3, 0.4])
    y = go.layernorm(np.full((2, 4), 3.25), g, b)
    assert np.array_equal(y, np.broadcast_to(b, (2, 4)))


def test_layernorm_moments_closed_form():
    row = [0.5, -1.25, 2.0, 3.5, -0.75, 0.0]
    var = statistics.pvariance(row)             # biased variance, independent routine
    eps = 1e-5
    y = go.layernorm(np.array([row]), np.ones(6), np.zeros(6), eps)[0]
    assert abs(y.mean()) < 1e-14
    assert abs((y ** 2).mean() - var / (var + eps)) < 1e-14


def test_layernorm_vs_torch():
    import torch
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 24)) * 3 + 1
    g = rng.standard_normal(24)
    b = rng.standard_normal(24)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (24,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.max(np.abs(go.layernorm(x, g, b) - ref)) < 1e-13


def test_gelu_tanh_against_exact_gelu():
    x = np.linspace(-6, 6, 2401)
    exact = np.array([v * 0.5 * (1 + math.erf(v / math.sqrt(2))) for v in x])
    d = np.abs(go.gelu(x) - exact)
    assert d.max() < 1e-3          # the tanh form approximates x*Phi(x) closely ...
    assert d.max() > 1e-5          # ... but is not identical to it
    assert go.gelu(np.array([0.0]))[0] == 0.0
    assert abs(go.gelu(np.array([10.0]))[0] - 10.0) < 1e-12
    assert abs(go.gelu(np.array([-10.0]))[0]) < 1e-12


@pytest.mark.parametrize("mode,approx", [(0, "tanh"), (GELU_ERF, "none")])
def test_gelu_vs_torch(mode, approx):
    import torch
    x = np.linspace(-8, 8, 1001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate=approx).numpy()
    assert np.max(np.abs(go.gelu(x, mode) - ref)) < 1e-13


# ---------------------------------------------------------------- linear orientation

def test_linear_orientation_asymmetric():
    # "第 25 章" §25.5: a Conv1D weight W_conv [in,out] computes X W_conv; the
    # Linear weight is its transpose. An asymmetric square matrix tells them apart.
    rng = np.random.default_rng(2)
    X = rng.standard_normal((3, 4))
    W_conv = rng.standard_normal((4, 4))
    ref = np.array([[sum(X[i, k] * W_conv[k, j] for k in range(4)) for j in range(4)] for i in range(3)])
    assert np.max(np.abs(go.linear(X, W_conv.T) - ref)) < 1e-13
    assert np.max(np.abs(go.linear(X, W_conv) - ref)) > 1e-3


# ---------------------------------------------------------------- embedding and head

def test_embed_brute_force():
    rng = np.random.default_rng(4)
    E = rng.standard_normal((9, 5))
    P = rng.standard_normal((6, 5))
    ids = rng.integers(0, 9, size=(2, 4))
    x = go.embed(E, P, ids)
    for b, t, c in itertools.product(range(2), range(4), range(5)):
        assert x[b, t, c] == E[ids[b, t], c] + P[t, c]
    with pytest.raises(ValueError):
        go.embed(E, P, np.array([[9]]))
    with pytest.raises(ValueError):
        go.embed(E, P, np.zeros((1, 7), int))     # T > ctx


def test_tied_head_identity():
    cfg = _cfg()
    w, rng = _rand_model(cfg)
    ids = rng.integers(0, cfg.V, size=(2, 6))
    h = go.forward_hidden(cfg, w, ids)
    _, logits = go.forward(cfg, w, ids)
    for (b, t, j) in [(0, 0, 0), (1, 5, 16), (0, 3, 7), (1, 2, 11)]:
        dot = math.fsum(float(h[b, t, c]) * float(w["wte"][j, c]) for c in range(cfg.C))
        assert abs(logits[b, t, j] - dot) < 1e-13


def test_zero_layers_closed_form():
    # L=0, P=0, E = s*I (V=C): x0 = s*e_id; ln_f (gain 1, shift 0) then E^T gives
    # logit j = s*(s*[j==id] - s/C) / sqrt(s^2 (C-1)/C^2 + eps)
    C = 8
    s = 3.0
    eps = 1e-5
    cfg = GPTConfig(V=C, C=C, H=2, L=0, ctx=4, ffn=4 * C, dtype=DT_FP32, ln_eps=eps)
    w = {"wte": s * np.eye(C), "wpe": np.zeros((4, C)), "layers": [],
         "lnf_g": np.ones(C), "lnf_b": np.zeros(C)}
    ids = np.array([[3, 0, 7, 3]])
    _, logits = go.forward(cfg, w, ids)
    den = math.sqrt(s * s * (C - 1) / C ** 2 + eps)
    for t in range(4):
        for j in range(C):
            ref = s * (s * (j == ids[0, t]) - s / C) / den
            assert abs(logits[0, t, j] - ref) < 1e-12


# ---------------------------------------------------------------- attention

def _brute_attention(qkv, H):
    """Per query position, per head, per allowed key: explicit loops."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    D = C // H
    y = np.zeros((B, T, C))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                q = [qkv[b, t, h * D + d] for d in range(D)]
                sc = []
                for s in range(t + 1):
                    k = [qkv[b, s, C + h * D + d] for d in range(D)]
                    sc.append(math.fsum(q[d] * k[d] for d in range(D)) / math.sqrt(D))
                m = max(sc)
                e = [math.exp(v - m) for v in sc]
                z = math.fsum(e)
                for d in range(D):
                    y[b, t, h * D + d] = math.fsum(e[s] / z * qkv[b, s, 2 * C + h * D + d] for s in range(t + 1))
    return y


@pytest.mark.parametrize("B,T,H,D", [(2, 12, 2, 4), (1, 7, 3, 2), (2, 1, 2, 8)])
def test_attention_brute_force(B, T, H, D):
    rng = np.random.default_rng(5)
    qkv = rng.standard_normal((B, T, 3 * H * D)) * 2.0
    assert np.max(np.abs(go.causal_self_attention(qkv, H) - _brute_attention(qkv, H))) < 1e-13


def test_attention_rows_sum_to_one_and_causal():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, 10, 4)) * 4
    k = rng.standard_normal((3, 10, 4)) * 4
    A = go.attention_probs(q, k)
    assert np.max(np.abs(A.sum(-1) - 1)) < 1e-14
    assert np.all(A[:, np.triu_indices(10, 1)[0], np.triu_indices(10, 1)[1]] == 0)
    assert np.all(A[:, 0, 0] == 1.0)


def test_attention_t1_returns_u0():
    rng = np.random.default_rng(7)
    qkv = rng.standard_normal((2, 1, 24))
    assert np.array_equal(go.causal_self_attention(qkv, 2), qkv[..., 16:24])


def test_causal_invariance():
    cfg = _cfg(L=2)
    w, rng = _rand_model(cfg, wstd=0.3)
    ids = rng.integers(0, cfg.V, size=(2, 12))
    _, z0 = go.forward(cfg, w, ids)
    for t in (0, 4, 10):
        ids2 = ids.copy()
        ids2[:, t + 1:] = (ids2[:, t + 1:] + 5) % cfg.V
        _, z1 = go.forward(cfg, w, ids2)
        assert np.max(np.abs(z1[:, :t + 1] - z0[:, :t + 1])) < 1e-12
        if t + 1 < 12:
            assert np.max(np.abs(z1[:, t + 1:] - z0[:, t + 1:])) > 1e-6


# ---------------------------------------------------------------- whole model vs library routines

@pytest.mark.parametrize("variant", ["pre", "post", "erf", "toy_workload"])
def test_forward_vs_torch_functional(variant):
    import torch_ref
    if variant == "toy_workload":
        wl = workload("toy")
        cfg = wl.cfg
        w, ids, tg = generate(wl, affine="random")
    else:
        kw = {"post": dict(norm_mode=POST_NORM, final_ln=0), "erf": dict(gelu=GELU_ERF), "pre": {}}[variant]
        cfg = _cfg(C=24, H=3, L=3, V=29, ctx=10, ffn=96, **kw)
        w, rng = _rand_model(cfg, seed=11, wstd=0.25)
        ids, tg = make_tokens(cfg.V, 3, 10, rng)
    loss, z = go.forward(cfg, w, ids, tg)
    rloss, rz = torch_ref.forward(cfg, w, ids, tg)
    assert np.max(np.abs(z - rz)) < 1e-10
    assert abs(loss - rloss) < 1e-12


def test_config_errors():
    cfg = _cfg(C=16, H=3)
    w, rng = _rand_model(_cfg())
    with pytest.raises(ValueError):
        go.forward(cfg, w, np.zeros((1, 4), int))
    with pytest.raises(ValueError):
        go.forward(_cfg(), w, np.zeros((1, 13), int))   # T=13 > ctx=12


# ---------------------------------------------------------------- planted mistakes

def _pins_pass():
    """Run the structural pins against whatever go.* currently is."""
    try:
        test_attention_brute_force(2, 6, 2, 4)
        test_layernorm_moments_closed_form()
        test_gelu_tanh_against_exact_gelu()
        test_forward_vs_torch_functional("pre")
        test_forward_vs_torch_functional("post")
        test_tied_head_identity()
        test_zero_layers_closed_form()
    except AssertionError:
        return False
    return True


def test_pins_pass_on_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("mistake", ["no_scale", "k_for_q", "unbiased_var", "gelu_const",
                                     "no_residual", "w_untransposed", "mask_off_by_one", "head_bias"])
def test_planted_mistakes_are_caught(mistake, monkeypatch):
    orig_probs = go.attention_probs
    orig_ln = go.layernorm
    orig_gelu = go.gelu
    orig_lin = go.linear
    orig_attn = go.causal_self_attention
    orig_head = go.lm_head
    if mistake == "no_scale":
        monkeypatch.setattr(go, "attention_probs", lambda q, k: orig_probs(q * math.sqrt(q.shape[-1]), k))
    elif mistake == "k_for_q":
        def swapped(qkv, H):
            C = qkv.shape[-1] // 3
            q2 = qkv.copy()
            q2[..., :C], q2[..., C:2 * C] = qkv[..., C:2 * C], qkv[..., :C]
            return orig_attn(q2, H)
        monkeypatch.setattr(go, "causal_self_attention", swapped)
    elif mistake == "unbiased_var":
        def ln(x, g, b, eps=1e-5):
            x = np.asarray(x, np.float64)
            return g * (x - x.mean(-1, keepdims=True)) / np.sqrt(x.var(-1, ddof=1, keepdims=True) + eps) + b
        monkeypatch.setattr(go, "layernorm", ln)
    elif mistake == "gelu_const":
        monkeypatch.setattr(go, "gelu", lambda x, mode=0: 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.44715 * x ** 3))))
    elif mistake == "no_residual":
        def blk(x, p, cfg):
            x = go._attn_branch(orig_ln(x, p["ln1_g"], p["ln1_b"], cfg.ln_eps), p, cfg)
            return x + go._mlp_branch(orig_ln(x, p["ln2_g"], p["ln2_b"], cfg.ln_eps), p, cfg)
        monkeypatch.setattr(go, "block_pre_norm", blk)
    elif mistake == "w_untransposed":
        monkeypatch.setattr(go, "linear", lambda x, w, b=None: orig_lin(x, np.asarray(w).T if np.asarray(w).shape[0] == np.asarray(w).shape[1] else w, b))
    elif mistake == "mask_off_by_one":
        def probs(q, k):
            T = q.shape[-2]
            sc = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(q.shape[-1])
            allowed = np.tril(np.ones((T, T), bool), k=-1) | (np.arange(T)[:, None] == 0) & (np.arange(T)[None, :] == 0)
            sc = np.where(allowed, sc, -np.inf)
            e = np.where(allowed, np.exp(sc - sc.max(-1, keepdims=True)), 0)
            return e / e.sum(-1, keepdims=True)
        monkeypatch.setattr(go, "attention_probs", probs)
    elif mistake == "head_bias":
        monkeypatch.setattr(go, "lm_head", lambda h, wte: orig_head(h, wte) + 0.01)
    assert not _pins_pass(), f"planted mistake {mistake} went unnoticed"


# ---- next-token sampling ("预训练一个 Mini GPT" 第7步; "02 GPT 架构" 8.1-8.3)

def test_sample_greedy_is_argmax():
    rng = np.random.default_rng(3)
    z = rng.standard_normal(1000)
    for u in (0.0, 0.5, 0.999):
        assert go.sample_next(z, 0.0, 0, 1.0, u)[0] == int(np.argmax(z))
        assert go.sample_next(z, 1.3, 1, 1.0, u)[0] == int(np.argmax(z))      # top-k = 1
        assert go.sample_next(z, 0.7, 0, 1e-9, u)[0] == int(np.argmax(z))     # a nucleus of one token


def test_sample_plain_is_inverse_cdf():
    # no filter: the draw is the inverse CDF of softmax(z / T) in index order (np.random.choice's rule)
    rng = np.random.default_rng(4)
    z = rng.standard_normal(300) * 2
    T = 0.8
    p = np.exp(z / T - np.max(z / T))
    p /= p.sum()
    cdf = np.cumsum(p)
    for u in rng.random(50):
        assert go.sample_next(z, T, 0, 1.0, u)[0] == int(np.searchsorted(cdf, u, side="right"))


def test_sample_worked_nucleus_and_top_k():
    # p = (0.5, 0.3, 0.2): top-p 0.75 keeps tokens 0 and 1 (0.5 < 0.75 <= 0.8), renormalised to
    # (0.625, 0.375); top-k 2 keeps the same two
    z = np.log(np.array([0.5, 0.3, 0.2]))
    for kw in (dict(top_k=0, top_p=0.75), dict(top_k=2, top_p=1.0)):
        i0, q = go.sample_next(z, 1.0, kw["top_k"], kw["top_p"], 0.6)
        assert i0 == 0 and np.allclose(q, [0.625, 0.375, 0.0])
        assert go.sample_next(z, 1.0, kw["top_k"], kw["top_p"], 0.7)[0] == 1
    # top-p 0.85 needs all three (0.8 < 0.85)
    assert go.sample_next(z, 1.0, 0, 0.85, 0.95)[0] == 2


def test_sample_ties_and_temperature():
    z = np.array([2.0, 2.0, 1.0])
    assert go.sample_next(z, 1.0, 1, 1.0, 0.99)[0] == 0          # equal maxima: the lower index
    assert go.sample_next(z, 0.0, 0, 1.0, 0.99)[0] == 0
    # a very high temperature flattens the distribution: CDF (0.25, 0.5, 0.75, 1)
    z4 = np.array([0.3, -1.0, 2.0, 0.5])
    assert go.sample_next(z4, 1e9, 0, 1.0, 0.5)[0] == 2
    assert go.sample_next(z4, 1e9, 0, 1.0, 0.49)[0] == 1
