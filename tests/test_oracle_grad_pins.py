"""Pins of the fp64 gradient oracle (oracle/gpt_grad.py) to the forward oracle and to mathematics.

The gradient is pinned to the loss it differentiates: central finite differences
of ``oracle.forward``'s loss (a separate code path from the backward's own
forward) along random directions, per parameter tensor and per step, in fp64 on
tiny models. Invariances pin the structure: LayerNorm's input gradient has zero
row sums and is orthogonal to the normalised row (shift and scale invariance),
the key gradient of one head sums to zero over keys (a shift common to every
key moves each query's scores by one constant), and the head's share of the
tied table gradient has zero column sums (each row of dz sums to zero). The
planted-mistake tests show that plausible errors fail these pins.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import gpt_grad as gg
from oracle import gpt_oracle as go
from workloads import GPTConfig, POST_NORM, GELU_ERF, DT_FP32
from workloads.generate import make_weights, make_tokens

EPS = 1e-6


def _cfg(**kw):
    base = dict(V=17, C=16, H=2, L=2, ctx=12, ffn=64, dtype=DT_FP32)
    base.update(kw)
    return GPTConfig(**base)


VARIANTS = {
    "pre": {},
    "post": dict(norm_mode=POST_NORM, final_ln=0),
    "erf": dict(gelu=GELU_ERF),
    "noln_f": dict(final_ln=0),
    "untied": dict(untied_head=1),
}


def _model(cfg, seed, B=2, T=8, wstd=0.3):
    rng = np.random.Generator(np.random.PCG64(seed))
    w = make_weights(cfg, rng, affine="random", wstd=wstd)
    w64 = {k: (np.asarray(v, np.float64) if k != "layers" else [{n: np.asarray(a, np.float64) for n, a in p.items()}
                                                                 for p in v]) for k, v in w.items()}
    ids, tg = make_tokens(cfg.V, B, T, rng)
    return w64, ids, tg, rng


def _tensors(cfg, w):
    """(getter name, array) for every parameter tensor of the model."""
    out = [("wte", w["wte"]), ("wpe", w["wpe"])]
    if "head" in w:
        out.append(("head", w["head"]))
    if cfg.final_ln:
        out += [("lnf_g", w["lnf_g"]), ("lnf_b", w["lnf_b"])]
    for i, p in enumerate(w["layers"]):
        out += [(f"layers.{i}.{n}", a) for n, a in p.items()]
    return out


def _grad_of(grads, name):
    if name.startswith("layers."):
        _, i, n = name.split(".")
        return grads["layers"][int(i)][n]
    return grads[name]


def _loss(cfg, w, ids, tg):
    return go.forward(cfg, w, ids, tg)[0]


def _fd_checks(cfg, w, ids, tg, rng, tol=1e-7):
    """Largest relative disagreement between the directional derivative from the gradient
    oracle and the central difference of the forward oracle's loss, over every tensor."""
    loss, grads = oracle.backward(cfg, w, ids, tg)
    worst = abs(loss - _loss(cfg, w, ids, tg))
    for name, a in _tensors(cfg, w):
        d = rng.standard_normal(a.shape)
        a0 = a.copy()
        a[...] = a0 + EPS * d
        lp = _loss(cfg, w, ids, tg)
        a[...] = a0 - EPS * d
        lm = _loss(cfg, w, ids, tg)
        a[...] = a0
        fd = (lp - lm) / (2 * EPS)
        an = float((_grad_of(grads, name) * d).sum())
        worst = max(worst, abs(fd - an) / max(1.0, abs(an)))
    return worst


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_gradient_matches_finite_differences_per_tensor(variant):
    cfg = _cfg(**VARIANTS[variant])
    w, ids, tg, rng = _model(cfg, seed=101)
    assert _fd_checks(cfg, w, ids, tg, rng) < 1e-7


def test_gradient_single_entries():
    cfg = _cfg()
    w, ids, tg, rng = _model(cfg, seed=102)
    _, grads = oracle.backward(cfg, w, ids, tg)
    picks = [("wte", (int(ids[0, 3]), 5)), ("wte", (0, 0)), ("wpe", (7, 2)), ("wpe", (11, 2)),
             ("layers.1.attn_w", (40, 3)), ("layers.0.mp_b", (9,)), ("layers.0.ln1_g", (4,)), ("lnf_b", (1,))]
    for name, idx in picks:
        a = dict(_tensors(cfg, w))[name]
        a0 = a[idx]
        a[idx] = a0 + EPS
        lp = _loss(cfg, w, ids, tg)
        a[idx] = a0 - EPS
        lm = _loss(cfg, w, ids, tg)
        a[idx] = a0
        assert abs((lp - lm) / (2 * EPS) - _grad_of(grads, name)[idx]) < 1e-8, name
    assert np.all(grads["wpe"][8:] == 0.0)            # positions past T are not used


def test_gradient_of_longer_sequence_and_wider_heads():
    cfg = _cfg(V=23, C=24, H=3, L=1, ctx=20, ffn=96)
    w, ids, tg, rng = _model(cfg, seed=103, B=3, T=20, wstd=0.25)
    assert _fd_checks(cfg, w, ids, tg, rng) < 1e-7


# ---------------------------------------------------------------- one step at a time

def _fd_step(f, args, i, dy, rng):
    """Directional derivative of <dy, f(*args)> in argument i, by central differences."""
    d = rng.standard_normal(np.shape(args[i]))
    a = list(args)
    a[i] = args[i] + EPS * d
    lp = float((dy * f(*a)).sum())
    a[i] = args[i] - EPS * d
    lm = float((dy * f(*a)).sum())
    return (lp - lm) / (2 * EPS), d


def test_layernorm_backward_steps_and_invariances():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 10)) * 3 + 1
    g = 1 + 0.2 * rng.standard_normal(10)
    b = 0.1 * rng.standard_normal(10)
    dy = rng.standard_normal((6, 10))
    dx, dg, db = oracle.layernorm_backward(x, g, dy, 1e-5)
    for i, grad in ((0, dx), (1, dg), (2, db)):
        fd, d = _fd_step(lambda x_, g_, b_: go.layernorm(x_, g_, b_, 1e-5), (x, g, b), i, dy, rng)
        assert abs(fd - (grad * d).sum()) < 1e-7
    var = x.var(-1)
    xc = x - x.mean(-1, keepdims=True)
    xh = xc / np.sqrt(var[:, None] + 1e-5)
    assert np.allclose(dx.sum(-1), 0.0, atol=1e-12)              # shift invariance
    # scaling the deviations by a moves xh only through eps: d/da at a = 1 is xh * eps / (var + eps)
    want = 1e-5 / (var + 1e-5) * (dy * g * xh).sum(-1)
    assert np.allclose((dx * xc).sum(-1), want, rtol=1e-9, atol=1e-14)


@pytest.mark.parametrize("mode", [0, 1])
def test_gelu_backward_steps(mode):
    rng = np.random.default_rng(6)
    u = np.concatenate([np.linspace(-6, 6, 41), rng.standard_normal(20) * 2])
    dg = rng.standard_normal(u.shape)
    fd = (go.gelu(u + EPS, mode) - go.gelu(u - EPS, mode)) / (2 * EPS)
    assert np.max(np.abs(oracle.gelu_backward(u, dg, mode) - dg * fd)) < 1e-8
    assert abs(oracle.gelu_backward(np.zeros(1), np.ones(1), mode)[0] - 0.5) < 1e-15    # gelu'(0) = 1/2


def test_attention_backward_steps_and_key_sum():
    rng = np.random.default_rng(7)
    H, T, D = 2, 9, 4
    q, k, v = (rng.standard_normal((H, T, D)) for _ in range(3))
    dy = rng.standard_normal((H, T, D))
    grads = oracle.attention_backward(q, k, v, dy)
    f = lambda q_, k_, v_: go.attention_probs(q_, k_) @ v_
    for i in range(3):
        fd, d = _fd_step(f, (q, k, v), i, dy, rng)
        assert abs(fd - (grads[i] * d).sum()) < 1e-7, i
    assert np.allclose(grads[1].sum(axis=-2), 0.0, atol=1e-12)   # keys share any common shift
    assert np.allclose(grads[0][:, 0], 0.0)                       # row 0 attends to itself only


def test_attention_backward_t1():
    # one position: Y = V, so dV = dY and no score has a gradient
    rng = np.random.default_rng(8)
    q, k, v, dy = (rng.standard_normal((3, 1, 5)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, dy)
    assert np.array_equal(dv, dy) and not dq.any() and not dk.any()


def test_cross_entropy_backward_steps():
    rng = np.random.default_rng(9)
    z = rng.standard_normal((5, 7)) * 2
    y = rng.integers(0, 7, 5)
    dz = oracle.cross_entropy_backward(z, y)
    assert np.allclose(dz.sum(-1), 0.0, atol=1e-15)
    d = rng.standard_normal(z.shape)
    fd = (go.cross_entropy(z + EPS * d, y) - go.cross_entropy(z - EPS * d, y)) / (2 * EPS)
    assert abs(fd - (dz * d).sum()) < 1e-9
    # equal logits: (1/V - onehot) / N
    dz0 = oracle.cross_entropy_backward(np.zeros((2, 4)), np.array([1, 3]))
    want = np.full((2, 4), 0.25 / 2)
    want[0, 1] -= 0.5
    want[1, 3] -= 0.5
    assert np.allclose(dz0, want, atol=1e-16)


def test_linear_and_embed_backward_steps():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((2, 3, 5))
    w = rng.standard_normal((4, 5))
    b = rng.standard_normal(4)
    dy = rng.standard_normal((2, 3, 4))
    dx, dw, db = oracle.linear_backward(x, w, dy)
    for i, grad in ((0, dx), (1, dw), (2, db)):
        fd, d = _fd_step(go.linear, (x, w, b), i, dy, rng)
        assert abs(fd - (grad * d).sum()) < 1e-8
    ids = np.array([[3, 1, 3], [0, 3, 2]])
    dx0 = rng.standard_normal((2, 3, 5))
    dE, dP = oracle.embed_backward(dx0, ids, V=6, ctx=4)
    assert np.allclose(dE[3], dx0[0, 0] + dx0[0, 2] + dx0[1, 1]) and not dE[4:].any() and not dE[5].any()
    assert np.allclose(dP[:3], dx0.sum(0)) and not dP[3].any()


def test_tied_table_collects_both_uses():
    cfg = _cfg()
    w, ids, tg, rng = _model(cfg, seed=104)
    _, grads = oracle.backward(cfg, w, ids, tg, parts=True)
    assert np.allclose(grads["wte"], grads["wte_embed"] + grads["wte_head"], rtol=0, atol=1e-15)
    assert np.allclose(grads["wte_head"].sum(axis=0), 0.0, atol=1e-12)   # rows of dz sum to zero
    # the head's share alone: perturb only the table the head reads
    d = rng.standard_normal(w["wte"].shape)
    h = go.forward_hidden(cfg, w, ids)
    lp = go.cross_entropy(go.lm_head(h, w["wte"] + EPS * d), tg)
    lm = go.cross_entropy(go.lm_head(h, w["wte"] - EPS * d), tg)
    assert abs((lp - lm) / (2 * EPS) - (grads["wte_head"] * d).sum()) < 1e-8
    # only the ids that occur get an embedding share
    absent = np.setdiff1d(np.arange(cfg.V), ids)
    assert not grads["wte_embed"][absent].any()


def test_overfit_one_batch_with_plain_gradient_steps():
    # the pages' pre-training sanity check: repeated steps on one batch drive its loss down;
    # and a small step along -g lowers the loss by lr * |g|^2 to first order
    cfg = _cfg()
    w, ids, tg, _ = _model(cfg, seed=105, wstd=0.1)
    loss0, g0 = oracle.backward(cfg, w, ids, tg)
    gnorm2 = sum(float((_grad_of(g0, n) ** 2).sum()) for n, _ in _tensors(cfg, w))
    saved = [a.copy() for _, a in _tensors(cfg, w)]
    lr = 1e-4
    for name, a in _tensors(cfg, w):
        a -= lr * _grad_of(g0, name)
    assert abs((loss0 - _loss(cfg, w, ids, tg)) / (lr * gnorm2) - 1.0) < 1e-3
    for (_, a), a0 in zip(_tensors(cfg, w), saved):
        a[...] = a0
    losses = []
    for _ in range(40):
        loss, g = oracle.backward(cfg, w, ids, tg)
        losses.append(loss)
        for name, a in _tensors(cfg, w):
            a -= 0.1 * _grad_of(g, name)
    assert losses[-1] < 0.2 * losses[0]


# ---------------------------------------------------------------- planted mistakes

def _grad_pins_pass():
    try:
        for variant in ("pre", "post"):
            cfg = _cfg(**VARIANTS[variant], L=1)
            w, ids, tg, rng = _model(cfg, seed=106)
            if _fd_checks(cfg, w, ids, tg, rng) > 1e-7:
                return False
        return True
    except Exception:
        return False


def test_grad_pins_pass_on_oracle():
    assert _grad_pins_pass()


@pytest.mark.parametrize("mistake", ["ln_no_xh_term", "gelu_no_u_term", "attn_k_unscaled", "attn_no_rowsum",
                                     "ce_not_mean", "no_tied_head_share", "no_position_grad", "dw_transposed"])
def test_planted_grad_mistakes_are_caught(mistake, monkeypatch):
    ln_b, gelu_b, attn_b = gg.layernorm_backward, gg.gelu_backward, gg.attention_backward
    ce_b, emb_b, lin_b = gg.cross_entropy_backward, gg.embed_backward, gg.linear_backward
    if mistake == "ln_no_xh_term":
        def bad(x, g, dy, eps=1e-5):
            x = np.asarray(x, np.float64)
            r = 1 / np.sqrt(x.var(-1, keepdims=True) + eps)
            dxh = dy * g
            dx = r * (dxh - dxh.mean(-1, keepdims=True))
            _, dg, db = ln_b(x, g, dy, eps)
            return dx, dg, db
        monkeypatch.setattr(gg, "layernorm_backward", bad)
    elif mistake == "gelu_no_u_term":
        monkeypatch.setattr(gg, "gelu_backward",
                            lambda u, dg, mode=0: dg * 0.5 * (1 + np.tanh(math.sqrt(2 / math.pi) * (u + 0.044715 * u ** 3))))
    elif mistake == "attn_k_unscaled":
        def bad(q, k, v, dy):
            dq, dk, dv = attn_b(q, k, v, dy)
            return dq, dk * math.sqrt(q.shape[-1]), dv
        monkeypatch.setattr(gg, "attention_backward", bad)
    elif mistake == "attn_no_rowsum":
        def bad(q, k, v, dy):
            a = go.attention_probs(q, k)
            ds = a * (dy @ np.swapaxes(v, -1, -2))
            D = q.shape[-1]
            return ds @ k / math.sqrt(D), np.swapaxes(ds, -1, -2) @ q / math.sqrt(D), np.swapaxes(a, -1, -2) @ dy
        monkeypatch.setattr(gg, "attention_backward", bad)
    elif mistake == "ce_not_mean":
        monkeypatch.setattr(gg, "cross_entropy_backward", lambda z, y: ce_b(z, y) * np.asarray(y).size)
    elif mistake == "no_tied_head_share":
        orig = gg.backward

        def bad(cfg, w, ids, tg, parts=False):
            loss, g = orig(cfg, w, ids, tg, parts=True)
            g["wte"] = g["wte_embed"]
            return loss, g
        monkeypatch.setattr(oracle, "backward", bad)
    elif mistake == "no_position_grad":
        monkeypatch.setattr(gg, "embed_backward", lambda dx0, ids, V, ctx: (emb_b(dx0, ids, V, ctx)[0], np.zeros((ctx, dx0.shape[-1]))))
    elif mistake == "dw_transposed":
        def bad(x, w, dy):
            dx, dw, db = lin_b(x, w, dy)
            return dx, (dw.T if dw.shape[0] == dw.shape[1] else dw[::-1]), db
        monkeypatch.setattr(gg, "linear_backward", bad)
    assert not _grad_pins_pass(), f"planted mistake {mistake} went unnoticed"


# ---------------------------------------------------------------- the optimiser step

def test_adamw_step_matches_torch_adamw():
    # the written-out update against torch.optim.AdamW (fp64, CPU), three steps, decay on matrices only
    torch = pytest.importorskip("torch")
    cfg = _cfg(L=1)
    w, ids, tg, rng = _model(cfg, seed=107)
    names = [n for n, _ in _tensors(cfg, w)]
    tp = {n: torch.tensor(a.copy(), dtype=torch.float64, requires_grad=True) for n, a in _tensors(cfg, w)}
    decay = [tp[n] for n in names if n.endswith("_w") or n in ("wte", "wpe")]
    rest = [tp[n] for n in names if not (n.endswith("_w") or n in ("wte", "wpe"))]
    opt = torch.optim.AdamW([{"params": decay, "weight_decay": 0.1}, {"params": rest, "weight_decay": 0.0}],
                            lr=3e-3, betas=(0.9, 0.95), eps=1e-8)
    state = {}
    for _ in range(3):
        _, g = oracle.backward(cfg, w, ids, tg)
        for n in names:
            tp[n].grad = torch.tensor(_grad_of(g, n), dtype=torch.float64)
        opt.step()
        oracle.adamw_step(w, g, state, lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
        for n, a in _tensors(cfg, w):
            assert np.allclose(a, tp[n].detach().numpy(), rtol=1e-12, atol=1e-14), n


def test_adamw_first_step_moves_each_weight_by_lr():
    # at t = 1, m / (1 - b1) = g and sqrt(v / (1 - b2)) = |g|: each weight moves by lr * sign(g) (eps aside)
    cfg = _cfg(L=1)
    w, ids, tg, _ = _model(cfg, seed=108)
    before = {n: a.copy() for n, a in _tensors(cfg, w)}
    _, g = oracle.backward(cfg, w, ids, tg)
    oracle.adamw_step(w, g, {}, lr=1e-3, eps=1e-12)
    for n, a in _tensors(cfg, w):
        gr = _grad_of(g, n)
        big = np.abs(gr) > 1e-6
        assert np.allclose((before[n] - a)[big], 1e-3 * np.sign(gr[big]), rtol=1e-5), n


def test_untied_head_with_the_table_as_head_equals_tied():
    # an untied head whose matrix equals E computes the tied model; its two gradients add to the tied one
    from dataclasses import replace
    cfg = _cfg()
    w, ids, tg, _ = _model(cfg, seed=109)
    cu = replace(cfg, untied_head=1)
    wu = dict(w)
    wu["head"] = w["wte"].copy()
    lt, gt = oracle.backward(cfg, w, ids, tg)
    lu, gu = oracle.backward(cu, wu, ids, tg)
    assert abs(lt - lu) < 1e-14
    assert np.allclose(gu["wte"] + gu["head"], gt["wte"], rtol=0, atol=1e-15)
    assert go.param_count(cu) == go.param_count(cfg) + cfg.V * cfg.C


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_gradient_matches_torch_autograd(variant):
    # the whole gradient against autograd through torch.nn.functional routines (fp64, CPU)
    pytest.importorskip("torch")
    import torch_ref
    cfg = _cfg(V=50, C=32, H=4, L=2, ctx=24, ffn=128, **VARIANTS[variant])
    w, ids, tg, _ = _model(cfg, seed=110, B=2, T=24, wstd=0.2)
    loss, grads = oracle.backward(cfg, w, ids, tg)
    rloss, ref = torch_ref.grads(cfg, w, ids, tg)
    assert abs(loss - rloss) < 1e-12
    for name, a in _tensors(cfg, w):
        r = ref[name] if not name.startswith("layers.") else ref["layers"][int(name.split(".")[1])][name.split(".")[2]]
        g = _grad_of(grads, name)
        assert np.max(np.abs(g - r)) <= 1e-10 * max(1.0, np.max(np.abs(r))), name
