"""Plain fp64 oracle of the gradient of the mean next-token cross-entropy.

TEST INFRASTRUCTURE ONLY, like the rest of this package.

The training step of "预训练一个 Mini GPT" (训练循环: forward, loss, then
back-propagation gives the gradient of every parameter) needs the derivative
of the loss that ``gpt_oracle.forward`` defines. Here it is the chain rule
written out step by step, in the reverse order of the forward, each function
the derivative of one forward step (numpy float64, ``@`` the only library
primitive). The tied table E collects both of its uses: the embedding lookup
and the head ("第 25 章 从小 GPT 到 GPT-2" §25.4: a shared parameter's
gradient is the sum of the contributions of every path that uses it).

Pins (tests/test_oracle_grad_pins.py): central finite differences of the
forward oracle's loss along random directions, tensor by tensor and for the
whole model; per-step finite differences; the shift and scale invariances of
softmax and LayerNorm; the zero column sums of the head's table gradient.
"""
import math

import numpy as np

from workloads.configs import GPTConfig, PRE_NORM, GELU_TANH
from .gpt_oracle import (embed, layernorm, gelu, linear, attention_probs, causal_self_attention,
                         lm_head, head_matrix, cross_entropy)


# ---------------------------------------------------------------- one step each

def linear_backward(x: np.ndarray, w: np.ndarray, dy: np.ndarray):
    """y = x w^T + b  =>  dx = dy w, dw = dy^T x, db = sum of dy over rows."""
    x2 = np.asarray(x, np.float64).reshape(-1, x.shape[-1])
    d2 = np.asarray(dy, np.float64).reshape(-1, dy.shape[-1])
    dx = (d2 @ np.asarray(w, np.float64)).reshape(*dy.shape[:-1], x.shape[-1])
    return dx, d2.T @ x2, d2.sum(axis=0)


def layernorm_backward(x: np.ndarray, g: np.ndarray, dy: np.ndarray, eps: float = 1e-5):
    """Derivative of y = g * (x - mean) * r + b, r = 1 / sqrt(var + eps), per row.

    With xh = (x - mean) r and dxh = dy g:
    dx = r (dxh - mean(dxh) - xh mean(dxh xh)); dg = sum dy xh; db = sum dy.
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(var + eps)
    xh = (x - mean) * r
    dxh = dy * np.asarray(g, np.float64)
    dx = r * (dxh - dxh.mean(axis=-1, keepdims=True) - xh * (dxh * xh).mean(axis=-1, keepdims=True))
    C = x.shape[-1]
    return dx, (dy * xh).reshape(-1, C).sum(axis=0), dy.reshape(-1, C).sum(axis=0)


def gelu_backward(u: np.ndarray, dg: np.ndarray, mode: int = GELU_TANH) -> np.ndarray:
    """dg * gelu'(u).

    tanh form 0.5 u (1 + tanh s), s = c (u + 0.044715 u^3), c = sqrt(2/pi):
    gelu' = 0.5 (1 + tanh s) + 0.5 u (1 - tanh^2 s) c (1 + 3 * 0.044715 u^2).
    erf form u Phi(u): gelu' = Phi(u) + u phi(u), phi the standard normal density.
    """
    u = np.asarray(u, np.float64)
    if mode == GELU_TANH:
        c = math.sqrt(2.0 / math.pi)
        t = np.tanh(c * (u + 0.044715 * u ** 3))
        d = 0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * c * (1.0 + 3.0 * 0.044715 * u * u)
    else:
        erf = np.vectorize(math.erf, otypes=[np.float64])
        d = 0.5 * (1.0 + erf(u / math.sqrt(2.0))) + u * np.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)
    return np.asarray(dg, np.float64) * d


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dy: np.ndarray):
    """Derivative of Y = softmax(Q K^T / sqrt(D) + M) V for one sequence's heads.

    q, k, v, dy: [..., T, D]. With A the probabilities: dV = A^T dY; dA = dY V^T;
    the softmax gives dS = A * (dA - rowsum(dA * A)) (masked entries have A = 0
    and so dS = 0); S = Q K^T / sqrt(D) gives dQ = dS K / sqrt(D), dK = dS^T Q / sqrt(D).
    """
    D = q.shape[-1]
    a = attention_probs(q, k)
    dv = np.swapaxes(a, -1, -2) @ dy
    da = dy @ np.swapaxes(v, -1, -2)
    ds = a * (da - (da * a).sum(axis=-1, keepdims=True))
    dq = ds @ k / math.sqrt(D)
    dk = np.swapaxes(ds, -1, -2) @ q / math.sqrt(D)
    return dq, dk, dv


def causal_self_attention_backward(qkv: np.ndarray, dy: np.ndarray, H: int) -> np.ndarray:
    """Gradient of the fused projection's output [B,T,3C] from that of the merged heads [B,T,C]."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    D = C // H

    def heads(t):
        return t.reshape(B, T, H, D).transpose(0, 2, 1, 3)

    q, k, v = heads(qkv[..., 0:C]), heads(qkv[..., C:2 * C]), heads(qkv[..., 2 * C:])
    dyh = heads(np.asarray(dy, np.float64))
    dqkv = np.empty((B, T, C3), np.float64)
    for b in range(B):
        dq, dk, dv = attention_backward(q[b], k[b], v[b], dyh[b])
        for j, d in enumerate((dq, dk, dv)):
            dqkv[b, :, j * C:(j + 1) * C] = d.transpose(1, 0, 2).reshape(T, C)
    return dqkv


def cross_entropy_backward(logits: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """d(mean over N rows of LSE(z) - z[y]) / dz = (softmax(z) - onehot(y)) / N."""
    z = np.asarray(logits, np.float64).reshape(-1, logits.shape[-1])
    y = np.asarray(targets).reshape(-1)
    p = np.exp(z - z.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    p[np.arange(z.shape[0]), y] -= 1.0
    return (p / z.shape[0]).reshape(logits.shape)


def embed_backward(dx0: np.ndarray, ids: np.ndarray, V: int, ctx: int):
    """x0[b,t] = E[ids[b,t]] + P[t]: rows of E collect the gradient of every position holding that id."""
    C = dx0.shape[-1]
    dE = np.zeros((V, C), np.float64)
    np.add.at(dE, np.asarray(ids).reshape(-1), dx0.reshape(-1, C))
    dP = np.zeros((ctx, C), np.float64)
    dP[:dx0.shape[-2]] = dx0.sum(axis=0)
    return dE, dP


# ---------------------------------------------------------------- whole model

def backward(cfg: GPTConfig, w: dict, ids: np.ndarray, targets: np.ndarray, parts: bool = False):
    """(loss, grads) of the mean next-token cross-entropy.

    grads has the keys of the weight dict: "wte", "wpe", "lnf_g", "lnf_b" (when
    the model has a final LayerNorm), "head" (an untied head) and "layers", one
    dict per block with the parameters' names. With parts=True it also holds "wte_embed" and "wte_head",
    the two contributions whose sum is "wte".
    """
    ids = np.asarray(ids)
    eps = cfg.ln_eps
    pre = cfg.norm_mode == PRE_NORM

    # forward, keeping what the derivatives need
    x = embed(w["wte"], w["wpe"], ids)
    saved = []
    for p in w["layers"]:
        s = {"x": x}
        a1 = layernorm(x, p["ln1_g"], p["ln1_b"], eps) if pre else x
        s["a1"] = a1
        s["qkv"] = linear(a1, p["attn_w"], p["attn_b"])
        s["y"] = causal_self_attention(s["qkv"], cfg.H)
        s1 = x + linear(s["y"], p["proj_w"], p["proj_b"])
        s["s1"] = s1
        n = s1 if pre else layernorm(s1, p["ln1_g"], p["ln1_b"], eps)
        s["n"] = n
        a2 = layernorm(n, p["ln2_g"], p["ln2_b"], eps) if pre else n
        s["a2"] = a2
        s["u"] = linear(a2, p["fc_w"], p["fc_b"])
        s["g"] = gelu(s["u"], cfg.gelu)
        s2 = n + linear(s["g"], p["mp_w"], p["mp_b"])
        s["s2"] = s2
        x = s2 if pre else layernorm(s2, p["ln2_g"], p["ln2_b"], eps)
        saved.append(s)
    h = layernorm(x, w["lnf_g"], w["lnf_b"], eps) if cfg.final_ln else x
    Wh = head_matrix(cfg, w)
    z = lm_head(h, Wh)
    loss = cross_entropy(z, targets)

    # backward
    grads = {"layers": [None] * cfg.L}
    dz = cross_entropy_backward(z, targets)
    C = cfg.C
    dz2 = dz.reshape(-1, cfg.V)
    dh = dz @ np.asarray(Wh, np.float64)
    dE_head = dz2.T @ h.reshape(-1, C)
    if cfg.final_ln:
        dx, grads["lnf_g"], grads["lnf_b"] = layernorm_backward(x, w["lnf_g"], dh, eps)
    else:
        dx = dh
    for li in range(cfg.L - 1, -1, -1):
        p, s = w["layers"][li], saved[li]
        gl = {}
        if pre:
            ds2 = dx
        else:
            ds2, gl["ln2_g"], gl["ln2_b"] = layernorm_backward(s["s2"], p["ln2_g"], dx, eps)
        # s2 = n + mlp(a2)
        dgv, gl["mp_w"], gl["mp_b"] = linear_backward(s["g"], p["mp_w"], ds2)
        du = gelu_backward(s["u"], dgv, cfg.gelu)
        da2, gl["fc_w"], gl["fc_b"] = linear_backward(s["a2"], p["fc_w"], du)
        if pre:
            dn_ln, gl["ln2_g"], gl["ln2_b"] = layernorm_backward(s["n"], p["ln2_g"], da2, eps)
            dn = ds2 + dn_ln
            ds1 = dn
        else:
            dn = ds2 + da2
            ds1, gl["ln1_g"], gl["ln1_b"] = layernorm_backward(s["s1"], p["ln1_g"], dn, eps)
        # s1 = x + proj(attn(a1))
        dy, gl["proj_w"], gl["proj_b"] = linear_backward(s["y"], p["proj_w"], ds1)
        dqkv = causal_self_attention_backward(s["qkv"], dy, cfg.H)
        da1, gl["attn_w"], gl["attn_b"] = linear_backward(s["a1"], p["attn_w"], dqkv)
        if pre:
            dx_ln, gl["ln1_g"], gl["ln1_b"] = layernorm_backward(s["x"], p["ln1_g"], da1, eps)
            dx = ds1 + dx_ln
        else:
            dx = ds1 + da1
        grads["layers"][li] = gl
    dE_embed, grads["wpe"] = embed_backward(dx, ids, cfg.V, w["wpe"].shape[0])
    if getattr(cfg, "untied_head", 0):
        grads["wte"] = dE_embed
        grads["head"] = dE_head
    else:
        grads["wte"] = dE_embed + dE_head
    if parts:
        grads["wte_embed"] = dE_embed
        grads["wte_head"] = dE_head
    return loss, grads


# ---------------------------------------------------------------- the optimiser step

def adamw_step(w: dict, grads: dict, state: dict, lr: float, beta1: float = 0.9, beta2: float = 0.999,
               eps: float = 1e-8, weight_decay: float = 0.0) -> dict:
    """One AdamW update of every parameter, in place on fp64 copies of the weights.

    "Day 16 从零组装 MiniGPT" (the training loop: loss, backward, AdamW, parameters change, repeated) and
    "预训练一个 Mini GPT" 训练循环 (the optimiser step after back-propagation; GPT-2 uses Adam). The update is
    Adam with decoupled weight decay: p <- p - lr wd p; m <- b1 m + (1 - b1) g; v <- b2 v + (1 - b2) g^2;
    p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), t the step count from 1. Reading: the decay
    applies to the weight matrices and the two tables, not to biases and LayerNorm parameters.
    state: {} on the first call; it keeps the step count and both moments per tensor.
    Returns w (its arrays replaced by fp64 arrays holding the new values).
    """
    t = state.get("t", 0) + 1
    state["t"] = t
    bc1, bc2 = 1.0 - beta1 ** t, 1.0 - beta2 ** t

    def upd(key, p, g, decay):
        p = np.asarray(p, np.float64).copy()
        g = np.asarray(g, np.float64)
        m, v = state.get(key, (np.zeros_like(p), np.zeros_like(p)))
        if decay:
            p -= lr * weight_decay * p
        m = beta1 * m + (1.0 - beta1) * g
        v = beta2 * v + (1.0 - beta2) * g * g
        p -= lr * (m / bc1) / (np.sqrt(v / bc2) + eps)
        state[key] = (m, v)
        return p

    for k in ("wte", "wpe", "head"):
        if k in grads:
            w[k] = upd(k, w[k], grads[k], True)
    for k in ("lnf_g", "lnf_b"):
        if k in grads:
            w[k] = upd(k, w[k], grads[k], False)
    for i, (p, gl) in enumerate(zip(w["layers"], grads["layers"])):
        for k in list(p):
            p[k] = upd(f"{i}.{k}", p[k], gl[k], k.endswith("_w"))
    return w
