"""Plain fp64 oracle of the GPT-2-style forward pass and mean next-token CE.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.

Every function follows a passage of the source pages, cited by page title and
section. The computation is the definition written out in numpy float64 with
``@`` (matrix product) as the only library primitive: no blocking, no fusion,
no online softmax. Inputs (weights stored as fp32, bf16-representable on bf16
workloads) are upcast exactly to fp64.

Readings where the pages are silent or disagree:
  * LayerNorm uses the biased variance with eps inside the square root.
  * GELU is the tanh approximation unless the erf form is asked for.
  * Q, K and U are the first, second and third C-wide thirds of c_attn's
    output; head h owns columns [h*D, (h+1)*D) of each third.
  * The causal mask excludes s > t exactly (the pages' -inf / -1e9 additive
    masks give the same probabilities in fp64).
  * The head is tied: logits = h . E^T with no bias.
  * The loss is the mean over all B*T positions, with no ignore index.
  * Post-norm (GPT-1) has no final LayerNorm.

Parity pins for every function live in tests/test_oracle_pins.py.
"""
import math

import numpy as np

from workloads.configs import GPTConfig, PRE_NORM, GELU_TANH


def param_count(cfg: GPTConfig, tied=None) -> int:
    """Unique trainable parameters, counted tensor by tensor.

    "第 25 章 从小 GPT 到 GPT-2" §25.4: per block the four attention
    projections, the two MLP linears and two LayerNorms; plus the token table,
    the position table and the final LayerNorm; a tied head adds nothing.
    """
    C, F = cfg.C, cfg.ffn
    per_block = 0
    per_block += 2 * C                      # ln_1 gain and shift
    per_block += 3 * C * C + 3 * C          # c_attn weight and bias
    per_block += C * C + C                  # attention c_proj
    per_block += 2 * C                      # ln_2
    per_block += F * C + F                  # c_fc
    per_block += C * F + C                  # mlp c_proj
    total = cfg.L * per_block
    total += cfg.V * C                      # token table E
    total += cfg.ctx * C                    # position table P
    if cfg.final_ln:
        total += 2 * C                      # ln_f
    if tied is None:
        tied = not cfg.untied_head
    if not tied:
        total += cfg.V * C
    return total


def linear(x: np.ndarray, w: np.ndarray, b=None) -> np.ndarray:
    """nn.Linear orientation: w is [out, in], y = x w^T + b.

    "第 25 章" §25.5: a Conv1D source stores W as [in, out] and computes XW;
    the Linear form stores its transpose and computes X W_linear^T.
    """
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


def layernorm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Per-position normalisation over the last (C) axis.

    "预训练一个 Mini GPT" 第4步 (mean, np.var, gamma*(x-mean)/sqrt(var+eps)+beta)
    and "GPT-1 学习笔记" §3.2 (the mean of squared deviations, eps inside the root).
    """
    x = np.asarray(x, np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return np.asarray(g, np.float64) * (x - mean) / np.sqrt(var + eps) + np.asarray(b, np.float64)


def gelu(x: np.ndarray, mode: int = GELU_TANH) -> np.ndarray:
    """GELU, elementwise.

    tanh form: "GPT-1 学习笔记" §3.6 and "第 25 章" §25.3 (tanh approximation);
    erf form x * Phi(x) with Phi(x) = (1 + erf(x/sqrt 2))/2: "GPT-1 学习笔记" §3.6.
    """
    x = np.asarray(x, np.float64)
    if mode == GELU_TANH:
        inner = math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)
        return 0.5 * x * (1.0 + np.tanh(inner))
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return x * 0.5 * (1.0 + erf(x / math.sqrt(2.0)))


def embed(wte: np.ndarray, wpe: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """x0[b,t] = E[ids[b,t]] + P[t] ("第 25 章" §25.1; "预训练一个 Mini GPT" 第1步)."""
    ids = np.asarray(ids)
    V = wte.shape[0]
    if ids.size and (ids.min() < 0 or ids.max() >= V):
        raise ValueError("token id out of range [0, V)")
    T = ids.shape[-1]
    if T > wpe.shape[0]:
        raise ValueError("sequence longer than the position table")
    return np.asarray(wte, np.float64)[ids] + np.asarray(wpe, np.float64)[:T]


def attention_probs(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """A = softmax(Q K^T / sqrt(D) + M) per head, M = -inf where s > t.

    q, k: [..., T, D]. "第 25 章" §25.2 (scores, mask for s > t, softmax over
    the last axis); "预训练一个 Mini GPT" 第2步 (max-subtracted softmax).
    The masked entries are left out of the max and the sum and set to 0.
    """
    D = q.shape[-1]
    T = q.shape[-2]
    scores = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(D)
    allowed = np.tril(np.ones((T, T), dtype=bool))          # s <= t
    scores = np.where(allowed, scores, -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    e = np.where(allowed, np.exp(scores - m), 0.0)
    return e / e.sum(axis=-1, keepdims=True)


def causal_self_attention(qkv: np.ndarray, H: int) -> np.ndarray:
    """Heads of the fused projection -> merged attention output y [B,T,C].

    "第 25 章" §25.2: c_attn gives B x T x 3C, split along the last axis into
    Q, K, U; each becomes B x H x T x D; Y = A U; heads are merged back to
    B x T x C before c_proj.
    """
    B, T, C3 = qkv.shape
    C = C3 // 3
    D = C // H
    q = qkv[..., 0:C].reshape(B, T, H, D).transpose(0, 2, 1, 3)
    k = qkv[..., C:2 * C].reshape(B, T, H, D).transpose(0, 2, 1, 3)
    u = qkv[..., 2 * C:3 * C].reshape(B, T, H, D).transpose(0, 2, 1, 3)
    y = np.empty((B, H, T, D), np.float64)
    for b in range(B):                       # one sequence at a time bounds memory
        y[b] = attention_probs(q[b], k[b]) @ u[b]
    return y.transpose(0, 2, 1, 3).reshape(B, T, C)


def _attn_branch(a: np.ndarray, p: dict, cfg: GPTConfig) -> np.ndarray:
    qkv = linear(a, p["attn_w"], p["attn_b"])
    y = causal_self_attention(qkv, cfg.H)
    return linear(y, p["proj_w"], p["proj_b"])


def _mlp_branch(a: np.ndarray, p: dict, cfg: GPTConfig) -> np.ndarray:
    """C -> ffn -> C with GELU in between ("第 25 章" §25.3)."""
    return linear(gelu(linear(a, p["fc_w"], p["fc_b"]), cfg.gelu), p["mp_w"], p["mp_b"])


def block_pre_norm(x: np.ndarray, p: dict, cfg: GPTConfig) -> np.ndarray:
    """x += attn(LN1 x); x += mlp(LN2 x) ("第 25 章" §25.1; "预训练一个 Mini GPT" 第4步)."""
    x = x + _attn_branch(layernorm(x, p["ln1_g"], p["ln1_b"], cfg.ln_eps), p, cfg)
    x = x + _mlp_branch(layernorm(x, p["ln2_g"], p["ln2_b"], cfg.ln_eps), p, cfg)
    return x


def block_post_norm(x: np.ndarray, p: dict, cfg: GPTConfig) -> np.ndarray:
    """n = LN1(x + attn x); h = LN2(n + mlp n) ("GPT-1 学习笔记" §3.1, §3.2)."""
    n = layernorm(x + _attn_branch(x, p, cfg), p["ln1_g"], p["ln1_b"], cfg.ln_eps)
    return layernorm(n + _mlp_branch(n, p, cfg), p["ln2_g"], p["ln2_b"], cfg.ln_eps)


def forward_hidden(cfg: GPTConfig, w: dict, ids: np.ndarray) -> np.ndarray:
    """Embedding, L blocks and (pre-norm only) ln_f: the head's input h [B,T,C]."""
    x = embed(w["wte"], w["wpe"], ids)
    blk = block_pre_norm if cfg.norm_mode == PRE_NORM else block_post_norm
    for p in w["layers"]:
        x = blk(x, p, cfg)
    if cfg.final_ln:
        x = layernorm(x, w["lnf_g"], w["lnf_b"], cfg.ln_eps)
    return x


def head_matrix(cfg: GPTConfig, w: dict) -> np.ndarray:
    """The head's [V, C] matrix: E itself (tied, "第 25 章" §25.4) or the untied head of
    "Day 16 从零组装 MiniGPT" (its own nn.Linear(C, V) without bias)."""
    return w["head"] if getattr(cfg, "untied_head", 0) else w["wte"]


def lm_head(h: np.ndarray, wte: np.ndarray) -> np.ndarray:
    """Tied head: logit j = <h, E_j>, no bias ("第 25 章" §25.4; "GPT-1 学习笔记" §4.1)."""
    return np.asarray(h, np.float64) @ np.asarray(wte, np.float64).T


def cross_entropy_rows(logits: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """Per-position -log softmax(z)[y], max-subtracted ("预训练一个 Mini GPT" 第6步)."""
    z = np.asarray(logits, np.float64).reshape(-1, logits.shape[-1])
    y = np.asarray(targets).reshape(-1)
    V = z.shape[-1]
    if y.size and (y.min() < 0 or y.max() >= V):
        raise ValueError("target out of range [0, V)")
    m = z.max(axis=-1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z - m).sum(axis=-1))
    return lse - z[np.arange(z.shape[0]), y]


def cross_entropy(logits: np.ndarray, targets: np.ndarray) -> float:
    """Mean over all B*T positions ("第 25 章" §25.7; "GPT-1 学习笔记" §4.1)."""
    return float(cross_entropy_rows(logits, targets).mean())


def forward(cfg: GPTConfig, w: dict, ids: np.ndarray, targets=None):
    """(loss or None, logits [B,T,V] fp64) for one batch."""
    ids = np.asarray(ids)
    if cfg.C % cfg.H != 0:
        raise ValueError("C must be divisible by H")
    logits = lm_head(forward_hidden(cfg, w, ids), head_matrix(cfg, w))
    loss = None if targets is None else cross_entropy(logits, targets)
    return loss, logits


def sample_next(logits: np.ndarray, temperature: float, top_k: int, top_p: float, u: float):
    """Next token of one row of logits: (index, kept probabilities in index order).

    "预训练一个 Mini GPT", 第7步 文本生成: probabilities are softmax(logits / T)
    and the token is drawn from them (the draw takes the first index whose
    cumulative probability, in index order, exceeds the uniform number u);
    temperature 0 is greedy decoding (the most probable token; here the lowest
    index among equal maxima). "02 GPT 架构", 8.1-8.3: top-k keeps the k most
    probable tokens; top-p sorts by probability from high to low and keeps the
    smallest leading set whose probabilities add up to p. Readings: top-k is
    applied first, top-p to the renormalised top-k distribution; equal
    probabilities are ordered by index (lower first); the kept set is
    renormalised before the draw; top_k <= 0 or >= V and top_p <= 0 or >= 1
    mean no filter.
    """
    z = np.asarray(logits, dtype=np.float64)
    V = z.shape[0]
    if temperature <= 0:
        return int(np.argmax(z)), None            # argmax returns the first maximum
    z = z / temperature
    p = np.exp(z - z.max())
    p = p / p.sum()
    # rank tokens by probability, high to low, lower index first among equals
    order = sorted(range(V), key=lambda i: (-p[i], i))
    keep = np.zeros(V, dtype=bool)
    kcount = V if (top_k <= 0 or top_k >= V) else top_k
    for i in order[:kcount]:
        keep[i] = True
    if 0 < top_p < 1:
        mass = sum(p[i] for i in order[:kcount])
        acc = 0.0
        nucleus = np.zeros(V, dtype=bool)
        for i in order[:kcount]:
            nucleus[i] = True
            acc += p[i]
            if acc >= top_p * mass:
                break
        keep = nucleus
    q = np.where(keep, p, 0.0)
    q = q / q.sum()
    cdf = 0.0
    for i in range(V):
        cdf += q[i]
        if cdf > u:
            return i, q
    last = int(np.nonzero(keep)[0][-1])           # u at the very top: the last kept token
    return last, q
