"""The attention derivative step (gptk_attention_bwd) and the forward's log-sum-exp
(gptk_attention_lse) against the fp64 oracle, element by element, through the C ABI.

Inputs are seeded and bf16-exact (qkv, dy); y and lse2 come from the GPU forward,
as in training. The bound on each output element follows the kernel's arithmetic:
  * dS^T and P^T are rounded to bf16 before their products (relative 2^-9 per
    term): dQ, dK get 2^-9 * sum|dS||K or Q| / sqrt(D), dU gets 2^-9 * sum A |dY|
  * Dsum is formed from the bf16 forward output y, whose error e_y is the forward's
    bound (2^-8 max|U| + 1 ulp): dS_ts moves by A_ts * dDsum_t, dDsum_t = sum_d |dY_td| e_y,td
  * the outputs are bf16 (one ulp), fp32 accumulation adds far less
Each bound is doubled for headroom, which still fails a dropped key tile, a wrong
sign or a transposed operand by orders of magnitude.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import bf16_ulp, dev_bf16, host, rand_bf16  # noqa: E402

TWO9 = 2.0 ** -9


def _inputs(B, T, H, D, seed, qk_scale=2.0, dy_scale=1.0):
    rng = np.random.default_rng(seed)
    C = H * D
    qkv = rand_bf16(rng, (B, T, 3 * C))
    qkv[..., :2 * C] *= qk_scale
    dy = rand_bf16(rng, (B, T, C), dy_scale)
    return qkv, dy


def _gpu(qkv, dy, H):
    from decoder_only_transformer_gpt_gb300 import binding
    B, T, C3 = qkv.shape
    C = C3 // 3
    q_d = dev_bf16(qkv)
    y = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
    lse2 = torch.empty((B * H * T,), dtype=torch.float32, device="cuda")
    binding.attention_lse(q_d, y, lse2, H)
    dqkv = torch.empty((B, T, C3), dtype=torch.bfloat16, device="cuda")
    dy_d = dev_bf16(dy)
    binding.attention_bwd(q_d, y, dy_d, lse2, dqkv, H)
    binding.status()
    return q_d, y, dy_d, lse2, dqkv


def _heads(t, H):
    T, C = t.shape
    return t.reshape(T, H, C // H).transpose(1, 0, 2)


def _check_sequence(qkv_b, dy_b, y_b, lse_b, got_b, H, umax):
    """One sequence: lse2 and the three thirds of dqkv against the oracle within the derived bounds."""
    T, C3 = qkv_b.shape
    C = C3 // 3
    D = C // H
    x = qkv_b.astype(np.float64)
    ref = oracle.causal_self_attention_backward(x[None], dy_b.astype(np.float64)[None], H)[0]
    q, k, u = _heads(x[:, :C], H), _heads(x[:, C:2 * C], H), _heads(x[:, 2 * C:], H)
    dyh = _heads(dy_b.astype(np.float64), H)
    yh = _heads(y_b.astype(np.float64), H)
    A = oracle.attention_probs(q, k)                                       # [H, T, T]
    # the log-sum-exp of the scaled scores in base 2 (the definition, from the scores directly)
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(D)
    s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    lse_ref = (m[..., 0] + np.log(np.exp(s - m).sum(axis=-1))) / math.log(2.0)
    assert np.all(np.abs(lse_b.reshape(H, T) - lse_ref) <= 1e-4 * (1.0 + np.abs(lse_ref))), "lse2"
    # bound scales
    dA = dyh @ np.swapaxes(u, -1, -2)
    dS = A * (dA - (dA * A).sum(axis=-1, keepdims=True))
    y_ref = A @ u
    e_y = 2.0 ** -8 * umax + bf16_ulp(y_ref) + 1e-5
    assert np.all(np.abs(yh - y_ref) <= e_y), "forward output"
    dds = (np.abs(dyh) * e_y).sum(axis=-1)                                 # [H, T]
    aq, ak = np.abs(q), np.abs(k)
    tq = (TWO9 * (np.abs(dS) @ ak) + dds[..., None] * (A @ ak)) / math.sqrt(D)
    tk = (TWO9 * (np.swapaxes(np.abs(dS), -1, -2) @ aq) + np.swapaxes(A, -1, -2) @ (dds[..., None] * aq)) / math.sqrt(D)
    tu = TWO9 * (np.swapaxes(A, -1, -2) @ np.abs(dyh))

    def merged(t):                                                          # [H, T, D] -> [T, C]
        return t.transpose(1, 0, 2).reshape(T, C)

    tol = np.concatenate([merged(tq), merged(tk), merged(tu)], axis=1) * 2.0 + bf16_ulp(ref) + 1e-7
    bad = np.abs(got_b - ref) > tol
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} of {bad.size} outside bound; first at {tuple(idx)}: "
                             f"got {got_b[tuple(idx)]}, ref {ref[tuple(idx)]}, tol {tol[tuple(idx)]}")


@pytest.mark.parametrize("B,T,H,D", [(1, 128, 1, 64), (2, 300, 2, 64), (3, 40, 4, 32), (1, 1, 2, 64),
                                     (2, 1024, 3, 64), (1, 257, 2, 32), (4, 129, 3, 64)])
def test_attention_bwd_tc(gpt_lib, B, T, H, D):
    qkv, dy = _inputs(B, T, H, D, seed=T + 7 * H)
    _, y, _, lse2, dqkv = _gpu(qkv, dy, H)
    got, yv, lv = host(dqkv), host(y), host(lse2).reshape(B, H * T)
    umax = np.abs(qkv[..., 2 * H * D:]).max()
    for b in range(B):
        _check_sequence(qkv[b], dy[b], yv[b], lv[b], got[b], H, umax)


def test_attention_bwd_tc_full_size_sampled(gpt_lib):
    """The training shape (B = 16, T = 1024, 12 heads of 64: 1,536 key-tile work items over the
    persistent CTAs, query tiles receiving dQ from up to 8 key tiles in any order): the whole batch
    runs on the GPU; two sequences are checked against the oracle element by element."""
    B, T, H, D = 16, 1024, 12, 64
    qkv, dy = _inputs(B, T, H, D, seed=5, dy_scale=0.25)
    _, y, _, lse2, dqkv = _gpu(qkv, dy, H)
    got, yv, lv = host(dqkv), host(y), host(lse2).reshape(B, H * T)
    umax = np.abs(qkv[..., 2 * H * D:]).max()
    for b in (3, B - 1):
        _check_sequence(qkv[b], dy[b], yv[b], lv[b], got[b], H, umax)


def test_attention_bwd_tc_repeatable(gpt_lib):
    """dQ reaches each query tile as fp32 reduce-adds from its key tiles in whatever order the CTAs
    finish, and the last of them converts it to bf16: five runs at the training shape may differ
    only by that fp32 reordering (below one bf16 ulp plus 2^-20 of the largest value), never by a
    missing or doubled key tile."""
    from decoder_only_transformer_gpt_gb300 import binding
    B, T, H, D = 16, 1024, 12, 64
    qkv, dy = _inputs(B, T, H, D, seed=6, dy_scale=0.25)
    q_d, y, dy_d, lse2, dqkv = _gpu(qkv, dy, H)
    first = host(dqkv)
    scale = np.abs(first).max()
    for _ in range(4):
        out = torch.empty_like(dqkv)
        binding.attention_bwd(q_d, y, dy_d, lse2, out, H)
        binding.status()
        d = np.abs(host(out) - first)
        bound = bf16_ulp(np.maximum(np.abs(first), np.abs(host(out)))) + 2.0 ** -20 * scale
        assert np.all(d <= bound), f"{(d > bound).sum()} elements moved; worst {d.max()}"
