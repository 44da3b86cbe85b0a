"""Each CUDA step against the fp64 oracle, element by element, through the C ABI.

Inputs are seeded and bf16-exact, so the only differences come from the
kernel's arithmetic; the bounds below are derived from it:
  * fp32 accumulation of exact bf16 products over K terms: |err| <= K * 2^-23 * sum|a||w|
  * a bf16 output adds one bf16 ulp of the value
  * tanh.approx (GELU) adds at most 0.5|x| * 6e-4
  * attention rounds P to bf16 (relative 2^-9 per weight): |err| <= 2^-8 * max|U| + 1 ulp
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import bf16_ulp, dev_bf16, dev_f32, dev_i32, host, rand_bf16  # noqa: E402

EPS23 = 2.0 ** -23


def _gemm_case(gpt_lib, M, N, K, epi, seed=0):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(seed)
    A = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.5)
    b = rng.standard_normal(N).astype(np.float32)
    ref_lin = oracle.linear(A, W, b)
    acc_bound = K * EPS23 * (np.abs(A).astype(np.float64) @ np.abs(W).astype(np.float64).T) + 1e-6
    if epi in (binding.EPI_BIAS, binding.EPI_BIAS_GELU):
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    else:
        x0 = rng.standard_normal((M, N)).astype(np.float32)
        out = dev_f32(x0) if epi == binding.EPI_BIAS_RESID else torch.empty((M, N), dtype=torch.float32, device="cuda")
    binding.gemm(dev_bf16(A), dev_bf16(W), dev_f32(b), out, epi)
    binding.status()
    got = host(out)
    if epi == binding.EPI_BIAS:
        ref = ref_lin
        tol = bf16_ulp(ref) + acc_bound
    elif epi == binding.EPI_BIAS_GELU:
        ref = oracle.gelu(ref_lin)
        tol = bf16_ulp(ref) + 1.2 * acc_bound + 0.5 * np.abs(ref_lin) * 6e-4
    elif epi == binding.EPI_BIAS_RESID:
        ref = x0.astype(np.float64) + ref_lin
        tol = acc_bound + 4 * EPS23 * np.abs(ref)
    else:
        ref = ref_lin
        tol = acc_bound
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside bound; worst {np.max(np.abs(got - ref) - tol)}"


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 192), (1, 8, 8), (200, 2304, 768)])
@pytest.mark.parametrize("epi", [0, 1, 2, 3])
def test_gemm_tc_epilogues(gpt_lib, M, N, K, epi):
    _gemm_case(gpt_lib, M, N, K, epi)


@pytest.mark.parametrize("M,N,K", [(4096, 2304, 768), (1536, 768, 3072), (2000, 3072, 768)])
def test_gemm_tc_many_tiles_per_cta(gpt_lib, M, N, K):
    # more tiles than SMs: exercises the TMEM double buffer and the stage ring across tiles
    _gemm_case(gpt_lib, M, N, K, 0, seed=M)


@pytest.mark.parametrize("M,N,K", [(6500, 768, 3072), (4000, 2304, 1544), (5000, 2304, 1536), (4000, 1600, 1600)])
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_gemm_tc_stream_k(gpt_lib, M, N, K, epi):
    # more tiles than SMs, not a whole number of waves, K >= 1536: tiles are split
    # along K between CTAs. With 152 SMs: 153 tiles (151 splits), 288 tiles with a
    # ragged last K block, 360 tiles (a 208-tile split region, then a whole wave), and
    # 224 tiles whose last column tile is ragged (N = 1600, the GPT-2 XL width).
    _gemm_case(gpt_lib, M, N, K, epi, seed=K + epi)


@pytest.mark.parametrize("M,N,K,epi", [(16384, 768, 3072, 2), (16384, 2304, 768, 0), (16384, 3072, 768, 1),
                                        (16384, 768, 768, 2), (32768, 768, 3072, 2), (12432, 768, 3072, 2)])
def test_gemm_tc_full_size_sampled_rows(gpt_lib, M, N, K, epi):
    """The projections at the token counts of the timed runs (16,384 = 16 x 1024, 32,768 and the ragged
    12,432 = 16 x 777), whose tile schedules (the stream-K split region of mlp c_proj, several waves of
    whole tiles) the small cases do not reach. Every output is computed on the GPU; 128-row blocks at
    the start, inside and at the end of the split region and in the last wave are checked against the
    oracle with the same bounds as the small cases."""
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(M + N + K)
    A = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.5)
    b = rng.standard_normal(N).astype(np.float32)
    if epi == binding.EPI_BIAS_RESID:
        x0 = rng.standard_normal((M, N)).astype(np.float32)
        out = dev_f32(x0)
    else:
        x0 = None
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    binding.gemm(dev_bf16(A), dev_bf16(W), dev_f32(b), out, epi)
    binding.status()
    got_all = out
    MB = (M + 127) // 128
    blocks = sorted({0, 1, MB // 4, MB // 2, (3 * MB) // 4, MB - 2, MB - 1})
    for mb in blocks:
        r0, r1 = 128 * mb, min(M, 128 * mb + 128)
        ref_lin = oracle.linear(A[r0:r1], W, b)
        acc_bound = K * EPS23 * (np.abs(A[r0:r1]).astype(np.float64) @ np.abs(W).astype(np.float64).T) + 1e-6
        got = host(got_all[r0:r1])
        if epi == binding.EPI_BIAS:
            ref, tol = ref_lin, bf16_ulp(ref_lin) + acc_bound
        elif epi == binding.EPI_BIAS_GELU:
            ref = oracle.gelu(ref_lin)
            tol = bf16_ulp(ref) + 1.2 * acc_bound + 0.5 * np.abs(ref_lin) * 6e-4
        else:
            ref = x0[r0:r1].astype(np.float64) + ref_lin
            tol = acc_bound + 4 * EPS23 * np.abs(ref)
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"rows {r0}:{r1}: {bad.sum()} outside bound; worst {np.max(np.abs(got - ref) - tol)}"


def test_gemm_tc_stream_k_deterministic(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(5)
    M, N, K = 6500, 768, 3072
    A = dev_bf16(rand_bf16(rng, (M, K)))
    W = dev_bf16(rand_bf16(rng, (N, K), 0.5))
    b = dev_f32(rng.standard_normal(N).astype(np.float32))
    outs = []
    for _ in range(3):
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        binding.gemm(A, W, b, out, binding.EPI_BIAS)
        binding.status()
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def _attn_case(B, T, H, D, seed=0, qk_scale=1.5, boost_keys=None):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(seed)
    C = H * D
    qkv = rand_bf16(rng, (B, T, 3 * C))
    qkv[..., :2 * C] = qkv[..., :2 * C] * qk_scale          # peaky softmax (power of two keeps bf16 exact)
    if boost_keys is not None:                               # keys whose scores jump (x 8, still bf16-exact)
        qkv[:, boost_keys, C:2 * C] *= 8.0
    y = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
    binding.attention(dev_bf16(qkv), y, H)
    binding.status()
    ref = oracle.causal_self_attention(qkv.astype(np.float64), H)
    got = host(y)
    umax = np.abs(qkv[..., 2 * C:]).max()
    tol = 2.0 ** -8 * umax + bf16_ulp(ref) + 1e-5
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside bound; worst {np.max(np.abs(got - ref) - tol)}"


@pytest.mark.parametrize("B,T,H,D", [(1, 128, 1, 64), (2, 200, 2, 64), (1, 1, 3, 64), (3, 64, 4, 32),
                                     (2, 777, 2, 64), (1, 1024, 2, 64), (2, 300, 3, 32)])
def test_attention_tc(gpt_lib, B, T, H, D):
    _attn_case(B, T, H, D, qk_scale=2.0)


@pytest.mark.parametrize("B,T", [(16, 1024), (16, 777)])
def test_attention_tc_full_size_sampled(gpt_lib, B, T):
    """Attention at the timed shape (16 x 12 (sequence, head) pairs of 1024 tokens: 1,536 work items
    dealt over the persistent CTAs, every CTA running several items) and its ragged variant; the
    whole batch runs on the GPU and three sequences (all 12 heads) are checked against the oracle."""
    from decoder_only_transformer_gpt_gb300 import binding
    H, D = 12, 64
    C = H * D
    rng = np.random.default_rng(T)
    qkv = rand_bf16(rng, (B, T, 3 * C))
    qkv[..., :2 * C] *= 2.0
    y = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
    binding.attention(dev_bf16(qkv), y, H)
    binding.status()
    umax = np.abs(qkv[..., 2 * C:]).max()
    for b in (0, B // 2 + 1, B - 1):
        ref = oracle.causal_self_attention(qkv[b:b + 1].astype(np.float64), H)[0]
        got = host(y[b])
        tol = 2.0 ** -8 * umax + bf16_ulp(ref) + 1e-5
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"sequence {b}: {bad.sum()} outside bound; worst {np.max(np.abs(got - ref) - tol)}"


@pytest.mark.parametrize("D", [64, 32])
def test_attention_tc_late_max(gpt_lib, D):
    # keys 256..383 score 8x higher: queries 384..511 meet their running maximum's jump in an
    # off-diagonal key tile after two earlier ones (the raise-and-recompute path with a
    # rescale of the output), queries 256..383 on their diagonal tile
    _attn_case(2, 512, 2, D, seed=11, qk_scale=1.0, boost_keys=slice(256, 384))


@pytest.mark.parametrize("C,M", [(768, 37), (128, 300), (16, 5), (2048, 9)])
@pytest.mark.parametrize("odt", ["bf16", "f32"])
def test_layernorm(gpt_lib, C, M, odt):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(C)
    x = (rng.standard_normal((M, C)) * 3 + 0.5).astype(np.float32)
    g = (1 + 0.2 * rng.standard_normal(C)).astype(np.float32)
    b = (0.1 * rng.standard_normal(C)).astype(np.float32)
    out = torch.empty((M, C), dtype=torch.bfloat16 if odt == "bf16" else torch.float32, device="cuda")
    xf = dev_f32(x)
    binding.layernorm(xf, dev_f32(g), dev_f32(b), out, out_f32=xf)
    binding.status()
    ref = oracle.layernorm(x, g, b)
    tol = (bf16_ulp(ref) if odt == "bf16" else 0) + 2e-6 * (np.abs(ref) + 1)
    assert np.all(np.abs(host(out) - ref) <= tol)
    assert np.all(np.abs(host(xf) - ref) <= 2e-6 * (np.abs(ref) + 1))      # the in-place fp32 copy


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_embed(gpt_lib, dt):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(3)
    V, C, B, T = 1000, 768, 3, 50
    E = rand_bf16(rng, (V, C), 0.02)
    P = rand_bf16(rng, (64, C), 0.02)
    ids = rng.integers(0, V, size=(B, T)).astype(np.int32)
    x = torch.empty((B * T, C), dtype=torch.float32, device="cuda")
    mk = dev_bf16 if dt == "bf16" else dev_f32
    binding.embed(dev_i32(ids), mk(E), mk(P), x)
    binding.status()
    ref = oracle.embed(E, P, ids).reshape(B * T, C)
    assert np.all(np.abs(host(x) - ref) <= 1e-7 * np.abs(ref))


def test_embed_rejects_bad_token(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    E = torch.zeros((10, 16), dtype=torch.bfloat16, device="cuda")
    P = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((4, 16), dtype=torch.float32, device="cuda")
    binding.embed(dev_i32(np.array([[1, 2, 10, 3]])), E, P, x)
    with pytest.raises(binding.GptError) as e:
        binding.status()
    assert e.value.code == binding.GPT_ETOKEN
    binding.status()                                                    # the word was cleared


@pytest.mark.parametrize("M,V,C", [(300, 1000, 128), (128, 256, 64), (77, 50257, 768), (1, 17, 16)])
def test_lmhead_ce(gpt_lib, M, V, C):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(V)
    h = rand_bf16(rng, (M, C))
    E = rand_bf16(rng, (V, C), 0.1)
    tg = rng.integers(0, V, size=M).astype(np.int32)
    nll = torch.empty(M, dtype=torch.float32, device="cuda")
    logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
    if C % 8:
        pytest.skip("bf16 path needs C % 8 == 0")
    binding.lmhead_ce(dev_bf16(h), dev_bf16(E), dev_i32(tg), nll, logits)
    binding.status()
    zref = oracle.lm_head(h, E)
    acc_bound = C * EPS23 * (np.abs(h).astype(np.float64) @ np.abs(E).astype(np.float64).T) + 1e-6
    assert np.all(np.abs(host(logits) - zref) <= acc_bound)
    nref = oracle.cross_entropy_rows(zref, tg)
    assert np.max(np.abs(host(nll) - nref)) < 1e-4
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    binding.mean(nll, loss)
    assert abs(float(loss.item()) - float(host(nll).mean())) < 1e-5


def test_lmhead_ce_without_logits_matches(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(9)
    M, V, C = 500, 5000, 128
    h = dev_bf16(rand_bf16(rng, (M, C)))
    E = dev_bf16(rand_bf16(rng, (V, C), 0.1))
    tg = dev_i32(rng.integers(0, V, size=M))
    n1 = torch.empty(M, dtype=torch.float32, device="cuda")
    n2 = torch.empty(M, dtype=torch.float32, device="cuda")
    binding.lmhead_ce(h, E, tg, n1, torch.empty((M, V), dtype=torch.float32, device="cuda"))
    binding.lmhead_ce(h, E, tg, n2, None)
    binding.status()
    assert torch.equal(n1, n2)
