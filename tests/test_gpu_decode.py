"""Incremental decoding (key/value cache) against the fp64 oracle's full forward.

A decode step appends one token per sequence at position pos and must give the
logits that a full forward over the sequence gives at row pos (causality: row
pos depends only on tokens 0..pos). Prefill logits are the last prompt row.
Tolerance as for the bf16 forward: every logit within 5e-2 of the oracle.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import dev_i32, host  # noqa: E402
from workloads import GPTConfig, workload, POST_NORM, GELU_ERF, DT_FP32  # noqa: E402
from workloads.generate import generate, make_weights, make_tokens  # noqa: E402

TZ = 5e-2


def _decode_case(cfg, w, ids, T0, steps):
    """Prefill ids[:, :T0], then decode ids[:, T0 .. T0+steps-1] one at a time."""
    from decoder_only_transformer_gpt_gb300 import binding
    B = ids.shape[0]
    m = binding.GPTModel(cfg, w, B * T0)
    m.kv_reserve(B)
    lg = torch.empty((B, cfg.V), dtype=torch.float32, device="cuda")
    m.prefill(dev_i32(np.ascontiguousarray(ids[:, :T0])), lg)
    m.status()
    got = [host(lg)]
    for k in range(steps):
        pos = T0 + k
        m.decode_step(dev_i32(np.ascontiguousarray(ids[:, pos])), pos, lg)
        m.status()
        got.append(host(lg))
    m.close()
    _, rz = oracle.forward(cfg, w, ids[:, :T0 + steps])
    for k, z in enumerate(got):
        t = T0 - 1 + k                                   # the row these logits predict from
        err = np.max(np.abs(z - rz[:, t]))
        assert err <= TZ, (k, t, err)


@pytest.mark.parametrize("variant", ["pre", "post", "erf", "noln_f", "untied", "post_lnf"])
def test_decode_small_variants(gpt_lib, variant):
    kw = {"pre": {}, "post": dict(norm_mode=POST_NORM, final_ln=0), "erf": dict(gelu=GELU_ERF),
          "noln_f": dict(final_ln=0), "untied": dict(untied_head=1), "post_lnf": dict(norm_mode=POST_NORM)}[variant]
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512, **kw)
    rng = np.random.Generator(np.random.PCG64(31))
    w = make_weights(cfg, rng, affine="random", wstd=0.02)
    ids, _ = make_tokens(cfg.V, 3, 60, rng)
    _decode_case(cfg, w, ids, 40, 20)


def test_decode_head_width_32_and_many_rows(gpt_lib):
    # D = 32 attention, and 20 sequences: the projections run in row groups of 16
    cfg = GPTConfig(V=211, C=128, H=4, L=2, ctx=48, ffn=512)
    rng = np.random.Generator(np.random.PCG64(32))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, _ = make_tokens(cfg.V, 20, 40, rng)
    _decode_case(cfg, w, ids, 1, 39)                     # a one-token prompt, then up to the last position


@pytest.mark.parametrize("B", [2, 6])
def test_decode_gpt2_small(gpt_lib, B):
    # 2 rows: SIMT matrix-vector products; 6 rows: the mma.sync tiles (rows 6..15 of the tile empty)
    wl = workload("gpt2_small")
    w, ids, _ = generate(wl, B=B, T=160)
    _decode_case(wl.cfg, w, ids, 150, 10)


def test_decode_to_the_last_position(gpt_lib):
    # the final step writes cache row ctx - 1
    cfg = GPTConfig(V=97, C=64, H=1, L=1, ctx=32, ffn=256)
    rng = np.random.Generator(np.random.PCG64(33))
    w = make_weights(cfg, rng, affine="random", wstd=0.1)
    ids, _ = make_tokens(cfg.V, 2, 32, rng)
    _decode_case(cfg, w, ids, 30, 2)


def test_decode_errors(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    cfg = GPTConfig(V=97, C=64, H=1, L=1, ctx=32, ffn=256)
    rng = np.random.Generator(np.random.PCG64(34))
    w = make_weights(cfg, rng, affine="random", wstd=0.1)
    ids, _ = make_tokens(cfg.V, 2, 8, rng)
    m = binding.GPTModel(cfg, w, 64)
    lg = torch.empty((2, cfg.V), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.GptError) as e:           # no cache reserved
        m.prefill(dev_i32(ids), lg)
    assert e.value.code == binding.GPT_EINVAL
    m.kv_reserve(2)
    m.prefill(dev_i32(ids), lg)
    m.status()
    with pytest.raises(binding.GptError) as e:           # position past the table
        m.decode_step(dev_i32(ids[:, 0].copy()), 32, lg)
    assert e.value.code == binding.GPT_ESEQ
    with pytest.raises(binding.GptError) as e:           # more sequences than reserved
        m.decode_step(dev_i32(np.zeros(3, np.int32)), 8, lg)
    assert e.value.code == binding.GPT_EINVAL
    bad = np.array([1, cfg.V], np.int32)
    m.decode_step(dev_i32(bad), 8, lg)
    with pytest.raises(binding.GptError) as e:           # a token outside [0, V), found on the device
        m.status()
    assert e.value.code == binding.GPT_ETOKEN
    m.decode_step(dev_i32(ids[:, 0].copy()), 8, lg)      # the handle still works
    m.status()
    m.close()
    f32 = GPTConfig(V=97, C=64, H=1, L=1, ctx=32, ffn=256, dtype=DT_FP32)
    mf = binding.GPTModel(f32, make_weights(f32, rng, affine="random", wstd=0.1), 64)
    with pytest.raises(binding.GptError) as e:           # the cache path is bf16 only
        mf.kv_reserve(2)
    assert e.value.code == binding.GPT_ECONFIG
    mf.close()


# ---- next-token sampling against the oracle's draw

def _sample_case(z, T, k, p, u):
    from decoder_only_transformer_gpt_gb300 import binding
    B = z.shape[0]
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    binding.sample(torch.from_numpy(z.astype(np.float32)).cuda(), torch.from_numpy(u.astype(np.float32)).cuda(),
                   ids, T, k, p)
    torch.cuda.synchronize()
    got = host(ids)
    for b in range(B):
        want, q = oracle.sample_next(z[b].astype(np.float32).astype(np.float64), T, k, p, float(u[b]))
        if got[b] == want:
            continue
        # several draws can be right only where u sits on a boundary of the oracle's CDF, or a
        # filter's cut falls within rounding of its threshold: check the GPU's choice is one of them
        assert q is not None, (b, got[b], want)
        cdf = np.cumsum(q)
        g = int(got[b])
        lo, hi = (cdf[g - 1] if g > 0 else 0.0), cdf[g]
        assert q[g] > 0 and lo - 1e-5 <= u[b] <= hi + 1e-5, (b, g, want, u[b], lo, hi)


@pytest.mark.parametrize("T,k,p", [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.7, 50, 1.0), (1.0, 0, 0.9), (1.3, 40, 0.8),
                                   (1.0, 1, 1.0), (1.0, 0, 1e-7)])
def test_sample_gpt2_vocab(gpt_lib, T, k, p):
    rng = np.random.default_rng(41)
    B, V = 16, 50257
    z = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    u = rng.random(B)
    _sample_case(z, T, k, p, u)


def test_sample_ties_and_small_vocab(gpt_lib):
    rng = np.random.default_rng(42)
    # many equal logits: top-k and top-p cut inside a run of ties (kept in index order)
    z = np.round(rng.standard_normal((8, 3000)), 1).astype(np.float32)
    u = rng.random(8)
    for T, k, p in [(1.0, 17, 1.0), (1.0, 0, 0.5), (0.5, 200, 0.3), (0.0, 0, 1.0)]:
        _sample_case(z, T, k, p, u)
    z1 = np.array([[0.5, 2.0, 2.0, -1.0]], np.float32)            # V = 4, equal maxima
    _sample_case(z1, 0.0, 0, 1.0, np.array([0.3]))
    _sample_case(z1, 1.0, 1, 1.0, np.array([0.9]))


def test_sample_after_decode(gpt_lib):
    # greedy generation through prefill, decode and the sampler matches the oracle's greedy tokens
    from decoder_only_transformer_gpt_gb300 import binding
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512)
    rng = np.random.Generator(np.random.PCG64(43))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, _ = make_tokens(cfg.V, 2, 16, rng)
    m = binding.GPTModel(cfg, w, 2 * 16)
    m.kv_reserve(2)
    lg = torch.empty((2, cfg.V), dtype=torch.float32, device="cuda")
    nxt = torch.empty(2, dtype=torch.int32, device="cuda")
    uni = torch.zeros(2, dtype=torch.float32, device="cuda")
    m.prefill(dev_i32(ids), lg)
    seq = ids.copy()
    for pos in range(16, 24):
        binding.sample(lg, uni, nxt, 0.0)
        tok = host(nxt).astype(np.int32)
        seq = np.concatenate([seq, tok[:, None]], axis=1)
        m.decode_step(dev_i32(tok), pos, lg)
    m.status()
    m.close()
    # the oracle's greedy choice at each generated position, from the GPU's own sequence
    _, rz = oracle.forward(cfg, w, seq[:, :-1])
    for b in range(2):
        for t in range(16, seq.shape[1]):
            zrow = rz[b, t - 1]
            best = np.sort(zrow)[-2:]
            if best[1] - best[0] > 1e-3:                 # a clear maximum: the pick is unique
                assert seq[b, t] == int(np.argmax(zrow)), (b, t)
