"""Back-propagation on the GPU (gpt_backward) against the fp64 gradient oracle.

Both sides start from the same bf16-representable weights and the same tokens.
The GPU keeps activations and the gradients between steps in bf16 (dz, dg, du,
dy, dqkv and the transposed operands of the weight products) and accumulates in
fp32, so each gradient tensor carries a few bf16 roundings (2^-9 relative each)
per step it passed through; the bar is the norm-wise relative error of every
tensor, ||g - g_ref|| / ||g_ref|| <= 2e-2, and |loss - loss_ref| <= 1e-2 as for
the forward. A tensor whose reference is exactly zero (ln_f of a model without
it) must be exactly zero.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import dev_i32, host  # noqa: E402
from workloads import GPTConfig, workload, POST_NORM, GELU_ERF, DT_FP32  # noqa: E402
from workloads.generate import generate, make_weights, make_tokens  # noqa: E402

REL = 2e-2
TLOSS = 1e-2


def _gpu_grads(cfg, w, ids, tg):
    from decoder_only_transformer_gpt_gb300 import binding
    B, T = ids.shape
    m = binding.GPTModel(cfg, w, B * T)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.backward(dev_i32(ids), dev_i32(tg), loss)
    g = m.grads()
    torch.cuda.synchronize()
    out = {k: host(v) for k, v in g.items() if k != "layers"}
    out["layers"] = [{k: host(v) for k, v in p.items()} for p in g["layers"]]
    lv = float(loss.item())
    m.close()
    return lv, out


def _pairs(cfg, got, ref):
    yield "wte", got["wte"], ref["wte"]
    yield "wpe", got["wpe"], ref["wpe"]
    if "head" in ref:
        yield "head", got["head"], ref["head"]
    for k in ("lnf_g", "lnf_b"):
        yield k, got[k], ref.get(k, np.zeros(cfg.C))
    for i, (pg, pr) in enumerate(zip(got["layers"], ref["layers"])):
        for k in pr:
            yield f"layers.{i}.{k}", pg[k], pr[k]


def _compare(cfg, w, ids, tg, rel=REL):
    lv, got = _gpu_grads(cfg, w, ids, tg)
    lref, ref = oracle.backward(cfg, w, ids, tg)
    assert abs(lv - lref) <= TLOSS, (lv, lref)
    worst = (0.0, "")
    for name, g, r in _pairs(cfg, got, ref):
        assert g.shape == r.shape, name
        assert np.isfinite(g).all(), name
        nr = np.linalg.norm(r)
        if nr == 0.0:
            assert not g.any(), name
            continue
        e = np.linalg.norm(g - r) / nr
        worst = max(worst, (e, name))
        assert e <= rel, (name, e)
    print(f"\nloss {lv:.6f} vs {lref:.6f}; worst relative gradient error {worst[0]:.2e} ({worst[1]})")
    return worst


@pytest.mark.parametrize("variant", ["pre", "post", "post_lnf", "erf", "noln_f", "untied"])
def test_backward_small_variants(gpt_lib, variant):
    kw = {"pre": {}, "post": dict(norm_mode=POST_NORM, final_ln=0), "post_lnf": dict(norm_mode=POST_NORM),
          "erf": dict(gelu=GELU_ERF), "noln_f": dict(final_ln=0), "untied": dict(untied_head=1)}[variant]
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512, **kw)
    rng = np.random.Generator(np.random.PCG64(51))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, tg = make_tokens(cfg.V, 2, 64, rng)
    _compare(cfg, w, ids, tg)


def test_backward_odd_token_count(gpt_lib):
    # B * T = 39 tokens: partial row tiles, a partial last K slice of every weight-gradient product
    cfg = GPTConfig(V=157, C=64, H=2, L=2, ctx=16, ffn=256)
    rng = np.random.Generator(np.random.PCG64(57))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, tg = make_tokens(cfg.V, 3, 13, rng)
    _compare(cfg, w, ids, tg)


def test_backward_ragged_head_width_32(gpt_lib):
    # D = 32 heads, T = 40 (ragged against the 16-row fragments and 64-row blocks), 3 sequences
    cfg = GPTConfig(V=211, C=128, H=4, L=2, ctx=48, ffn=512)
    rng = np.random.Generator(np.random.PCG64(52))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, tg = make_tokens(cfg.V, 3, 40, rng)
    _compare(cfg, w, ids, tg)


def test_backward_ragged_multi_tile(gpt_lib):
    # T = 300: three 128-query tiles, the last with 44 rows (a half tile partly and one wholly past T),
    # so the attention derivative's key tiles 0..2 all add into query tile 2 and its slabs past T stay empty
    cfg = GPTConfig(V=199, C=128, H=2, L=1, ctx=320, ffn=512)
    rng = np.random.Generator(np.random.PCG64(58))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, tg = make_tokens(cfg.V, 2, 300, rng)
    _compare(cfg, w, ids, tg)


def test_backward_gpt2_width_two_blocks(gpt_lib):
    # GPT-2 small widths and vocabulary (V = 50257: the padded dz rows), two blocks, 2 x 1024 tokens:
    # split-K weight products, stream-K head-table product, attention over 1024 positions
    base = workload("gpt2_small").cfg
    cfg = GPTConfig(V=base.V, C=base.C, H=base.H, L=2, ctx=base.ctx, ffn=base.ffn)
    rng = np.random.Generator(np.random.PCG64(53))
    w = make_weights(cfg, rng, scale_cproj=True)
    ids, tg = make_tokens(cfg.V, 2, 1024, rng)
    _compare(cfg, w, ids, tg)


def test_backward_full_size_properties(gpt_lib):
    # the bench workload (GPT-2 small, B = 16, T = 1024): the loss equals the forward's, every
    # gradient is finite and a second run agrees up to the reordering of fp32 sums. The attention
    # derivative adds each query tile's dQ from up to 8 key tiles in the order the CTAs finish (a few
    # 2^-24 relative per element), which flips some bf16 roundings of dqkv; every later bf16 rounding
    # of a quantity that depends on it (dx, dz, dg, ... through 12 blocks) can flip in turn, so the
    # gradients of the first layers and the embeddings differ by about 1e-3 of their norm between runs
    # (the step-level test of the attention derivative bounds the first stage to one bf16 ulp)
    from decoder_only_transformer_gpt_gb300 import binding
    wl = workload("gpt2_small")
    w, ids, tg = generate(wl)
    B, T = ids.shape
    m = binding.GPTModel(wl.cfg, w, B * T)
    d_ids, d_tg = dev_i32(ids), dev_i32(tg)
    lf = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.forward(d_ids, d_tg, lf)
    lb = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.backward(d_ids, d_tg, lb)
    assert float(lb.item()) == float(lf.item())
    g1 = {k: m.grad(k, l) for k, l in (("wte", -1), ("wpe", -1), ("lnf_g", -1), ("attn_w", 0), ("mp_w", 11),
                                          ("ln1_g", 5), ("fc_b", 3))}
    m.backward(d_ids, d_tg, lb)
    for (k, l), v in zip((("wte", -1), ("wpe", -1), ("lnf_g", -1), ("attn_w", 0), ("mp_w", 11), ("ln1_g", 5),
                          ("fc_b", 3)), g1.values()):
        v2 = m.grad(k, l)
        assert torch.isfinite(v).all() and v.abs().sum() > 0, k
        assert float((v - v2).norm() / v.norm()) < 3e-3, k
    m.close()


def test_backward_errors(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    cfg = GPTConfig(V=97, C=64, H=1, L=1, ctx=32, ffn=256)
    rng = np.random.Generator(np.random.PCG64(54))
    w = make_weights(cfg, rng, affine="random", wstd=0.1)
    ids, tg = make_tokens(cfg.V, 2, 8, rng)
    m = binding.GPTModel(cfg, w, 64)
    with pytest.raises(binding.GptError) as e:            # no gradients before the first backward
        m.grad("wte")
    assert e.value.code == binding.GPT_EINVAL
    long_ids = np.zeros((2, cfg.ctx + 1), np.int32)        # longer than the position table
    with pytest.raises(binding.GptError) as e:
        m.backward(dev_i32(long_ids), dev_i32(long_ids))
    assert e.value.code == binding.GPT_ESEQ
    tg2 = tg.copy()
    tg2[1, 2] = cfg.V                                      # a target outside [0, V), found on the device
    with pytest.raises(binding.GptError) as e:
        m.backward(dev_i32(ids), dev_i32(tg2))
    assert e.value.code == binding.GPT_ETOKEN
    m.backward(dev_i32(ids), dev_i32(tg))                  # the handle still works
    with pytest.raises(binding.GptError) as e:
        m.grad("attn_w", 1)                                # a block past the last
    assert e.value.code == binding.GPT_EINVAL
    m.close()
    f32 = GPTConfig(V=97, C=64, H=1, L=1, ctx=32, ffn=256, dtype=DT_FP32)
    mf = binding.GPTModel(f32, make_weights(f32, rng, affine="random", wstd=0.1), 64)
    with pytest.raises(binding.GptError) as e:             # the backward path is bf16 only
        mf.backward(dev_i32(ids), dev_i32(tg))
    assert e.value.code == binding.GPT_ECONFIG
    mf.close()


# ---- the optimiser step

def _w64(w):
    return {k: (np.asarray(v, np.float64).copy() if k != "layers" else
                [{n: np.asarray(a, np.float64).copy() for n, a in p.items()} for p in v]) for k, v in w.items()}


def test_adamw_step_against_oracle_and_next_gradient(gpt_lib):
    # one AdamW step from the GPU's own gradients equals the oracle's update (fp32 vs fp64); the next
    # backward then runs on the updated weights (bf16 matrices) and matches the oracle's gradient there
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import round_to_bf16
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512)
    rng = np.random.Generator(np.random.PCG64(55))
    w = make_weights(cfg, rng, affine="random", wstd=0.05)
    ids, tg = make_tokens(cfg.V, 2, 64, rng)
    m = binding.GPTModel(cfg, w, 128)
    d_ids, d_tg = dev_i32(ids), dev_i32(tg)
    m.backward(d_ids, d_tg)
    g = m.grads()
    gh = {k: host(v) for k, v in g.items() if k != "layers"}
    gh["layers"] = [{k: host(v) for k, v in p.items()} for p in g["layers"]]
    lr, b1, b2, eps, wd = 1e-2, 0.9, 0.95, 1e-8, 0.1
    m.adamw_step(lr, b1, b2, eps, wd)
    want = oracle.adamw_step(_w64(w), gh, {}, lr, b1, b2, eps, wd)
    got = {k: host(m.master(k)) for k in ("wte", "wpe", "lnf_g", "lnf_b")}
    got["layers"] = [{k: host(m.master(k, l)) for k in want["layers"][l]} for l in range(cfg.L)]
    for name, a, r in _pairs(cfg, got, want):
        assert np.max(np.abs(a - r)) <= 1e-6 + 1e-3 * lr, name
    # the weights the GPU now holds: bf16 matrices and tables, fp32 vectors
    w1 = {k: (round_to_bf16(got[k]) if k in ("wte", "wpe") else got[k].astype(np.float32))
          for k in ("wte", "wpe", "lnf_g", "lnf_b")}
    w1["layers"] = [{k: (round_to_bf16(v) if k.endswith("_w") else v.astype(np.float32)) for k, v in p.items()}
                    for p in got["layers"]]
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.backward(d_ids, d_tg, loss)
    g2 = m.grads()
    lref, ref = oracle.backward(cfg, w1, ids, tg)
    assert abs(float(loss.item()) - lref) <= TLOSS
    g2h = {k: host(v) for k, v in g2.items() if k != "layers"}
    g2h["layers"] = [{k: host(v) for k, v in p.items()} for p in g2["layers"]]
    for name, a, r in _pairs(cfg, g2h, ref):
        nr = np.linalg.norm(r)
        assert nr == 0.0 or np.linalg.norm(a - r) / nr <= REL, name
    m.close()


def test_overfit_one_batch_on_the_gpu(gpt_lib):
    # the pages' sanity check before real training: repeated steps on one batch drive its loss down
    from decoder_only_transformer_gpt_gb300 import binding
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512)
    rng = np.random.Generator(np.random.PCG64(56))
    w = make_weights(cfg, rng)
    ids, tg = make_tokens(cfg.V, 4, 64, rng)
    m = binding.GPTModel(cfg, w, 256)
    d_ids, d_tg = dev_i32(ids), dev_i32(tg)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    losses = []
    for _ in range(60):
        m.backward(d_ids, d_tg, loss, check=False)
        losses.append(float(loss.item()))
        m.adamw_step(3e-3, 0.9, 0.95, 1e-8, 0.0)
    m.status()
    m.close()
    print(f"\nloss {losses[0]:.3f} -> {losses[-1]:.3f}")
    assert abs(losses[0] - np.log(cfg.V)) < 0.05           # about ln V at initialisation
    assert losses[-1] < 0.3 * losses[0]
