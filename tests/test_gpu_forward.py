"""The whole forward pass + loss through gpt_create / gpt_forward against the oracle.

Tolerances (stated for this path): bf16 weights with fp32 accumulation:
|loss - oracle| <= 1e-2 and max |logit - oracle| <= 5e-2; fp32 mode: 1e-4 and 1e-3.
Full-size workloads are checked on sampled rows: by causality the logits of a
sequence prefix do not depend on later tokens, so the oracle runs on prefixes.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import dev_i32, host  # noqa: E402
from workloads import GPTConfig, workload, DT_FP32, DT_BF16, POST_NORM, GELU_ERF  # noqa: E402
from workloads.generate import generate, make_weights, make_tokens  # noqa: E402

TOL = {DT_BF16: (1e-2, 5e-2), DT_FP32: (1e-4, 1e-3)}


def _run(cfg, w, ids, tg, want_logits=True, max_tokens=None, on_device=False):
    from decoder_only_transformer_gpt_gb300 import binding
    B, T = ids.shape
    m = binding.GPTModel(cfg, w, max_tokens or B * T)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    logits = torch.empty((B, T, cfg.V), dtype=torch.float32, device="cuda") if want_logits else None
    m.forward(dev_i32(ids), dev_i32(tg), loss, logits)
    if on_device:
        out = (float(loss.item()), logits)
    else:
        out = (float(loss.item()), host(logits) if want_logits else None)
    m.close()
    return out


def _check(cfg, w, ids, tg):
    loss, z = _run(cfg, w, ids, tg)
    rloss, rz = oracle.forward(cfg, w, ids, tg)
    tl, tz = TOL[cfg.dtype]
    assert abs(loss - rloss) <= tl, (loss, rloss)
    err = np.max(np.abs(z - rz))
    assert err <= tz, err
    return loss, rloss, err


def test_toy_fp32_parity(gpt_lib):
    wl = workload("toy")
    w, ids, tg = generate(wl)
    _check(wl.cfg, w, ids, tg)


@pytest.mark.parametrize("affine", ["init", "random"])
def test_toy_fp32_random_affine_and_stress(gpt_lib, affine):
    wl = workload("toy")
    w, ids, tg = generate(wl, affine=affine, wstd=0.3)
    _check(wl.cfg, w, ids, tg)


@pytest.mark.parametrize("variant", ["post", "erf", "noln_f", "untied", "post_lnf"])
def test_fp32_variants(gpt_lib, variant):
    kw = {"post": dict(norm_mode=POST_NORM, final_ln=0), "erf": dict(gelu=GELU_ERF),
          "noln_f": dict(final_ln=0), "untied": dict(untied_head=1),
          "post_lnf": dict(norm_mode=POST_NORM)}[variant]
    cfg = GPTConfig(V=29, C=24, H=3, L=3, ctx=10, ffn=96, dtype=DT_FP32, **kw)
    rng = np.random.Generator(np.random.PCG64(5))
    w = make_weights(cfg, rng, affine="random", wstd=0.25)
    ids, tg = make_tokens(cfg.V, 3, 10, rng)
    _check(cfg, w, ids, tg)


@pytest.mark.parametrize("variant", ["post", "erf", "noln_f", "pre", "untied", "post_lnf"])
def test_bf16_variants(gpt_lib, variant):
    """The tensor-core path for each norm / GELU / final-LayerNorm / head variant."""
    kw = {"post": dict(norm_mode=POST_NORM, final_ln=0), "erf": dict(gelu=GELU_ERF),
          "noln_f": dict(final_ln=0), "pre": {}, "untied": dict(untied_head=1),
          "post_lnf": dict(norm_mode=POST_NORM)}[variant]
    cfg = GPTConfig(V=300, C=128, H=2, L=2, ctx=80, ffn=512, dtype=DT_BF16, **kw)
    rng = np.random.Generator(np.random.PCG64(11))
    w = make_weights(cfg, rng, affine="random", wstd=0.02)     # GPT-2 initialisation scale
    ids, tg = make_tokens(cfg.V, 3, 80, rng)
    _check(cfg, w, ids, tg)


def test_minigpt_bf16_parity(gpt_lib):
    wl = workload("minigpt")
    w, ids, tg = generate(wl, affine="random")
    _check(wl.cfg, w, ids, tg)


def test_minigpt_fp32_parity(gpt_lib):
    wl = workload("minigpt")
    cfg = GPTConfig(**{**wl.cfg.__dict__, "dtype": DT_FP32})
    w, ids, tg = generate(wl, affine="random")
    _check(cfg, w, ids, tg)


@pytest.mark.parametrize("B,T", [(2, 64), (1, 200)])
def test_gpt2_small_bf16_short(gpt_lib, B, T):
    wl = workload("gpt2_small")
    w, ids, tg = generate(wl, B=B, T=T, affine="random")
    _check(wl.cfg, w, ids, tg)


def test_gpt2_xl_width_bf16_short(gpt_lib):
    """The GPT-2 XL block shape (C = 1600, 25 heads of 64, FFN 6400: ragged 256-column tiles in
    every projection, stream-K in both residual projections) with two blocks."""
    from dataclasses import replace
    cfg = replace(workload("gpt2_xl").cfg, L=2)
    rng = np.random.Generator(np.random.PCG64(21))
    w = make_weights(cfg, rng, affine="random", wstd=0.02)
    ids, tg = make_tokens(cfg.V, 2, 200, rng)
    _check(cfg, w, ids, tg)


def test_gpt1_postnorm_bf16_short(gpt_lib):
    wl = workload("gpt1_postnorm")
    w, ids, tg = generate(wl, B=2, T=96, affine="random")
    _check(wl.cfg, w, ids, tg)


@pytest.mark.parametrize("name", ["gpt2_small", "gpt1_postnorm", "gpt2_xl"])
def test_full_size_sampled_rows(gpt_lib, name):
    """The timed configurations: full B x T on the GPU, sampled rows/prefixes on the oracle.
    GPT-2 XL (48 blocks, 1.56 B parameters) runs at B = 4 with two 64-token prefixes on the oracle."""
    wl = workload(name)
    if name == "gpt2_xl":
        wl = wl.with_shape(4, 1024)
    cfg = wl.cfg
    w, ids, tg = generate(wl)
    B, T = ids.shape
    loss, zd = _run(cfg, w, ids, tg, on_device=True)
    tl, tz = TOL[cfg.dtype]
    # row 0 prefix of 96 tokens, the last row in full (prefixes of 64 tokens at the XL size)
    rows = ((0, 64), (B - 1, 64)) if name == "gpt2_xl" else ((0, 96), (B - 1, T))
    for b, t in rows:
        z = host(zd[b, :t])
        _, rz = oracle.forward(cfg, w, ids[b:b + 1, :t])
        err = np.max(np.abs(z - rz[0]))
        assert err <= tz, (b, t, err)
        nll_ref = oracle.cross_entropy_rows(rz, tg[b:b + 1, :t])
        nll_gpu = oracle.cross_entropy_rows(z[None].astype(np.float64), tg[b:b + 1, :t])
        if name == "gpt2_xl":
            # 48 blocks: the stated bounds are on the mean loss and on each logit; a token's
            # nll moves by at most twice the logit error (log-sum-exp and target logit)
            assert abs(float(np.mean(nll_ref - nll_gpu))) <= tl
            assert np.max(np.abs(nll_ref - nll_gpu)) <= 2 * tz
        else:
            assert np.max(np.abs(nll_ref - nll_gpu)) <= tl
    # the fused loss equals the mean CE of the GPU's own stored logits (checked with torch)
    full = torch.nn.functional.cross_entropy(zd.view(-1, cfg.V).double(), dev_i32(tg).view(-1).long())
    assert abs(float(full) - loss) < 1e-3


@pytest.mark.parametrize("B,T", [(16, 1024), (32, 1024), (1, 1024), (16, 777)])
def test_sweep_shapes_against_oracle(gpt_lib, B, T):
    """The GPT-2-small sweep (seed 4, Zipf ids) at each of its batch shapes, B = 16, T = 1024 being the
    timed configuration: the whole batch runs on the GPU with logits stored; sampled rows (a 96-token
    prefix of row 0, a 64-token prefix of the middle row, the last row in full) match the oracle
    logit by logit (5e-2) and token by token in the loss (1e-2); the fused loss equals the mean
    cross-entropy of the GPU's own logits, and the logits-free run (the timed path) gives the same loss."""
    wl = workload("gpt2_sweep")
    cfg = wl.cfg
    w, ids, tg = generate(wl, B=B, T=T)
    loss, zd = _run(cfg, w, ids, tg, on_device=True)
    loss_fused, _ = _run(cfg, w, ids, tg, want_logits=False)
    assert loss_fused == loss, (loss_fused, loss)
    tl, tz = TOL[cfg.dtype]
    rows = {(0, min(96, T)), (B // 2, 64), (B - 1, T)}
    nll_gpu_rows, nll_ref_rows = [], []
    for b, t in sorted(rows):
        z = host(zd[b, :t])
        _, rz = oracle.forward(cfg, w, ids[b:b + 1, :t])
        err = np.max(np.abs(z - rz[0]))
        assert err <= tz, (b, t, err)
        nll_ref = oracle.cross_entropy_rows(rz, tg[b:b + 1, :t])
        nll_gpu = oracle.cross_entropy_rows(z[None].astype(np.float64), tg[b:b + 1, :t])
        assert np.max(np.abs(nll_ref - nll_gpu)) <= tl, (b, t)
        if t == T:
            nll_gpu_rows.append(nll_gpu)
            nll_ref_rows.append(nll_ref)
    # the full rows' mean loss, oracle against GPU
    assert abs(float(np.concatenate(nll_gpu_rows).mean() - np.concatenate(nll_ref_rows).mean())) <= tl
    full = torch.nn.functional.cross_entropy(zd.view(-1, cfg.V).double(), dev_i32(tg).view(-1).long())
    assert abs(float(full) - loss) < 1e-4, (float(full), loss)


def test_causal_invariance_bitwise(gpt_lib):
    wl = workload("minigpt")
    w, ids, tg = generate(wl, affine="random")
    _, z0 = _run(wl.cfg, w, ids, tg)
    ids2 = ids.copy()
    t = 40
    ids2[:, t + 1:] = (ids2[:, t + 1:] + 7) % wl.cfg.V
    _, z1 = _run(wl.cfg, w, ids2, tg)
    assert np.array_equal(z0[:, :t + 1], z1[:, :t + 1])
    assert not np.array_equal(z0[:, t + 1:], z1[:, t + 1:])


def test_determinism(gpt_lib):
    wl = workload("minigpt")
    w, ids, tg = generate(wl)
    a = _run(wl.cfg, w, ids, tg)
    b = _run(wl.cfg, w, ids, tg)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_forward_host_matches_device(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    wl = workload("minigpt")
    w, ids, tg = generate(wl)
    m = binding.GPTModel(wl.cfg, w, 512)
    loss_h, z_h = m.forward_host(ids, tg, want_logits=True)
    loss_d = torch.zeros(1, dtype=torch.float32, device="cuda")
    z_d = torch.empty((*ids.shape, wl.cfg.V), dtype=torch.float32, device="cuda")
    m.forward(dev_i32(ids), dev_i32(tg), loss_d, z_d)
    assert loss_h == float(loss_d.item())
    assert np.array_equal(z_h, z_d.cpu().numpy())
    m.close()


def test_errors(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    wl = workload("minigpt")
    w, ids, tg = generate(wl)
    m = binding.GPTModel(wl.cfg, w, 256)
    with pytest.raises(binding.GptError) as e:               # T > ctx
        m.forward(dev_i32(np.zeros((1, 129), np.int32)))
    assert e.value.code == binding.GPT_ESEQ
    with pytest.raises(binding.GptError) as e:               # B*T > max_tokens
        m.forward(dev_i32(np.zeros((3, 128), np.int32)))
    assert e.value.code == binding.GPT_EINVAL
    bad = ids.copy()
    bad[1, 3] = wl.cfg.V
    with pytest.raises(binding.GptError) as e:
        m.forward_host(bad, tg)
    assert e.value.code == binding.GPT_ETOKEN
    badt = tg.copy()
    badt[0, 0] = -1
    with pytest.raises(binding.GptError) as e:
        m.forward_host(ids, badt)
    assert e.value.code == binding.GPT_ETOKEN
    loss, _ = m.forward_host(ids, tg)                        # the handle still works
    assert np.isfinite(loss)
    m.close()


def test_time_step_probe_through_replayed_graphs(gpt_lib):
    """The timing probe on the captured forward. The first probed call captures the graph with the
    probe's event-record nodes; later calls replay it with the nodes pointed at their own events
    (runtime-created events) or capture it again (PyTorch's events, which the driver does not let
    a replay retarget). Every call gives the same loss and a timed interval."""
    import bench
    from decoder_only_transformer_gpt_gb300 import binding
    wl = workload("minigpt")
    w, ids, tg = generate(wl)
    B, T = ids.shape
    m = binding.GPTModel(wl.cfg, w, B * T)
    d_ids, d_tg = dev_i32(ids), dev_i32(tg)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    rte = bench.RuntimeEvents()
    losses = []
    for k in range(6):
        if k < 3:
            a, b = rte.create(), rte.create()
            m.lib.gpt_time_step(m.handle, 5, 1, a, b)                      # c_fc of block 1
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            e1.record()
            m.lib.gpt_time_step(m.handle, 5, 1, e0.cuda_event, e1.cuda_event)
        m.forward(d_ids, d_tg, loss, None, check=True)
        assert m.lib.gpt_last_probe_hits(m.handle) == 1
        torch.cuda.synchronize()
        if k < 3:
            assert rte.elapsed_ms(a, b) > 0.0
            rte.destroy(a)
            rte.destroy(b)
        else:
            assert e0.elapsed_time(e1) > 0.0
        losses.append(float(loss.item()))
    m.forward(d_ids, d_tg, loss, None, check=True)                          # no probe: another graph
    losses.append(float(loss.item()))
    assert len(set(losses)) == 1
    m.close()


def test_bounded_wait_expires_and_the_handle_recovers(gpt_lib):
    """Failure detection without a GPU fault: the armed forward's stream-K projections (mlp c_proj,
    K = 3072, 168 tiles on the GPU's SMs) wait on partial-tile flags that nothing sets, with a limit
    of 2e6 SM cycles (about 1 ms). Every such wait must expire and the kernels return; gpt_status
    then reports GPT_EDEVICE, and the next forwards on the same handle give the loss of the
    undisturbed run bit for bit (the flags the aborted launches left set were cleared)."""
    import time
    from decoder_only_transformer_gpt_gb300 import binding
    cfg = GPTConfig(V=1000, C=768, H=12, L=2, ctx=1024, ffn=3072)
    rng = np.random.Generator(np.random.PCG64(31))
    w = make_weights(cfg, rng, affine="random", wstd=0.02)
    ids, tg = make_tokens(cfg.V, 7, 1024, rng)
    m = binding.GPTModel(cfg, w, 7 * 1024)
    d_ids, d_tg = dev_i32(ids), dev_i32(tg)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.forward(d_ids, d_tg, loss, None, check=True)
    ref = float(loss.item())
    m.debug_expire_waits(2_000_000)
    t0 = time.perf_counter()
    m.forward(d_ids, d_tg, loss, None, check=False)
    with pytest.raises(binding.GptError) as e:
        m.status()
    assert e.value.code == binding.GPT_EDEVICE
    assert time.perf_counter() - t0 < 10.0              # the waits ended at their short limit
    for _ in range(3):
        m.forward(d_ids, d_tg, loss, None, check=True)
        assert float(loss.item()) == ref
    m.close()
