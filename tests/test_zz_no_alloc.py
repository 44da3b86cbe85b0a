"""The allocation-free head + cross-entropy entry against the allocating one.

gptk_lmhead_ce_noalloc exists for callers that cannot allocate device memory
while they run: a server whose memory budget is fixed at start-up, a framework
whose caching allocator already holds the free device memory, or a loop that
cannot take the synchronisation an allocation may bring. It keeps its scratch in
a fixed library array instead. Here it must give the per-row losses of
gptk_lmhead_ce (which allocates its scratch per call) within the tolerance the
head's parity test uses (1e-4), on two calls in a row with different inputs, so
that a stale scratch array would show. This file sorts last so that a run that
stops at the first failure has run every other test before it.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import dev_bf16, dev_i32, rand_bf16  # noqa: E402

TOL = 1e-4


def _inputs(seed, M, V, C):
    rng = np.random.default_rng(seed)
    h = dev_bf16(rand_bf16(rng, (M, C)))
    E = dev_bf16(rand_bf16(rng, (V, C), 0.1))
    tg = dev_i32(rng.integers(0, V, size=M))
    return h, E, tg


def _reference(h, E, tg):
    from decoder_only_transformer_gpt_gb300 import binding
    nll = torch.empty(h.shape[0], dtype=torch.float32, device="cuda")
    binding.lmhead_ce(h, E, tg, nll)
    binding.status()
    return nll


@pytest.mark.parametrize("V,C", [(5000, 128), (50257, 768)])
def test_noalloc_matches_allocating_entry_twice(gpt_lib, V, C):
    from decoder_only_transformer_gpt_gb300 import binding
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, (seed, M) in enumerate(((11, 300), (12, 517))):
        h, E, tg = _inputs(seed + V, M, V, C)
        ref = _reference(h, E, tg)
        nll = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
        binding.lmhead_ce_noalloc(h, E, tg, nll, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        d = (nll - ref).abs().max().item()
        assert d <= TOL, f"call {call}: max |noalloc - allocating| = {d}"


def test_noalloc_rejects_sizes_beyond_its_scratch(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    V, C = 50257, 64
    M = 5310                                # 5310 * (2 * 197 + 1) floats > 2,097,152
    h = torch.zeros((M, C), dtype=torch.bfloat16, device="cuda")
    E = torch.zeros((V, C), dtype=torch.bfloat16, device="cuda")
    tg = torch.zeros(M, dtype=torch.int32, device="cuda")
    nll = torch.empty(M, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.GptError) as e:
        binding.lmhead_ce_noalloc(h, E, tg, nll)
    assert e.value.code == binding.GPT_EINVAL
    assert "scratch" in str(e.value)


def test_noalloc_reports_a_bad_target_and_runs_without_an_error_word(gpt_lib):
    """A target equal to V reaches the caller's error word while every other row still matches
    the allocating entry; with no error word (NULL) the result on valid inputs is the same."""
    from decoder_only_transformer_gpt_gb300 import binding
    V, C, M = 5000, 128, 300
    h, E, tg = _inputs(77, M, V, C)
    ref = _reference(h, E, tg)
    bad = tg.clone()
    bad[17] = V
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nll = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    binding.lmhead_ce_noalloc(h, E, bad, nll, err)
    torch.cuda.synchronize()
    assert int(err.item()) != 0
    keep = torch.ones(M, dtype=torch.bool, device="cuda")
    keep[17] = False
    assert (nll[keep] - ref[keep]).abs().max().item() <= TOL
    nll2 = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    binding.lmhead_ce_noalloc(h, E, tg, nll2, None)
    torch.cuda.synchronize()
    assert (nll2 - ref).abs().max().item() <= TOL
