"""The fp32 products on CTA pairs (gptk_gemm_pair: clusters of two, tcgen05.mma.cta_group::2,
256 x 256 tiles) against the fp64 oracle, element by element, through the C ABI.

out (fp32) += A W^T + bias (the residual add) or out = A W^T + bias, with exact bf16 inputs; the
bound is the fp32 accumulation bound of the single-CTA tests (K 2^-23 sum|a||w|) plus the roundings
of the additions into out: one for whole tiles and stream-K (the finishing CTA adds the other's
partial before its one store), one per slice for split-K.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import dev_bf16, dev_f32, host, rand_bf16  # noqa: E402

EPS23 = 2.0 ** -23


def _inputs(M, N, K, seed, bias=True):
    rng = np.random.default_rng(seed)
    A = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.5)
    b = rng.standard_normal(N).astype(np.float32) if bias else None
    x0 = rng.standard_normal((M, N)).astype(np.float32)
    return A, W, b, x0


def _check_rows(A, W, b, x0, got, r0, r1, adds):
    K = A.shape[1]
    ref = oracle.linear(A[r0:r1], W, b if b is not None else np.zeros(W.shape[0], np.float32))
    if x0 is not None:
        ref = ref + x0[r0:r1].astype(np.float64)
    tol = K * EPS23 * (np.abs(A[r0:r1]).astype(np.float64) @ np.abs(W).astype(np.float64).T) + 1e-6
    tol = tol + (3 + adds) * EPS23 * np.abs(ref)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"rows {r0}:{r1}: {bad.sum()} of {bad.size} outside bound; worst {np.max(np.abs(got - ref) - tol)}"


def _run(M, N, K, seed, ksplit=0, bias=True, store=False):
    """store: out = A W^T + bias over a buffer of NaNs (every element must be written)."""
    from decoder_only_transformer_gpt_gb300 import binding
    A, W, b, x0 = _inputs(M, N, K, seed, bias)
    if store:
        x0 = None
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    else:
        out = dev_f32(x0)
    epi = binding.EPI_F32 if store else binding.EPI_BIAS_RESID
    binding.gemm_pair(dev_bf16(A), dev_bf16(W), dev_f32(b) if b is not None else None, out, ksplit, epi)
    binding.status()
    return A, W, b, x0, out


# With 76 resident pairs (152 SMs): (256, 256, 64) one pair tile; (300, 520, 192) two row tiles, the
# second CTA of the second one entirely past M (its A box reads zeros, its stores are clipped) and a
# ragged last column tile; (1, 8, 8) a single row; (129, 768, 3072) the second CTA's rows start at 128;
# (200, 2304, 768) nine column tiles; (2000, 3072, 768) 96 tiles, more than the pairs.
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 520, 192), (1, 8, 8), (129, 768, 3072), (200, 2304, 768),
                                   (2000, 3072, 768)])
def test_gemm_pair_whole_tiles(gpt_lib, M, N, K):
    A, W, b, x0, out = _run(M, N, K, seed=M + N + K)
    _check_rows(A, W, b, x0, host(out), 0, M, 1)


# Stream-K on pairs (K >= 1536, tiles not a whole number of waves): (6500, 768, 3072) 78 pair tiles,
# (4000, 2304, 1544) 144 tiles with a ragged last K block, (5000, 1600, 1600) 140 tiles with a ragged
# last column tile (the GPT-2 XL width).
@pytest.mark.parametrize("M,N,K", [(6500, 768, 3072), (4000, 2304, 1544), (5000, 1600, 1600)])
@pytest.mark.parametrize("store", [False, True])
def test_gemm_pair_stream_k(gpt_lib, M, N, K, store):
    A, W, b, x0, out = _run(M, N, K, seed=K, store=store)
    _check_rows(A, W, b, x0, host(out), 0, M, 1)


@pytest.mark.parametrize("M,N,K", [(300, 520, 192), (129, 768, 2304)])
def test_gemm_pair_store_whole_tiles(gpt_lib, M, N, K):
    A, W, b, x0, out = _run(M, N, K, seed=M + K, store=True)
    _check_rows(A, W, b, x0, host(out), 0, M, 1)


@pytest.mark.parametrize("M,N,K,ks", [(300, 520, 1000, 3), (4096, 768, 12800, 5), (2000, 768, 3072, 2)])
def test_gemm_pair_split_k(gpt_lib, M, N, K, ks):
    A, W, b, x0, out = _run(M, N, K, seed=K + ks, ksplit=ks, bias=False)
    _check_rows(A, W, b, x0, host(out), 0, M, ks)


@pytest.mark.parametrize("M", [16384, 32768, 12432])
def test_gemm_pair_full_size_sampled_rows(gpt_lib, M):
    """The MLP down-projection at the token counts of the timed runs (16,384 = 16 x 1024: 192 pair
    tiles, a 116-tile stream-K region then a whole wave; 32,768; the ragged 12,432 = 16 x 777). Every
    output is computed; 128-row blocks of both CTAs' halves across the schedule are checked."""
    N, K = 768, 3072
    A, W, b, x0, out = _run(M, N, K, seed=M)
    MB = (M + 127) // 128
    for mb in sorted({0, 1, 2, 3, MB // 4, MB // 2 + 1, (3 * MB) // 4, MB - 2, MB - 1}):
        r0, r1 = 128 * mb, min(M, 128 * mb + 128)
        _check_rows(A, W, b, x0, host(out[r0:r1]), r0, r1, 1)


def test_gemm_pair_deterministic(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    rng = np.random.default_rng(9)
    M, N, K = 6500, 768, 3072
    A = dev_bf16(rand_bf16(rng, (M, K)))
    W = dev_bf16(rand_bf16(rng, (N, K), 0.5))
    b = dev_f32(rng.standard_normal(N).astype(np.float32))
    outs = []
    for _ in range(3):
        out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        binding.gemm_pair(A, W, b, out, 0)
        binding.status()
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_gemm_pair_rejects_bad_arguments(gpt_lib):
    from decoder_only_transformer_gpt_gb300 import binding
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(64, dtype=torch.float32, device="cuda")
    out = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.GptError):
        binding.gemm_pair(A, W, b, out, 2)               # split-K with a bias
    with pytest.raises(binding.GptError):
        binding.gemm_pair(A, W, None, out, 5)            # more slices than K blocks
    with pytest.raises(binding.GptError):
        binding.gemm_pair(A, W, None, out, 2, binding.EPI_F32)   # split-K of a store
    with pytest.raises(binding.GptError):
        binding.gemm_pair(A, W, b, out, 0, 7)                    # no such epilogue


# bf16 outputs on pairs (the QKV projection and c_fc's epilogues): one bf16 ulp of the value on top of
# the accumulation bound, and tanh.approx's error for the GELU (as for the single-CTA kernel).
@pytest.mark.parametrize("M,N,K", [(300, 520, 192), (2000, 3072, 768), (6500, 768, 3072), (129, 2304, 768)])
@pytest.mark.parametrize("gelu", [False, True])
def test_gemm_pair_bf16_out(gpt_lib, M, N, K, gelu):
    from decoder_only_transformer_gpt_gb300 import binding
    from gpu_util import bf16_ulp
    rng = np.random.default_rng(M + N + K + gelu)
    A = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.5)
    b = rng.standard_normal(N).astype(np.float32)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    epi = binding.EPI_BIAS_GELU if gelu else binding.EPI_BIAS
    binding.gemm_pair(dev_bf16(A), dev_bf16(W), dev_f32(b), out, 0, epi)
    binding.status()
    got = host(out)
    ref_lin = oracle.linear(A, W, b)
    acc = K * EPS23 * (np.abs(A).astype(np.float64) @ np.abs(W).astype(np.float64).T) + 1e-6
    if gelu:
        ref = oracle.gelu(ref_lin)
        tol = bf16_ulp(ref) + 1.2 * acc + 0.5 * np.abs(ref_lin) * 6e-4
    else:
        ref, tol = ref_lin, bf16_ulp(ref_lin) + acc
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside bound"
