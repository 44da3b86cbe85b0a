"""Helpers for the GPU parity tests: numpy <-> CUDA tensors, bf16 rounding."""
import numpy as np
import torch

from workloads import round_to_bf16


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    """A numpy array (already bf16-representable or not) as a CUDA bf16 tensor (RNE)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rand_bf16(rng, shape, scale=1.0) -> np.ndarray:
    """Normal samples rounded to bf16, returned as fp32 (exact bf16 values)."""
    return round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-30)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)
