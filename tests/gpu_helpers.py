"""Shared helpers of the GPU parity tests: device setup, comparisons with the
oracle, and the tolerance the tests use.

Tolerances (written out here and used by every GEMM parity test):
  - UE8M0 scale bytes: bit-exact.
  - FP8 codes: at least 99.99% bit-exact, every other code within one E4M3 step.
  - GEMM outputs (z, out): max_i |gpu_i - ref_i| / max(|ref_i|, rms(ref)) <= 1e-2,
    with ref the fp64-accumulated product of the dequantised operands.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

GEMM_RTOL = 1e-2
CODE_EXACT_MIN = 0.9999


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_v4_attention_gb300 import _build
    _build.build()
    return torch.device("cuda", 0)


def e4m3_step_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between two arrays of e4m3 codes (+-0 equal)."""
    def ordinal(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b))


def assert_codes_match(gpu: np.ndarray, ref: np.ndarray, what: str = "codes"):
    gpu = gpu.reshape(-1)
    ref = ref.reshape(-1)
    same = (gpu == ref) | (((gpu & 0x7F) == 0) & ((ref & 0x7F) == 0))
    frac = same.mean() if same.size else 1.0
    dist = e4m3_step_distance(gpu, ref)
    assert frac >= CODE_EXACT_MIN, f"{what}: only {frac:.6f} bit-exact"
    assert dist.max(initial=0) <= 1, f"{what}: a code differs by {dist.max()} steps"
    return frac


def gemm_rel_err(gpu_bf16_bits: np.ndarray, ref64: np.ndarray) -> float:
    g = torch.from_numpy(np.ascontiguousarray(gpu_bf16_bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    ref = ref64.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    den = np.maximum(np.abs(ref), rms)
    return float(np.max(np.abs(g - ref) / den)) if ref.size else 0.0


def to_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.uint16).numpy()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.numpy()
