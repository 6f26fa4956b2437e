"""Shared helpers of the GPU parity tests: device setup, comparisons with the
oracle, and the tolerance the tests use.

Tolerances (written out here and used by every GEMM parity test):
  - UE8M0 scale bytes: bit-exact.
  - FP8 codes: at least 99.99% bit-exact, every other code within one E4M3 step.
  - GEMM outputs (z, out): max_i |gpu_i - ref_i| / max(|ref_i|, rms(ref)) <= 1e-2,
    with ref the fp64-accumulated product of the dequantised operands, when the
    GPU and the oracle multiply the same FP8 operands (every GEMM test on oracle
    inputs, and wo_a inside the chain).
  - The chained O-projection (out after the z re-quantisation): the GPU rounds
    z to bf16 from an fp32 tensor-core sum, the oracle from an fp64 sum, so a z
    within an fp32 rounding error of a bf16 tie may round the other way and move
    one FP8 code of zq by one step; both are results of the method.  As for the
    FP8 codes: at least 99.99 % of the outputs within 1e-2, every output within
    3e-2 (CHAIN_RTOL_ALL).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

GEMM_RTOL = 1e-2
CODE_EXACT_MIN = 0.9999
CHAIN_WITHIN_MIN = 0.9999
CHAIN_RTOL_ALL = 3e-2


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


def chain_rel_errs(gpu_bf16_bits: np.ndarray, ref64: np.ndarray) -> np.ndarray:
    g = torch.from_numpy(np.ascontiguousarray(gpu_bf16_bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    ref = ref64.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    return np.abs(g - ref) / np.maximum(np.abs(ref), rms)


def assert_chain_matches(gpu_bf16_bits: np.ndarray, ref64: np.ndarray, what: str = "out"):
    err = chain_rel_errs(gpu_bf16_bits, ref64)
    within = float((err <= GEMM_RTOL).mean()) if err.size else 1.0
    assert within >= CHAIN_WITHIN_MIN, f"{what}: only {within:.6f} within {GEMM_RTOL}"
    assert float(err.max(initial=0.0)) <= CHAIN_RTOL_ALL, f"{what}: max {err.max()}"
    return within, float(err.max(initial=0.0))
