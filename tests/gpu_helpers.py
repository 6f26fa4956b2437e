"""Shared helpers of the GPU parity tests: device setup, comparisons with the
oracle, and the tolerances the tests use.

Tolerances (written out here and used by every parity test):
  - UE8M0 scale bytes: bit-exact.
  - FP8 codes: at least 99.99% bit-exact, every other code within one E4M3 step.
  - GEMM outputs (z, out): max_i |gpu_i - ref_i| / max(|ref_i|, rms(ref)) <= 1e-2
    (GEMM_RTOL), with ref the fp64-accumulated product of the dequantised FP8
    operands the GPU itself consumed.  Inside the O-projection those operands
    are read back from the caller's workspace: the quantised groups x for
    wo_a, the re-quantised zq for wo_b.
  - The O-projection stage by stage (check_o_proj_parts): x and its scales
    against the oracle's quantiser, zq and its scales against the oracle's
    per-128 quantisation of the oracle's bf16 z (the code criterion above;
    this also holds wo_a to its result), out against the fp64 product of the
    GPU's own zq with wo_b (GEMM_RTOL).
  - The chained output against the oracle's whole chain is a secondary check
    (chain_allowance): GEMM_RTOL plus, for every zq code that differs from
    the oracle's by one step, that step's exact effect on the output,
    step x 2^e_z x |dequantised wo_b element|.  No slack beyond that: a zq
    code that moves one step is a legitimate result of the method (the GPU
    rounds z to bf16 from an fp32 tensor-core sum, the oracle from an fp64 sum).
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


def codes_equal(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    return (gpu == ref) | (((gpu & 0x7F) == 0) & ((ref & 0x7F) == 0))


def assert_codes_match(gpu: np.ndarray, ref: np.ndarray, what: str = "codes"):
    gpu = gpu.reshape(-1)
    ref = ref.reshape(-1)
    same = codes_equal(gpu, ref)
    frac = same.mean() if same.size else 1.0
    dist = e4m3_step_distance(gpu, ref)
    assert frac >= CODE_EXACT_MIN, f"{what}: only {frac:.6f} bit-exact"
    assert dist.max(initial=0) <= 1, f"{what}: a code differs by {dist.max()} steps"
    return frac


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def rel_errs(gpu_bf16_bits: np.ndarray, ref64: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(|gpu - ref|, max(|ref|, rms(ref))) element by element."""
    g = bf16_bits_to_f64(gpu_bf16_bits)
    ref = ref64.astype(np.float64).reshape(g.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    if rms == 0.0:
        rms = 1.0        # an identically zero reference: the absolute error
    return np.abs(g - ref), np.maximum(np.abs(ref), rms)


def gemm_rel_err(gpu_bf16_bits: np.ndarray, ref64: np.ndarray) -> float:
    err, den = rel_errs(gpu_bf16_bits, ref64)
    return float(np.max(err / den)) if err.size else 0.0


def to_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.uint16).numpy()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def scale_bytes(words: np.ndarray) -> np.ndarray:
    """Packed int32 UE8M0 words [PK, n] -> bytes [4*PK, n] (block 4j+b = byte b of word j)."""
    w = np.ascontiguousarray(words).view(np.uint32)
    return np.stack([(w >> (8 * b)) & 0xFF for b in range(4)], axis=1).reshape(
        4 * w.shape[0], w.shape[1]).astype(np.int64)


def chain_allowance(zq_gpu, zq_ref, zs_bytes, wo_b, wo_b_scale, decode) -> np.ndarray:
    """Per-output effect [n, hidden] on out = zq . wo_b^T of the zq codes in
    which the GPU and the oracle differ: sum over those codes c of
    |dq(gpu code) - dq(oracle code)| * 2^e_z(t, c/128) * |dq(wo_b[h, c])|."""
    n, C = zq_gpu.shape
    wb = np.ascontiguousarray(wo_b.numpy() if hasattr(wo_b, "numpy") else wo_b)
    wbs = np.ascontiguousarray(wo_b_scale.numpy() if hasattr(wo_b_scale, "numpy")
                               else wo_b_scale).astype(np.int64)
    hidden = wb.shape[0]
    allow = np.zeros((n, hidden), dtype=np.float64)
    ts, cs = np.nonzero(~codes_equal(zq_gpu, zq_ref))
    for t, c in zip(ts, cs):
        step = abs(decode[zq_gpu[t, c]] - decode[zq_ref[t, c]]) * 2.0 ** (zs_bytes[c // 128, t] - 127)
        col = np.abs(decode[wb[:, c]]) * np.exp2(wbs[np.arange(hidden) // 128, c // 128] - 127)
        allow[t] += step * col
    return allow


def check_o_proj_parts(d: dict, w, out: torch.Tensor, workspace: torch.Tensor,
                       idx: np.ndarray | None = None) -> dict:
    """Stage-by-stage parity of one dsv4_o_proj call on the rows idx (all rows
    when None): its workspace holds x, xs, zq, zs (include/dsv4.h)."""
    import deepseek_v4_attention_gb300 as k
    import oracle
    T, G, hpg, R, hidden = w.T, w.n_groups, w.heads_per_group, w.o_lora_rank, w.hidden
    C = G * R
    if idx is None:
        idx = np.arange(T)
    n = len(idx)
    ti = torch.from_numpy(np.asarray(idx, dtype=np.int64))
    parts = k.o_proj_workspace_views(workspace, T, G, hpg, w.head_dim, R)
    torch.cuda.synchronize()
    # the oracle's whole chain on the sampled rows, with its bf16 z
    _, out64, z_ref = oracle.o_proj(d["o"][ti], d["positions"][ti], d["cache"], d["wo_a"],
                                    d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], n_groups=G,
                                    heads_per_group=hpg, o_lora_rank=R, hidden=hidden,
                                    want_z=True)
    # 1. the quantiser: codes and scales of the sampled rows
    xr, xsr = oracle.inv_rope_fp8_quant(d["o"][ti], d["positions"][ti], d["cache"], G, hpg)
    xg = parts["x"].cpu().numpy()[:, idx]
    xsg = parts["xs"].cpu().numpy()[:, :, idx]
    assert np.array_equal(xsg, xsr[:, :, :n]), "x scale words differ"
    x_frac = assert_codes_match(xg, xr, "x codes")
    # 2. wo_a + the fused re-quantisation: zq against the oracle's per-128
    #    quantisation of the oracle's bf16 z
    zqr, zsr = oracle.block_quant_rows(z_ref.reshape(n, C))
    zqg = parts["zq"].cpu().numpy()[idx]
    zsg = parts["zs"].cpu().numpy()[:, idx]
    nb = C // 128       # bytes past the last block of a packed word are not results
    assert np.array_equal(scale_bytes(zsg)[:nb], scale_bytes(zsr[:, :n])[:nb]), \
        "zq scale bytes differ"
    zq_frac = assert_codes_match(zqg, zqr, "zq codes")
    # 3. wo_b on the GPU's own zq: fp64 product, GEMM_RTOL
    n_al = oracle.tma_aligned_tokens(n)
    zs_own = np.zeros((zsg.shape[0], n_al), dtype=np.int32)
    zs_own[:, :n] = zsg
    _, o64_own = oracle.grouped_gemm(np.ascontiguousarray(zqg), zs_own, d["wo_b"],
                                     d["wo_b_scale"], n, 1, C, hidden, want_fp64=True)
    og = to_bits(out)[idx]
    wo_b_err = gemm_rel_err(og, o64_own.reshape(n, hidden))
    assert wo_b_err <= GEMM_RTOL, f"wo_b on the GPU's own zq: {wo_b_err}"
    # 4. secondary: the chained output against the oracle's chain
    err, den = rel_errs(og, out64)
    allow = chain_allowance(zqg, zqr, scale_bytes(zsg), d["wo_b"], d["wo_b_scale"],
                            oracle.e4m3_decode_table())
    excess = err - (GEMM_RTOL * den + allow)
    assert float(excess.max(initial=-1.0)) <= 0.0, \
        f"chain: {int((excess > 0).sum())} outputs beyond the derived bound"
    return {"x_exact": x_frac, "zq_exact": zq_frac, "wo_b_err": wo_b_err,
            "chain_err": float((err / den).max(initial=0.0))}
