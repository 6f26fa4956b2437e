"""Seeded synthetic inputs for the DeepSeek-V4 attention O-projection.

This module is shared by the tests, the benchmark and the smoke check, and it
feeds both the CUDA library and the CPU oracle.  It draws random numbers and
lays them out; it holds none of the method's arithmetic (no rotation, no scale
rule, no quantisation decision, no GEMM).

Workloads (sizes of the pages' DeepSeek-V4 attention: 512-dim heads split into
448 "nope" lanes and 64 rope lanes, per-128 FP8 blocks, o_lora_rank 1024,
hidden 7168):

  tiny     T=16,   G=2,  hpg=2, R=128,  o ~ N(0,1), positions U[0,4096)
  decode   T=64,   G=8,  hpg=8, R=1024, o ~ N(0,1), positions U[0,32768)
  prefill  T=8192, G=8,  hpg=8, R=1024, o ~ N(0,1) with 1% of entries x50,
           positions = four sequences 0..2047 back to back
  quant    T in {1024, 8192, 32768}, G=16, hpg=8, o ~ Student-t(3) with 0.1%
           of the 128-element blocks all zero, positions U[0,65536)
  full     T=4096, G=16, hpg=8, R=1024, hidden=7168, o ~ N(0,1),
           positions U[0,65536)

The cos||sin cache is cos(p * theta^(-2i/rope_dim)) || sin(...), theta = 1e4,
computed in float64 and stored as float32 [max_pos, rope_dim].

FP8 weights are drawn directly in their stored form: every element is the
float8_e4m3fn rounding (torch's own cast) of N(0, 1) * 64, and every 128 x 128
block gets a UE8M0 scale byte 127 + e with e uniform in {-13, -12, -11}, so the
dequantised weights have a block-wise standard deviation around 0.02.
"""
from __future__ import annotations

import dataclasses
import math

import torch

ROPE_THETA = 10000.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    n_groups: int
    heads_per_group: int
    o_lora_rank: int
    hidden: int
    max_pos: int
    seed: int
    dist: str = "normal"           # "normal" | "outliers" | "student_t"
    positions: str = "uniform"     # "uniform" | "seq4x2048"
    nope_dim: int = 448
    rope_dim: int = 64
    quant_group_size: int = 128
    weight_seed: int | None = None  # None: derived from `seed`

    @property
    def head_dim(self) -> int:
        return self.nope_dim + self.rope_dim

    @property
    def H(self) -> int:
        return self.n_groups * self.heads_per_group

    @property
    def D(self) -> int:
        return self.heads_per_group * self.head_dim

    def with_tokens(self, T: int, seed: int | None = None) -> "Workload":
        return dataclasses.replace(self, T=T, seed=self.seed if seed is None else seed)


WORKLOADS = {
    "tiny": Workload("tiny", T=16, n_groups=2, heads_per_group=2, o_lora_rank=128, hidden=256,
                     max_pos=4096, seed=0),
    "decode": Workload("decode", T=64, n_groups=8, heads_per_group=8, o_lora_rank=1024,
                       hidden=7168, max_pos=32768, seed=1),
    "prefill": Workload("prefill", T=8192, n_groups=8, heads_per_group=8, o_lora_rank=1024,
                        hidden=7168, max_pos=32768, seed=2, dist="outliers",
                        positions="seq4x2048"),
    "quant1k": Workload("quant1k", T=1024, n_groups=16, heads_per_group=8, o_lora_rank=1024,
                        hidden=7168, max_pos=65536, seed=3 + 1024, dist="student_t"),
    "quant8k": Workload("quant8k", T=8192, n_groups=16, heads_per_group=8, o_lora_rank=1024,
                        hidden=7168, max_pos=65536, seed=3 + 8192, dist="student_t"),
    "quant32k": Workload("quant32k", T=32768, n_groups=16, heads_per_group=8, o_lora_rank=1024,
                         hidden=7168, max_pos=65536, seed=3 + 32768, dist="student_t"),
    "full": Workload("full", T=4096, n_groups=16, heads_per_group=8, o_lora_rank=1024,
                     hidden=7168, max_pos=65536, seed=4),
}


def _gen(seed: int, device: torch.device | str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def cos_sin_cache(max_pos: int, rope_dim: int = 64, theta: float = ROPE_THETA) -> torch.Tensor:
    """fp32 [max_pos, rope_dim]: cos in the first half, sin in the second."""
    half = rope_dim // 2
    inv_freq = theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / rope_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32).contiguous()


def attention_output(w: Workload, gen: torch.Generator | None = None,
                     device: torch.device | str = "cpu") -> torch.Tensor:
    """bf16 o [T, H, head_dim] with the workload's value distribution, drawn on
    `device` (with a CPU generator by default; on another device the same
    recipe runs on that device's random stream, so the values differ)."""
    gen = gen or _gen(w.seed, device)
    shape = (w.T, w.H, w.head_dim)
    if w.dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    elif w.dist == "outliers":
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
        hit = torch.rand(shape, generator=gen, device=device) < 0.01
        x = torch.where(hit, x * 50.0, x)
    elif w.dist == "student_t":
        z = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
        chi2 = torch.zeros(shape, dtype=torch.float32, device=device)
        for _ in range(3):
            chi2 += torch.randn(shape, generator=gen, dtype=torch.float32, device=device).square()
        x = z / torch.sqrt(chi2 / 3.0)
        del chi2
        qgs = w.quant_group_size
        blocks = x.view(w.T * w.H * (w.head_dim // qgs), qgs)
        nblk = blocks.shape[0]
        nzero = max(1, round(nblk * 0.001))
        idx = torch.randperm(nblk, generator=gen, device=device)[:nzero]
        blocks[idx] = 0.0
    else:
        raise ValueError(w.dist)
    return x.to(torch.bfloat16).contiguous()


def positions(w: Workload, gen: torch.Generator | None = None) -> torch.Tensor:
    gen = gen or _gen(w.seed + 7919)
    if w.positions == "uniform":
        return torch.randint(0, w.max_pos, (w.T,), generator=gen, dtype=torch.int64)
    if w.positions == "seq4x2048":
        seq = torch.arange(2048, dtype=torch.int64)
        p = seq.repeat(math.ceil(w.T / 2048))[: w.T]
        return p.contiguous()
    raise ValueError(w.positions)


def fp8_block_weight(rows: int, cols: int, seed: int):
    """(codes uint8 [rows, cols] holding float8_e4m3fn bits, UE8M0 bytes [rows/128, cols/128])."""
    assert rows % 128 == 0 and cols % 128 == 0
    gen = _gen(seed)
    x = (torch.randn((rows, cols), generator=gen, dtype=torch.float32) * 64.0).clamp_(-448.0, 448.0)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    e = torch.randint(-13, -10, (rows // 128, cols // 128), generator=gen, dtype=torch.int32)
    scale = (e + 127).to(torch.uint8).contiguous()
    return codes, scale


def bf16_weight(rows: int, cols: int, seed: int) -> torch.Tensor:
    """bf16 [rows, cols] drawn N(0, 0.02): the wo_a of a model served without FP8."""
    gen = _gen(seed)
    return (torch.randn((rows, cols), generator=gen, dtype=torch.float32) * 0.02).to(
        torch.bfloat16).contiguous()


def make_inputs(w: Workload, with_wo_b: bool = True,
                o_device: torch.device | str | None = None) -> dict:
    """All tensors of one workload: o, positions, cache, wo_a (+ wo_b), on the
    CPU; with o_device, o is drawn on that device instead (same recipe, that
    device's random stream)."""
    gen = _gen(w.seed) if o_device is None else _gen(w.seed, o_device)
    d = {
        "o": attention_output(w, gen, "cpu" if o_device is None else o_device),
        "positions": positions(w),
        "cache": cos_sin_cache(w.max_pos, w.rope_dim),
    }
    ws = w.seed if w.weight_seed is None else w.weight_seed
    d["wo_a"], d["wo_a_scale"] = fp8_block_weight(w.n_groups * w.o_lora_rank, w.D, ws + 101)
    if with_wo_b:
        d["wo_b"], d["wo_b_scale"] = fp8_block_weight(w.hidden, w.n_groups * w.o_lora_rank,
                                                      ws + 202)
    return d


def random_fp8_activation(T: int, G: int, D: int, seed: int, tma_aligned_T: int):
    """Random but valid quantised activations for the GEMM alone: codes [G, T, D] (never NaN)
    and packed UE8M0 scales [G, D/512, T_al] with bytes in [120, 130]."""
    gen = _gen(seed)
    x = (torch.randn((G, T, D), generator=gen) * 64.0).clamp_(-448.0, 448.0)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    nb = D // 128
    pk = (nb + 3) // 4
    b = torch.randint(120, 131, (G, pk * 4, tma_aligned_T), generator=gen, dtype=torch.int64)
    b[:, nb:, :] = 0
    words = b[:, 0::4] | (b[:, 1::4] << 8) | (b[:, 2::4] << 16) | (b[:, 3::4] << 24)
    words = torch.where(words >= 2**31, words - 2**32, words)
    return codes, words.to(torch.int32).contiguous()
