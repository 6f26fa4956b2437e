"""Plain CPU oracle of the DeepSeek-V4 attention O-projection hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``deepseek_v4_attention_gb300``) and does not
import it; the two meet only through the seeded input generators in
``dsv4_inputs``.

The arithmetic lives in ``dsv4_oracle.c`` (plain C, fp64 accumulation, built
with ``-ffp-contract=off`` and no fast-math); this module only marshals numpy
arrays through ctypes.  Every entry point cites the page it follows in the C
source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsv4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, ERR_SHAPE, ERR_NULL, ERR_RANGE = 0, -1, -2, -8

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11 + OpenMP, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        sig = {
            "oracle_num_threads": (ctypes.c_int, []),
            "oracle_set_num_threads": (None, [ctypes.c_int]),
            "oracle_bf16_to_float": (ctypes.c_float, [ctypes.c_uint16]),
            "oracle_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "oracle_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "oracle_ue8m0_exponent": (ctypes.c_int, [ctypes.c_float]),
            "oracle_ue8m0_exponent_array": (None, [P, I64, P]),
            "oracle_e4m3_encode_array": (None, [P, I64, P]),
            "oracle_bf16_from_double_array": (None, [P, I64, P]),
            "oracle_inv_rope_pairs": (None, [P, P, P, P, I64, P, P]),
            "oracle_fwd_rope_pairs": (None, [P, P, P, P, I64, P, P]),
            "oracle_tma_aligned_tokens": (I64, [I64]),
            "oracle_check_quant_shapes": (ctypes.c_int, [I64] * 8),
            "oracle_inv_rope_fp8_quant": (ctypes.c_int, [P, P, P, I64, I64, I64, I64, I64, I64,
                                                         I64, P, P]),
            "oracle_block_quant_rows": (ctypes.c_int, [P, I64, I64, I64, P, P]),
            "oracle_grouped_gemm": (ctypes.c_int, [P, P, I64, I64, I64, I64, P, P, P, P]),
            "oracle_o_proj": (ctypes.c_int, [P, P, P, I64, I64, I64, I64, I64, I64, I64, I64, I64,
                                             P, P, P, P, P, P, P]),
            "oracle_inv_rope_bf16": (ctypes.c_int, [P, P, P, I64, I64, I64, I64, I64, I64, P]),
            "oracle_grouped_gemm_bf16": (ctypes.c_int, [P, P, I64, I64, I64, I64, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(x, dtype):
    """torch CPU tensor or numpy array -> contiguous numpy array viewed as dtype."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous()
        if str(x.dtype) in ("torch.bfloat16", "torch.float8_e4m3fn", "torch.uint8"):
            import torch
            x = x.view(torch.uint16 if x.element_size() == 2 else torch.uint8)
        x = x.numpy()
    return np.ascontiguousarray(x).view(dtype)


class OracleError(RuntimeError):
    def __init__(self, rc: int, what: str):
        super().__init__(f"{what}: oracle status {rc}")
        self.rc = rc


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(rc, what)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Thread count of the oracle's parallel loops (results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


# -- number formats -------------------------------------------------------------

def bf16_to_float(bits: int) -> float:
    return _load().oracle_bf16_to_float(bits)


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(q) -> np.ndarray:
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64).ravel())
    out = np.empty(q.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(q), q.size, _ptr(out))
    return out


def bf16_from_double(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_from_double_array(_ptr(x), x.size, _ptr(out))
    return out


def ue8m0_exponent(amax) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(amax, dtype=np.float32).ravel())
    out = np.empty(a.shape, dtype=np.int32)
    _load().oracle_ue8m0_exponent_array(_ptr(a), a.size, _ptr(out))
    return out


def inv_rope_pairs(a, b, c, s):
    arrs = [np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel()) for v in (a, b, c, s)]
    y0 = np.empty_like(arrs[0]); y1 = np.empty_like(arrs[0])
    _load().oracle_inv_rope_pairs(*[_ptr(v) for v in arrs], arrs[0].size, _ptr(y0), _ptr(y1))
    return y0, y1


def fwd_rope_pairs(a, b, c, s):
    arrs = [np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel()) for v in (a, b, c, s)]
    y0 = np.empty_like(arrs[0]); y1 = np.empty_like(arrs[0])
    _load().oracle_fwd_rope_pairs(*[_ptr(v) for v in arrs], arrs[0].size, _ptr(y0), _ptr(y1))
    return y0, y1


def tma_aligned_tokens(T: int) -> int:
    return int(_load().oracle_tma_aligned_tokens(T))


def check_quant_shapes(num_heads, head_dim, n_groups, heads_per_group, nope_dim, rope_dim,
                       quant_group_size, cache_last_dim) -> int:
    return int(_load().oracle_check_quant_shapes(num_heads, head_dim, n_groups, heads_per_group,
                                                 nope_dim, rope_dim, quant_group_size,
                                                 cache_last_dim))


# -- the path ------------------------------------------------------------------

def inv_rope_fp8_quant(o, positions, cache, n_groups: int, heads_per_group: int,
                       nope_dim: int = 448, rope_dim: int = 64, quant_group_size: int = 128,
                       max_pos: int | None = None):
    """O-1.  Returns (fp8 codes uint8 physical [G, T, D], scales int32 physical [G, PK, T_al]).

    The scale pad columns [T, T_al) are zero-filled here (the oracle leaves them
    untouched; the buffer starts at zero)."""
    o = _np(o, np.uint16)
    T, H, hd = o.shape
    positions = _np(positions, np.int64)
    cache = _np(cache, np.float32)
    if max_pos is None:
        max_pos = cache.shape[0]
    D = heads_per_group * (nope_dim + rope_dim)
    NB = D // quant_group_size if quant_group_size > 0 else 0
    PK = (NB + 3) // 4
    T_al = tma_aligned_tokens(T)
    out = np.zeros((n_groups, T, D), dtype=np.uint8)
    sc = np.zeros((n_groups, PK, T_al), dtype=np.int32)
    rc = _load().oracle_inv_rope_fp8_quant(_ptr(o), _ptr(positions), _ptr(cache), T, max_pos,
                                           n_groups, heads_per_group, nope_dim, rope_dim,
                                           quant_group_size, _ptr(out), _ptr(sc))
    _check(rc, "inv_rope_fp8_quant")
    return out, sc


def block_quant_rows(x_bf16_bits, quant_group_size: int = 128):
    """Per-token 1 x 128 quantisation of a bf16 [T, C] matrix -> ([T, C] codes, [PK, T_al])."""
    x = _np(x_bf16_bits, np.uint16)
    T, C = x.shape
    PK = (C // quant_group_size + 3) // 4
    out = np.zeros((T, C), dtype=np.uint8)
    sc = np.zeros((PK, tma_aligned_tokens(T)), dtype=np.int32)
    _check(_load().oracle_block_quant_rows(_ptr(x), T, C, quant_group_size, _ptr(out), _ptr(sc)),
           "block_quant_rows")
    return out, sc


def grouped_gemm(x_fp8, x_scale, w_fp8, w_scale, T: int, G: int, D: int, R: int,
                 want_fp64: bool = False):
    """O-2 (and O-3 with G = 1).  Returns bf16 bits [T, G, R] (and fp64 [T, G, R])."""
    x = _np(x_fp8, np.uint8); xs = _np(x_scale, np.int32)
    w = _np(w_fp8, np.uint8); ws = _np(w_scale, np.uint8)
    assert x.size == G * T * D and w.size == G * R * D
    z = np.empty((T, G, R), dtype=np.uint16)
    z64 = np.empty((T, G, R), dtype=np.float64) if want_fp64 else None
    _check(_load().oracle_grouped_gemm(_ptr(x), _ptr(xs), T, G, D, R, _ptr(w), _ptr(ws),
                                       _ptr(z64), _ptr(z)), "grouped_gemm")
    return (z, z64) if want_fp64 else z


def o_proj(o, positions, cache, wo_a, wo_a_scale, wo_b, wo_b_scale, *, n_groups: int,
           heads_per_group: int, o_lora_rank: int, hidden: int, nope_dim: int = 448,
           rope_dim: int = 64, quant_group_size: int = 128, max_pos: int | None = None,
           want_z: bool = False):
    """The whole O-projection.  Returns (out bf16 bits [T, hidden], out fp64 [T, hidden],
    z bf16 bits [T, G, R] or None)."""
    o = _np(o, np.uint16)
    T = o.shape[0]
    positions = _np(positions, np.int64)
    cache = _np(cache, np.float32)
    if max_pos is None:
        max_pos = cache.shape[0]
    wa = _np(wo_a, np.uint8); was = _np(wo_a_scale, np.uint8)
    wb = _np(wo_b, np.uint8); wbs = _np(wo_b_scale, np.uint8)
    out = np.empty((T, hidden), dtype=np.uint16)
    out64 = np.empty((T, hidden), dtype=np.float64)
    z = np.empty((T, n_groups, o_lora_rank), dtype=np.uint16) if want_z else None
    rc = _load().oracle_o_proj(_ptr(o), _ptr(positions), _ptr(cache), T, max_pos, n_groups,
                               heads_per_group, nope_dim, rope_dim, quant_group_size,
                               o_lora_rank, hidden, _ptr(wa), _ptr(was), _ptr(wb), _ptr(wbs),
                               _ptr(z), _ptr(out64), _ptr(out))
    _check(rc, "o_proj")
    return out, out64, z


def inv_rope_bf16(o, positions, cache, n_groups: int, heads_per_group: int,
                  nope_dim: int = 448, rope_dim: int = 64, max_pos: int | None = None):
    """quantize=False: bf16 bits, physical [G, T, D]."""
    o = _np(o, np.uint16)
    T = o.shape[0]
    positions = _np(positions, np.int64)
    cache = _np(cache, np.float32)
    if max_pos is None:
        max_pos = cache.shape[0]
    D = heads_per_group * (nope_dim + rope_dim)
    out = np.zeros((n_groups, T, D), dtype=np.uint16)
    _check(_load().oracle_inv_rope_bf16(_ptr(o), _ptr(positions), _ptr(cache), T, max_pos,
                                        n_groups, heads_per_group, nope_dim, rope_dim,
                                        _ptr(out)), "inv_rope_bf16")
    return out


def grouped_gemm_bf16(x_bf16, w_bf16, T: int, G: int, D: int, R: int, want_fp64: bool = False):
    """bf16 grouped product: x physical [G, T, D], w [G*R, D] -> bf16 bits [T, G, R]."""
    x = _np(x_bf16, np.uint16)
    w = _np(w_bf16, np.uint16)
    assert x.size == G * T * D and w.size == G * R * D
    z = np.empty((T, G, R), dtype=np.uint16)
    z64 = np.empty((T, G, R), dtype=np.float64) if want_fp64 else None
    _check(_load().oracle_grouped_gemm_bf16(_ptr(x), _ptr(w), T, G, D, R, _ptr(z64), _ptr(z)),
           "grouped_gemm_bf16")
    return (z, z64) if want_fp64 else z
