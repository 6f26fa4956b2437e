"""DeepSeek-V4 attention O-projection on GB300 (sm_103a).

A thin ctypes binding over the C ABI in include/dsv4.h (libdsv4.so, built
in-tree by ``_build.build()``).  The functions below only marshal torch CUDA
tensors into pointers and sizes; every step of the path runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or the device
is not an sm_103 GPU, the calls raise.

    dsv4_inv_rope_fp8_quant  fused inverse RoPE + block-scaled FP8 quantisation
    dsv4_grouped_wo_a        grouped wo_a block-scaled FP8 GEMM
    dsv4_o_proj              the whole O-projection (quant -> wo_a -> wo_b)
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsv4.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "dsv4.h")

DSV4_OK = 0
STATUS = {
    0: "DSV4_OK", -1: "DSV4_ERR_SHAPE", -2: "DSV4_ERR_NULL", -3: "DSV4_ERR_ALIGN",
    -4: "DSV4_ERR_UNSUPPORTED", -5: "DSV4_ERR_WORKSPACE", -6: "DSV4_ERR_CUDA",
    -7: "DSV4_ERR_TIMEOUT", -8: "DSV4_ERR_RANGE",
}
_NAME_TO_CODE = {v: k for k, v in STATUS.items()}


class DSV4Error(RuntimeError):
    def __init__(self, rc: int, what: str):
        super().__init__(f"{what} failed: {STATUS.get(rc, rc)}")
        self.rc = rc
        self.name = STATUS.get(rc, str(rc))


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libdsv4.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(or python -m deepseek_v4_attention_gb300._build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.dsv4_inv_rope_fp8_quant.argtypes = [P, P, P, I64, I64, I, I, I, I, I, P, P, P]
    lib.dsv4_inv_rope_fp8_quant.restype = I
    lib.dsv4_grouped_wo_a.argtypes = [P, P, I64, I, I, I, P, P, P, P]
    lib.dsv4_grouped_wo_a_ex.argtypes = [P, P, I64, I, I, I, P, P, P, ctypes.c_uint, P]
    lib.dsv4_grouped_wo_a_ex.restype = I
    lib.dsv4_inv_rope_grouped_wo_a.argtypes = [P, P, P, I64, I64, I, I, I, I, I, I, P, P, P, P]
    lib.dsv4_inv_rope_grouped_wo_a.restype = I
    lib.dsv4_grouped_wo_a.restype = I
    lib.dsv4_o_proj_workspace_bytes.argtypes = [I64, I, I, I, I]
    lib.dsv4_o_proj_workspace_bytes.restype = ctypes.c_size_t
    lib.dsv4_o_proj.argtypes = [P, P, P, I64, I64, I, I, I, I, I, I, I, P, P, P, P, P, P,
                                ctypes.c_size_t, P]
    lib.dsv4_o_proj.restype = I
    lib.dsv4_o_proj_with_events.argtypes = [P, P, P, I64, I64, I, I, I, I, I, I, I, P, P, P, P,
                                            P, P, ctypes.c_size_t, P, P]
    lib.dsv4_o_proj_with_events.restype = I
    lib.dsv4_o_proj_static.argtypes = [P, P, P, I64, I64, I, I, I, I, I, I, I, P, P, P, P, P, P]
    lib.dsv4_o_proj_static.restype = I
    lib.dsv4_o_proj_partial.argtypes = [P, P, P, I64, I64, I, I, I, I, I, I, I, P, P, P, P, P, P,
                                        ctypes.c_size_t, P]
    lib.dsv4_o_proj_partial.restype = I
    lib.dsv4_sum_partials.argtypes = [P, I, I64, P, P]
    lib.dsv4_sum_partials.restype = I
    lib.dsv4_rope_quant_unsupported_reason.argtypes = [I, I, I, ctypes.POINTER(ctypes.c_char_p)]
    lib.dsv4_rope_quant_unsupported_reason.restype = I
    lib.dsv4_o_proj_prequant_workspace_bytes.argtypes = [I64, I, I]
    lib.dsv4_o_proj_prequant_workspace_bytes.restype = ctypes.c_size_t
    lib.dsv4_o_proj_prequant.argtypes = [P, P, I64, I, I, I, I, I, P, P, P, P, P, P,
                                         ctypes.c_size_t, P]
    lib.dsv4_o_proj_prequant.restype = I
    lib.dsv4_static_scratch_bytes.argtypes = []
    lib.dsv4_static_scratch_bytes.restype = ctypes.c_size_t
    lib.dsv4_status_string.argtypes = [I]
    lib.dsv4_status_string.restype = ctypes.c_char_p
    lib.dsv4_device_status.argtypes = [P, I]
    lib.dsv4_device_status.restype = I
    lib.dsv4_inv_rope_bf16.argtypes = [P, P, P, I64, I64, I, I, I, I, P, P]
    lib.dsv4_inv_rope_bf16.restype = I
    lib.dsv4_grouped_wo_a_bf16.argtypes = [P, I64, I, I, I, P, P, P]
    lib.dsv4_grouped_wo_a_bf16.restype = I
    lib.dsv4_selftest_wait_timeout.argtypes = [I64, P]
    lib.dsv4_selftest_wait_timeout.restype = I
    lib.dsv4_last_launch_count.argtypes = []
    lib.dsv4_last_launch_count.restype = I
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/dsv4.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(dsv4_\w+)\s*\(", text)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(rc: int, what: str):
    if rc != DSV4_OK:
        raise DSV4Error(rc, what)


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def tma_aligned_tokens(T: int) -> int:
    return (T + 3) // 4 * 4


_FP8 = (torch.float8_e4m3fn, torch.uint8)
_SCALE8 = (torch.uint8, torch.float8_e8m0fnu) if hasattr(torch, "float8_e8m0fnu") else (torch.uint8,)


def dsv4_inv_rope_fp8_quant(o: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                            n_groups: int, heads_per_group: int, nope_dim: int = 448,
                            rope_dim: int = 64, quant_group_size: int = 128, *,
                            out_fp8: torch.Tensor | None = None,
                            out_scale: torch.Tensor | None = None, stream=None):
    """Returns (o_fp8 [T, G, D] float8_e4m3fn with strides (D, T*D, 1),
    o_scale [T, G, PK] int32 with strides (1, PK*T_al, T_al))."""
    lib = load_library()
    _cuda(o, "o", torch.bfloat16)
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if o.dim() != 3 or not o.is_contiguous():
        raise ValueError("o must be a contiguous [T, H, head_dim] tensor")
    if not positions.is_contiguous() or not cos_sin_cache.is_contiguous():
        raise ValueError("positions and cos_sin_cache must be contiguous")
    T, H, hd = o.shape
    if H != n_groups * heads_per_group:
        raise DSV4Error(-1, "dsv4_inv_rope_fp8_quant (num_heads != n_groups * heads_per_group)")
    if hd != nope_dim + rope_dim or cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != rope_dim:
        raise DSV4Error(-1, "dsv4_inv_rope_fp8_quant (head_dim / cache shape)")
    if positions.numel() != T:
        raise DSV4Error(-1, "dsv4_inv_rope_fp8_quant (positions length)")
    D = heads_per_group * hd
    PK = (D // quant_group_size + 3) // 4 if quant_group_size > 0 else 0
    T_al = tma_aligned_tokens(T)
    if out_fp8 is None:
        out_fp8 = torch.empty((n_groups, T, D), dtype=torch.float8_e4m3fn, device=o.device)
    if out_scale is None:
        out_scale = torch.empty((n_groups, PK, T_al), dtype=torch.int32, device=o.device)
    rc = lib.dsv4_inv_rope_fp8_quant(o.data_ptr(), positions.data_ptr(), cos_sin_cache.data_ptr(),
                                     T, cos_sin_cache.shape[0], n_groups, heads_per_group,
                                     nope_dim, rope_dim, quant_group_size, out_fp8.data_ptr(),
                                     out_scale.data_ptr(), _stream(stream))
    _check(rc, "dsv4_inv_rope_fp8_quant")
    return out_fp8.transpose(0, 1), out_scale.permute(2, 0, 1)[:T]


OVERLAP_PREVIOUS = 1   # DSV4_OVERLAP_PREVIOUS


def dsv4_grouped_wo_a(x_fp8: torch.Tensor, x_scale: torch.Tensor, w_fp8: torch.Tensor,
                      w_scale: torch.Tensor, n_groups: int, o_lora_rank: int, *,
                      z: torch.Tensor | None = None, overlap_previous: bool = False,
                      stream=None) -> torch.Tensor:
    """x_fp8: the [T, G, D] view (strides (D, T*D, 1)) the quantiser returns;
    x_scale: the matching [T, G, PK] view.  Returns bf16 z [T, G, R].
    overlap_previous: launch so that the kernel starts under the previous
    kernel of the stream, reading only the weights until that one completes
    (the caller guarantees that it does not write them)."""
    lib = load_library()
    _cuda(x_fp8, "x_fp8", _FP8)
    _cuda(x_scale, "x_scale", torch.int32)
    _cuda(w_fp8, "w_fp8", _FP8)
    _cuda(w_scale, "w_scale", _SCALE8)
    T, G, D = x_fp8.shape
    if G != n_groups or x_fp8.stride() != (D, T * D, 1):
        raise ValueError("x_fp8 must be the [T, G, D] view of a physical [G, T, D] buffer")
    PK = (D // 128 + 3) // 4
    T_al = tma_aligned_tokens(T)
    if T > 0 and (tuple(x_scale.shape) != (T, G, PK) or x_scale.stride() != (1, PK * T_al, T_al)):
        raise ValueError("x_scale must be the [T, G, PK] view of a physical [G, PK, T_al] buffer")
    if tuple(w_fp8.shape) != (G * o_lora_rank, D) or not w_fp8.is_contiguous():
        raise ValueError("w_fp8 must be a contiguous [G*R, D] tensor")
    if tuple(w_scale.shape) != (G * o_lora_rank // 128, D // 128) or not w_scale.is_contiguous():
        raise ValueError("w_scale must be a contiguous [G*R/128, D/128] tensor")
    if z is None:
        z = torch.empty((T, G, o_lora_rank), dtype=torch.bfloat16, device=x_fp8.device)
    rc = lib.dsv4_grouped_wo_a_ex(x_fp8.data_ptr(), x_scale.data_ptr(), T, G, D, o_lora_rank,
                                  w_fp8.data_ptr(), w_scale.data_ptr(), z.data_ptr(),
                                  OVERLAP_PREVIOUS if overlap_previous else 0, _stream(stream))
    _check(rc, "dsv4_grouped_wo_a")
    return z


FUSED_MAX_TOKENS = 64   # DSV4_FUSED_MAX_TOKENS


def dsv4_inv_rope_grouped_wo_a(o: torch.Tensor, positions: torch.Tensor,
                               cos_sin_cache: torch.Tensor, w_fp8: torch.Tensor,
                               w_scale: torch.Tensor, n_groups: int, heads_per_group: int,
                               o_lora_rank: int, nope_dim: int = 448, rope_dim: int = 64,
                               quant_group_size: int = 128, *, z: torch.Tensor | None = None,
                               stream=None) -> torch.Tensor:
    """Quantiser fused into the grouped wo_a (decode sizes, T <= FUSED_MAX_TOKENS):
    o [T, H, 512] bf16 -> z [T, G, R] bf16, equal to dsv4_grouped_wo_a of
    dsv4_inv_rope_fp8_quant's output."""
    lib = load_library()
    _cuda(o, "o", torch.bfloat16)
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    _cuda(w_fp8, "w_fp8", _FP8)
    _cuda(w_scale, "w_scale", _SCALE8)
    if o.dim() != 3 or not o.is_contiguous():
        raise ValueError("o must be a contiguous [T, H, head_dim] tensor")
    if not positions.is_contiguous() or not cos_sin_cache.is_contiguous():
        raise ValueError("positions and cos_sin_cache must be contiguous")
    T, H, hd = o.shape
    if H != n_groups * heads_per_group or hd != nope_dim + rope_dim:
        raise DSV4Error(-1, "dsv4_inv_rope_grouped_wo_a (o shape)")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != rope_dim or positions.numel() != T:
        raise DSV4Error(-1, "dsv4_inv_rope_grouped_wo_a (cache / positions shape)")
    D = heads_per_group * hd
    if tuple(w_fp8.shape) != (n_groups * o_lora_rank, D) or not w_fp8.is_contiguous():
        raise ValueError("w_fp8 must be a contiguous [G*R, D] tensor")
    if tuple(w_scale.shape) != (n_groups * o_lora_rank // 128, D // 128) or \
            not w_scale.is_contiguous():
        raise ValueError("w_scale must be a contiguous [G*R/128, D/128] tensor")
    if z is None:
        z = torch.empty((T, n_groups, o_lora_rank), dtype=torch.bfloat16, device=o.device)
    rc = lib.dsv4_inv_rope_grouped_wo_a(o.data_ptr(), positions.data_ptr(),
                                        cos_sin_cache.data_ptr(), T, cos_sin_cache.shape[0],
                                        n_groups, heads_per_group, nope_dim, rope_dim,
                                        quant_group_size, o_lora_rank, w_fp8.data_ptr(),
                                        w_scale.data_ptr(), z.data_ptr(), _stream(stream))
    _check(rc, "dsv4_inv_rope_grouped_wo_a")
    return z


def dsv4_inv_rope_bf16(o: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                       n_groups: int, heads_per_group: int, nope_dim: int = 448,
                       rope_dim: int = 64, *, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """quantize=False: returns the bf16 inverse-rotated groups [T, G, D] with
    strides (D, T*D, 1)."""
    lib = load_library()
    _cuda(o, "o", torch.bfloat16)
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if o.dim() != 3 or not o.is_contiguous():
        raise ValueError("o must be a contiguous [T, H, head_dim] tensor")
    T, H, hd = o.shape
    if H != n_groups * heads_per_group or hd != nope_dim + rope_dim or positions.numel() != T:
        raise DSV4Error(-1, "dsv4_inv_rope_bf16 (shapes)")
    D = heads_per_group * hd
    if out is None:
        out = torch.empty((n_groups, T, D), dtype=torch.bfloat16, device=o.device)
    rc = lib.dsv4_inv_rope_bf16(o.data_ptr(), positions.data_ptr(), cos_sin_cache.data_ptr(), T,
                                cos_sin_cache.shape[0], n_groups, heads_per_group, nope_dim,
                                rope_dim, out.data_ptr(), _stream(stream))
    _check(rc, "dsv4_inv_rope_bf16")
    return out.transpose(0, 1)


def dsv4_grouped_wo_a_bf16(x_bf16: torch.Tensor, w_bf16: torch.Tensor, n_groups: int,
                           o_lora_rank: int, *, z: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """bf16 grouped product (bmm path): x [T, G, D] view of a physical [G, T, D]
    buffer, w [G*R, D]; returns bf16 z [T, G, R]."""
    lib = load_library()
    _cuda(x_bf16, "x_bf16", torch.bfloat16)
    _cuda(w_bf16, "w_bf16", torch.bfloat16)
    T, G, D = x_bf16.shape
    if G != n_groups or x_bf16.stride() != (D, T * D, 1):
        raise ValueError("x_bf16 must be the [T, G, D] view of a physical [G, T, D] buffer")
    if tuple(w_bf16.shape) != (G * o_lora_rank, D) or not w_bf16.is_contiguous():
        raise ValueError("w_bf16 must be a contiguous [G*R, D] tensor")
    if z is None:
        z = torch.empty((T, G, o_lora_rank), dtype=torch.bfloat16, device=x_bf16.device)
    rc = lib.dsv4_grouped_wo_a_bf16(x_bf16.data_ptr(), T, G, D, o_lora_rank, w_bf16.data_ptr(),
                                    z.data_ptr(), _stream(stream))
    _check(rc, "dsv4_grouped_wo_a_bf16")
    return z


def dsv4_o_proj_workspace_bytes(num_tokens: int, n_groups: int, heads_per_group: int,
                                head_dim: int, o_lora_rank: int) -> int:
    return int(load_library().dsv4_o_proj_workspace_bytes(num_tokens, n_groups, heads_per_group,
                                                          head_dim, o_lora_rank))


def _round256(x: int) -> int:
    return (x + 255) // 256 * 256


def o_proj_workspace_views(workspace: torch.Tensor, num_tokens: int, n_groups: int,
                           heads_per_group: int, head_dim: int, o_lora_rank: int) -> dict:
    """Views of the parts of dsv4_o_proj's workspace, in the order and at the
    256-byte-aligned offsets include/dsv4.h fixes, holding the intermediate
    results of the last call that used it:

        x   uint8 [G, T, D]        the quantised groups (e4m3 codes)
        xs  int32 [G, PK, T_al]    their packed UE8M0 scales
        zq  uint8 [T, G*R]         the per-128 re-quantised bf16 z (e4m3 codes)
        zs  int32 [PKC, T_al]      their packed UE8M0 scales, PKC = ceil(G*R/512)
    """
    T, G, R = num_tokens, n_groups, o_lora_rank
    D = heads_per_group * head_dim
    PK = (D // 128 + 3) // 4
    C = G * R
    PKC = (C // 128 + 3) // 4
    T_al = tma_aligned_tokens(T)
    ws = workspace.view(torch.uint8)
    off = 0

    def take(nbytes):
        nonlocal off
        part = ws[off:off + nbytes]
        off += _round256(nbytes)
        return part

    x = take(G * T * D).view(G, T, D)
    xs = take(G * PK * T_al * 4).view(torch.int32).view(G, PK, T_al)
    zq = take(T * C).view(T, C)
    zs = take(PKC * T_al * 4).view(torch.int32).view(PKC, T_al)
    return {"x": x, "xs": xs, "zq": zq, "zs": zs}


def _check_o_proj_weights(wo_a, wo_a_scale, wo_b, wo_b_scale, C: int, D: int) -> int:
    """dtype, layout and shape checks of the two projections' weights; returns hidden."""
    for t, n in ((wo_a, "wo_a"), (wo_b, "wo_b")):
        _cuda(t, n, _FP8)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((wo_a_scale, "wo_a_scale"), (wo_b_scale, "wo_b_scale")):
        _cuda(t, n, _SCALE8)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    hidden = wo_b.shape[0]
    if tuple(wo_a.shape) != (C, D) or tuple(wo_b.shape) != (hidden, C):
        raise ValueError("weight shapes must be wo_a [G*R, D] and wo_b [hidden, G*R]")
    if tuple(wo_a_scale.shape) != (C // 128, D // 128) or \
            tuple(wo_b_scale.shape) != (hidden // 128, C // 128):
        raise ValueError("weight scales must be [rows/128, cols/128]")
    return hidden


def _check_o(o, positions, cos_sin_cache, n_groups, heads_per_group, what):
    _cuda(o, "o", torch.bfloat16)
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if o.dim() != 3 or not o.is_contiguous():
        raise ValueError("o must be a contiguous [T, H, head_dim] tensor")
    T, H, hd = o.shape
    if H != n_groups * heads_per_group or positions.numel() != T:
        raise DSV4Error(-1, f"{what} (head count / positions)")
    return T, hd


def dsv4_o_proj(o: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                wo_a: torch.Tensor, wo_a_scale: torch.Tensor, wo_b: torch.Tensor,
                wo_b_scale: torch.Tensor, *, n_groups: int, heads_per_group: int,
                o_lora_rank: int, nope_dim: int = 448, rope_dim: int = 64,
                quant_group_size: int = 128, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stage_events=None,
                stream=None) -> torch.Tensor:
    """The whole O-projection: returns bf16 out [T, hidden].

    stage_events: optional list of 4 torch.cuda.Event(enable_timing=True),
    recorded before the first kernel and after each of the three kernels."""
    lib = load_library()
    T, hd = _check_o(o, positions, cos_sin_cache, n_groups, heads_per_group, "dsv4_o_proj")
    C = n_groups * o_lora_rank
    D = heads_per_group * hd
    hidden = _check_o_proj_weights(wo_a, wo_a_scale, wo_b, wo_b_scale, C, D)
    need = dsv4_o_proj_workspace_bytes(T, n_groups, heads_per_group, hd, o_lora_rank)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=o.device)
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.bfloat16, device=o.device)
    args = (o.data_ptr(), positions.data_ptr(), cos_sin_cache.data_ptr(), cos_sin_cache.shape[0],
            T, n_groups, heads_per_group, nope_dim, rope_dim, quant_group_size, o_lora_rank,
            hidden, wo_a.data_ptr(), wo_a_scale.data_ptr(), wo_b.data_ptr(),
            wo_b_scale.data_ptr(), out.data_ptr(), workspace.data_ptr(), workspace.numel())
    if stage_events is None:
        rc = lib.dsv4_o_proj(*args, _stream(stream))
    else:
        if len(stage_events) != 4:
            raise ValueError("stage_events must hold 4 events")
        for ev in stage_events:
            if not ev.cuda_event:   # torch creates the event on its first record
                ev.record(torch.cuda.current_stream() if stream is None else stream)
        handles = (ctypes.c_void_p * 4)(*[ev.cuda_event for ev in stage_events])
        rc = lib.dsv4_o_proj_with_events(*args, handles, _stream(stream))
    _check(rc, "dsv4_o_proj")
    return out


def dsv4_o_proj_partial(o: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                        wo_a: torch.Tensor, wo_a_scale: torch.Tensor, wo_b: torch.Tensor,
                        wo_b_scale: torch.Tensor, *, n_groups: int, heads_per_group: int,
                        o_lora_rank: int, nope_dim: int = 448, rope_dim: int = 64,
                        quant_group_size: int = 128, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One group range's share of the O-projection (its heads of o, its wo_a
    rows, its wo_b columns): returns the fp32 partial output [T, hidden]."""
    lib = load_library()
    T, hd = _check_o(o, positions, cos_sin_cache, n_groups, heads_per_group,
                     "dsv4_o_proj_partial")
    C = n_groups * o_lora_rank
    hidden = _check_o_proj_weights(wo_a, wo_a_scale, wo_b, wo_b_scale, C, heads_per_group * hd)
    need = dsv4_o_proj_workspace_bytes(T, n_groups, heads_per_group, hd, o_lora_rank)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=o.device)
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=o.device)
    _cuda(out, "out", torch.float32)
    rc = lib.dsv4_o_proj_partial(o.data_ptr(), positions.data_ptr(), cos_sin_cache.data_ptr(),
                                 cos_sin_cache.shape[0], T, n_groups, heads_per_group, nope_dim,
                                 rope_dim, quant_group_size, o_lora_rank, hidden,
                                 wo_a.data_ptr(), wo_a_scale.data_ptr(), wo_b.data_ptr(),
                                 wo_b_scale.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                                 workspace.numel(), _stream(stream))
    _check(rc, "dsv4_o_proj_partial")
    return out


MAX_PARTIALS = 16   # DSV4_MAX_PARTIALS


def dsv4_sum_partials(partials, *, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16(sum of the fp32 partial outputs, in list order) with their shape."""
    lib = load_library()
    parts = list(partials)
    if not parts:
        raise ValueError("no partials")
    for t in parts:
        _cuda(t, "partial", torch.float32)
        if not t.is_contiguous() or t.shape != parts[0].shape:
            raise ValueError("partials must be contiguous and of one shape")
    if out is None:
        out = torch.empty(parts[0].shape, dtype=torch.bfloat16, device=parts[0].device)
    _cuda(out, "out", torch.bfloat16)
    ptrs = (ctypes.c_void_p * len(parts))(*[t.data_ptr() for t in parts])
    rc = lib.dsv4_sum_partials(ptrs, len(parts), parts[0].numel(), out.data_ptr(),
                               _stream(stream))
    _check(rc, "dsv4_sum_partials")
    return out


ROPE_QUANT_NUM_HEADS = 128         # DSV4_ROPE_QUANT_NUM_HEADS
ROPE_QUANT_HEADS_PER_GROUP = 8     # DSV4_ROPE_QUANT_HEADS_PER_GROUP


def rope_quant_unsupported_reason(n_local_heads: int, kv_cache_fp8: bool,
                                  wo_a_fp8: bool) -> str | None:
    """None if a layer may take a pre-quantised attention output, else why not."""
    why = ctypes.c_char_p()
    rc = load_library().dsv4_rope_quant_unsupported_reason(
        int(n_local_heads), 1 if kv_cache_fp8 else 0, 1 if wo_a_fp8 else 0, ctypes.byref(why))
    if rc == DSV4_OK:
        return None
    return why.value.decode()


def dsv4_o_proj_prequant_workspace_bytes(num_tokens: int, n_groups: int, o_lora_rank: int) -> int:
    return int(load_library().dsv4_o_proj_prequant_workspace_bytes(num_tokens, n_groups,
                                                                   o_lora_rank))


def dsv4_o_proj_prequant(x_fp8: torch.Tensor, x_scale: torch.Tensor, wo_a: torch.Tensor,
                         wo_a_scale: torch.Tensor, wo_b: torch.Tensor, wo_b_scale: torch.Tensor,
                         *, n_groups: int, o_lora_rank: int, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The O-projection from a pre-quantised attention output: x_fp8 the
    [T, n_slots, D] view of a physical [n_slots, T, D] buffer, x_scale the
    [T, n_slots, PK] view of a physical [n_slots, PK, T_al] one (the RopeQuant
    layout of rope_quant_attn_out); the first n_groups slots are the live
    groups.  Returns bf16 out [T, hidden]."""
    lib = load_library()
    _cuda(x_fp8, "x_fp8", _FP8)
    _cuda(x_scale, "x_scale", torch.int32)
    T, n_slots, D = x_fp8.shape
    if x_fp8.stride() != (D, T * D, 1):
        raise ValueError("x_fp8 must be the [T, slots, D] view of a physical [slots, T, D] buffer")
    PK = (D // 128 + 3) // 4
    T_al = tma_aligned_tokens(T)
    if T > 0 and (tuple(x_scale.shape) != (T, n_slots, PK) or
                  x_scale.stride() != (1, PK * T_al, T_al)):
        raise ValueError("x_scale must be the [T, slots, PK] view of a physical [slots, PK, T_al] "
                         "buffer")
    C = n_groups * o_lora_rank
    hidden = _check_o_proj_weights(wo_a, wo_a_scale, wo_b, wo_b_scale, C, D)
    need = dsv4_o_proj_prequant_workspace_bytes(T, n_groups, o_lora_rank)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x_fp8.device)
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.bfloat16, device=x_fp8.device)
    rc = lib.dsv4_o_proj_prequant(x_fp8.data_ptr(), x_scale.data_ptr(), T, n_slots, n_groups, D,
                                  o_lora_rank, hidden, wo_a.data_ptr(), wo_a_scale.data_ptr(),
                                  wo_b.data_ptr(), wo_b_scale.data_ptr(), out.data_ptr(),
                                  workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(rc, "dsv4_o_proj_prequant")
    return out


def prequant_workspace_views(workspace: torch.Tensor, num_tokens: int, n_groups: int,
                             o_lora_rank: int) -> dict:
    """zq uint8 [T, G*R] and zs int32 [PKC, T_al] inside dsv4_o_proj_prequant's workspace."""
    T, C = num_tokens, n_groups * o_lora_rank
    PKC = (C // 128 + 3) // 4
    T_al = tma_aligned_tokens(T)
    ws = workspace.view(torch.uint8)
    zq = ws[:T * C].view(T, C)
    off = _round256(T * C)
    zs = ws[off:off + PKC * T_al * 4].view(torch.int32).view(PKC, T_al)
    return {"zq": zq, "zs": zs}


def static_scratch_bytes() -> int:
    """Size of the library's own scratch for dsv4_o_proj_static (read from the library)."""
    return int(load_library().dsv4_static_scratch_bytes())


def dsv4_o_proj_static(o: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                       wo_a: torch.Tensor, wo_a_scale: torch.Tensor, wo_b: torch.Tensor,
                       wo_b_scale: torch.Tensor, *, n_groups: int, heads_per_group: int,
                       o_lora_rank: int, out: torch.Tensor, nope_dim: int = 448,
                       rope_dim: int = 64, quant_group_size: int = 128,
                       stream=None) -> torch.Tensor:
    """dsv4_o_proj for callers that cannot allocate device memory: the library
    uses its own fixed scratch (STATIC_SCRATCH_BYTES) and this wrapper
    allocates nothing either, so `out` must be given.  Calls that overlap on
    the GPU share that scratch and race."""
    lib = load_library()
    T, H, hd = o.shape
    rc = lib.dsv4_o_proj_static(o.data_ptr(), positions.data_ptr(), cos_sin_cache.data_ptr(),
                                cos_sin_cache.shape[0], T, n_groups, heads_per_group, nope_dim,
                                rope_dim, quant_group_size, o_lora_rank, wo_b.shape[0],
                                wo_a.data_ptr(), wo_a_scale.data_ptr(), wo_b.data_ptr(),
                                wo_b_scale.data_ptr(), out.data_ptr(), _stream(stream))
    _check(rc, "dsv4_o_proj_static")
    return out


def dsv4_device_status(clear: bool = True, stream=None) -> int:
    """Device status word (0 = OK, else a negative dsv4_status); synchronises the stream."""
    return int(load_library().dsv4_device_status(_stream(stream), 1 if clear else 0))


def dsv4_selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    """Runs the bounded-wait self-test kernel (see include/dsv4.h)."""
    _check(load_library().dsv4_selftest_wait_timeout(limit_us, _stream(stream)),
           "dsv4_selftest_wait_timeout")


def dsv4_status_string(status: int) -> str:
    return load_library().dsv4_status_string(status).decode()


def dsv4_last_launch_count() -> int:
    return int(load_library().dsv4_last_launch_count())
