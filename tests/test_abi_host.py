"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
function include/dsv4.h declares, and its host-side validation rejects bad
arguments before touching CUDA.  No compute call is made here."""
import ctypes
import subprocess

import pytest

import deepseek_v4_attention_gb300 as k
from deepseek_v4_attention_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return k.load_library()


def test_exports_every_header_function(lib):
    names = k.header_functions()
    assert set(names) == {"dsv4_inv_rope_fp8_quant", "dsv4_grouped_wo_a",
                          "dsv4_o_proj_workspace_bytes", "dsv4_o_proj", "dsv4_o_proj_with_events",
                          "dsv4_o_proj_static", "dsv4_selftest_wait_timeout",
                          "dsv4_inv_rope_bf16", "dsv4_grouped_wo_a_bf16",
                          "dsv4_inv_rope_grouped_wo_a", "dsv4_static_scratch_bytes",
                          "dsv4_grouped_wo_a_ex",
                          "dsv4_o_proj_partial", "dsv4_sum_partials",
                          "dsv4_rope_quant_unsupported_reason",
                          "dsv4_o_proj_prequant_workspace_bytes", "dsv4_o_proj_prequant",
                          "dsv4_status_string",
                          "dsv4_device_status", "dsv4_last_launch_count"}
    out = subprocess.run(["nm", "-D", "--defined-only", k.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code, name in k.STATUS.items():
        assert k.dsv4_status_string(code).startswith(name)
    assert "unknown" in k.dsv4_status_string(12345)


def test_quant_host_validation_without_gpu(lib):
    f = lib.dsv4_inv_rope_fp8_quant
    P = 4096  # any non-null, 16-byte aligned fake address: rejected before use
    good = [P, P, P, 4, 16, 2, 2, 448, 64, 128, P, P, None]
    for idx, val, rc in [(3, -1, -1), (4, 0, -1), (5, 0, -1), (6, 0, -1), (8, 63, -1),
                         (9, 100, -1), (9, 32, -1), (7, 192, -4), (9, 0, -1)]:
        a = list(good); a[idx] = val
        assert f(*a) == rc, (idx, val)
    # T == 0 is valid and launches nothing, even with null pointers
    a = list(good); a[3] = 0; a[0] = None
    assert f(*a) == 0 and k.dsv4_last_launch_count() == 0
    for idx in (0, 1, 2, 10, 11):
        a = list(good); a[idx] = None
        assert f(*a) == -2
    for idx in (0, 1, 2, 10, 11):
        a = list(good); a[idx] = P + 4
        assert f(*a) == -3


def test_gemm_host_validation_without_gpu(lib):
    f = lib.dsv4_grouped_wo_a
    P = 4096
    good = [P, P, 16, 2, 1024, 128, P, P, P, None]
    for idx, val in [(2, -1), (3, 0), (4, 1000), (5, 100), (4, 0), (5, 0)]:
        a = list(good); a[idx] = val
        assert f(*a) == -1, (idx, val)
    a = list(good); a[2] = 0
    assert f(*a) == 0
    for idx in (0, 1, 6, 7, 8):
        a = list(good); a[idx] = None
        assert f(*a) == -2
    for idx in (0, 1, 6, 8):
        a = list(good); a[idx] = P + 8
        assert f(*a) == -3


def test_fused_wo_a_host_validation_without_gpu(lib):
    """dsv4_inv_rope_grouped_wo_a: the quantiser's asserts, R, the decode-size
    limit (DSV4_FUSED_MAX_TOKENS = 64) and max_pos < 2^31, then pointers."""
    f = lib.dsv4_inv_rope_grouped_wo_a
    P = 4096
    good = [P, P, P, 16, 4096, 2, 2, 448, 64, 128, 128, P, P, P, None]
    for idx, val, rc in [(3, -1, -1), (4, 0, -1), (5, 0, -1), (6, 0, -1), (10, 100, -1),
                         (10, 0, -1), (7, 192, -4), (3, 65, -4), (4, 1 << 31, -4)]:
        a = list(good); a[idx] = val
        assert f(*a) == rc, (idx, val)
    assert k.FUSED_MAX_TOKENS == 64
    a = list(good); a[3] = 0; a[0] = None
    assert f(*a) == 0 and k.dsv4_last_launch_count() == 0
    for idx in (0, 1, 2, 11, 12, 13):
        a = list(good); a[idx] = None
        assert f(*a) == -2, idx
    for idx in (0, 1, 2, 11, 13):
        a = list(good); a[idx] = P + 8
        assert f(*a) == -3, idx


def test_o_proj_workspace_bytes(lib):
    T, G, hpg, R = 4096, 16, 8, 1024
    need = k.dsv4_o_proj_workspace_bytes(T, G, hpg, 512, R)
    D = hpg * 512
    expect = G * T * D + G * (D // 512) * T * 4 + T * G * R + (G * R // 512) * T * 4
    assert need == expect                  # every part is already a multiple of 256 here
    assert k.dsv4_o_proj_workspace_bytes(5, 2, 2, 512, 128) % 256 == 0
    assert k.dsv4_o_proj_workspace_bytes(-1, 2, 2, 512, 128) == 0
    assert k.dsv4_o_proj_workspace_bytes(4, 2, 2, 500, 128) == 0


def test_o_proj_host_validation_without_gpu(lib):
    f = lib.dsv4_o_proj
    P = 4096
    need = k.dsv4_o_proj_workspace_bytes(16, 2, 2, 512, 128)
    good = [P, P, P, 4096, 16, 2, 2, 448, 64, 128, 128, 256, P, P, P, P, P, 1 << 20, need, None]
    for idx, val, rc in [(4, -1, -1), (10, 100, -1), (11, 100, -1), (11, 0, -1), (3, 0, -1),
                         (9, 64, -4), (7, 192, -4), (9, 32, -1)]:
        a = list(good); a[idx] = val
        assert f(*a) == rc, (idx, val)
    a = list(good); a[18] = need - 1
    assert f(*a) == -5
    a = list(good); a[17] = None
    assert f(*a) == -5
    a = list(good); a[17] = (1 << 20) + 16
    assert f(*a) == -3
    for idx in (0, 1, 2, 12, 13, 14, 15, 16):
        a = list(good); a[idx] = None
        assert f(*a) == -2, idx


def test_o_proj_static_host_validation_without_gpu(lib):
    f = lib.dsv4_o_proj_static
    P = 4096
    good = [P, P, P, 65536, 64, 16, 8, 448, 64, 128, 1024, 7168, P, P, P, P, P, None]
    a = list(good); a[4] = -1
    assert f(*a) == -1
    a = list(good); a[4] = 0
    assert f(*a) == 0 and k.dsv4_last_launch_count() == 0
    a = list(good); a[4] = 813          # beyond the fixed scratch: rejected before any CUDA call
    assert f(*a) == -5
    a = list(good); a[16] = None
    assert f(*a) == -2


def test_selftest_limit_validation_without_gpu(lib):
    assert lib.dsv4_selftest_wait_timeout(0, None) == -1
    assert lib.dsv4_selftest_wait_timeout(2_000_000, None) == -1


def test_bf16_entries_host_validation_without_gpu(lib):
    P = 4096
    f = lib.dsv4_inv_rope_bf16
    good = [P, P, P, 4, 16, 2, 2, 448, 64, P, None]
    a = list(good); a[3] = -1
    assert f(*a) == -1
    a = list(good); a[3] = 0
    assert f(*a) == 0
    a = list(good); a[9] = None
    assert f(*a) == -2
    a = list(good); a[7] = 192
    assert f(*a) == -4
    g = lib.dsv4_grouped_wo_a_bf16
    good = [P, 16, 2, 1024, 128, P, P, None]
    for idx, val in [(3, 96), (4, 64), (1, -1)]:
        a = list(good); a[idx] = val
        assert g(*a) == -1
    a = list(good); a[5] = None
    assert g(*a) == -2
    a = list(good); a[6] = P + 2
    assert g(*a) == -3


def test_rope_quant_eligibility(lib):
    """rope_quant_unsupported_reason of the o_proj page: 128 local heads, the
    per-tensor FP8 KV cache and an FP8 wo_a, checked in that order."""
    assert k.rope_quant_unsupported_reason(128, True, True) is None
    assert "128" in k.rope_quant_unsupported_reason(64, True, True)
    assert "128" in k.rope_quant_unsupported_reason(256, False, False)
    assert "KV" in k.rope_quant_unsupported_reason(128, False, True)
    assert "wo_a" in k.rope_quant_unsupported_reason(128, True, False)
    assert lib.dsv4_rope_quant_unsupported_reason(128, 1, 1, None) == 0
    assert lib.dsv4_rope_quant_unsupported_reason(96, 1, 1, None) == -4
    assert k.ROPE_QUANT_NUM_HEADS == 128 and k.ROPE_QUANT_HEADS_PER_GROUP == 8


def test_static_scratch_size_matches_header(lib):
    import re
    with open(k.HEADER) as f:
        m = re.search(r"#define DSV4_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)",
                      f.read())
    assert m and k.static_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_prequant_and_partial_host_validation_without_gpu(lib):
    P = 4096
    T, slots, G, D, R, hidden = 8, 16, 12, 4096, 1024, 7168
    need = k.dsv4_o_proj_prequant_workspace_bytes(T, G, R)
    pkc, t_al = (G * R // 128 + 3) // 4, 8
    assert need == 256 * (-(-T * G * R // 256)) + 256 * (-(-pkc * t_al * 4 // 256))
    assert k.dsv4_o_proj_prequant_workspace_bytes(T, G, 100) == 0
    f = lib.dsv4_o_proj_prequant
    good = [P, P, T, slots, G, D, R, hidden, P, P, P, P, P, P, need, None]
    for idx, val, rc in [(2, -1, -1), (4, 0, -1), (4, 17, -1), (5, 4000, -1), (6, 1000, -1),
                         (7, 7000, -1), (14, need - 1, -5), (13, P + 16, -3)]:
        a = list(good); a[idx] = val
        assert f(*a) == rc, (idx, val)
    a = list(good); a[2] = 0; a[0] = None
    assert f(*a) == 0 and k.dsv4_last_launch_count() == 0
    for idx in (0, 1, 8, 9, 10, 11, 12):
        a = list(good); a[idx] = None
        assert f(*a) == -2, idx
    for idx in (0, 1, 8, 10, 12):
        a = list(good); a[idx] = P + 8
        assert f(*a) == -3, idx
    g = lib.dsv4_o_proj_partial
    wsz = k.dsv4_o_proj_workspace_bytes(T, 8, 8, 512, R)
    good = [P, P, P, 65536, T, 8, 8, 448, 64, 128, R, hidden, P, P, P, P, P, P, wsz, None]
    assert g(*[*good[:11], 100, *good[12:]]) == -1                 # hidden % 128
    a = list(good); a[16] = None
    assert g(*a) == -2
    a = list(good); a[18] = wsz - 1
    assert g(*a) == -5
    a = list(good); a[4] = 0
    assert g(*a) == 0 and k.dsv4_last_launch_count() == 0
