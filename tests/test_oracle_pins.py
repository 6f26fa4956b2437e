"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each checks it against a value
the pages print, a closed form, an invariant that determines the result, a
library routine the oracle does not call, or brute force on small inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import dsv4_inputs as di

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


@pytest.fixture(scope="module")
def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def f32_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny)))


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_and_page_max(oracle_mod, facts):
    tab = oracle_mod.e4m3_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(tab) & np.isnan(ref)
    assert np.all(both_nan | (tab == ref))
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])
    assert np.nanmax(tab) == facts["fp8_max"]["value"] == tab[0x7E]
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6 and tab[0x38] == 1.0


def _nearest_e4m3_bruteforce(q):
    """Nearest finite E4M3 value, ties to the even code, clamp to +-448, sign kept."""
    tab = torch.arange(128, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = np.arange(127)            # 0x00..0x7E, all finite non-negative
    vals = tab[:127]
    a = np.minimum(np.abs(q), 448.0)
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among the (at most two) nearest, prefer the even code
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    out = codes[pick].astype(np.uint8)
    return np.where(np.signbit(q), out | 0x80, out).astype(np.uint8)


def test_e4m3_encode_bruteforce_dense_and_ties(oracle_mod):
    rng = np.random.default_rng(0)
    tab = oracle_mod.e4m3_decode_table()[:127]
    mids = (tab[:-1] + tab[1:]) / 2.0
    dense = rng.uniform(-500, 500, 200000)
    small = rng.uniform(-0.05, 0.05, 100000)
    edges = np.concatenate([tab, -tab, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                            [0.0, -0.0, 448.0, 463.99, 464.0, 500.0, -1e30, 1e-30, -1e-30]])
    q = np.concatenate([dense, small, edges])
    got = oracle_mod.e4m3_encode(q)
    want = _nearest_e4m3_bruteforce(q)
    assert np.array_equal(got, want)


def test_e4m3_encode_matches_torch_cast_in_range(oracle_mod):
    rng = np.random.default_rng(1)
    q = np.concatenate([rng.standard_normal(100000) * 50, rng.standard_normal(10000) * 0.01])
    q = np.clip(q, -448, 448).astype(np.float32)
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode(q.astype(np.float64))
    # torch casts -0-rounding negatives to 0x80 as well; compare all codes
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch_on_floats_and_exact_ties(oracle_mod):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        rng.standard_normal(1000).astype(np.float32) * 1e-38])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy()
    got = oracle_mod.bf16_from_double(x.astype(np.float64))
    assert np.array_equal(got, ref)
    # a double just above a bf16 tie must round up even though the float cast
    # of it is the tie itself (no double rounding)
    tie = 1.0 + 2.0 ** -8          # halfway between 1 and 1 + 2^-7
    above = tie + 2.0 ** -40
    assert oracle_mod.bf16_from_double([tie])[0] == 0x3F80            # ties to even -> 1.0
    assert oracle_mod.bf16_from_double([above])[0] == 0x3F81          # just above -> up
    assert oracle_mod.bf16_from_double([-above])[0] == 0xBF81


# ---------------------------------------------------------------------------
# UE8M0 exponent: the scale rule
# ---------------------------------------------------------------------------

def _scale_samples():
    rng = np.random.default_rng(3)
    out = [np.array([0.0, 1e-4, 1e-6, 448.0, 896.0, 447.99, 1.0, 3.0e38], dtype=np.float32)]
    # every binade 2^-14 .. 2^40: the full mantissa neighbourhood of 1.75 (the
    # place where the rule switches) and a random sample elsewhere
    for E in range(-14, 41):
        base = np.uint32((E + 127) << 23)
        m = np.arange(0x600000 - 2048, 0x600000 + 2048, dtype=np.uint32)
        out.append((base | m).view(np.float32))
        r = rng.integers(0, 1 << 23, 4096, dtype=np.uint32)
        out.append((base | r).view(np.float32))
        out.append(np.array([base, base | 0x7FFFFF], dtype=np.uint32).view(np.float32))
    return np.concatenate(out)


def test_ue8m0_exponent_is_smallest_feasible(oracle_mod):
    a = _scale_samples()
    e = oracle_mod.ue8m0_exponent(a).astype(np.int64)
    af = np.maximum(a.astype(np.float64), float(np.float32(1e-4)))
    assert np.all(af <= 448.0 * np.exp2(e.astype(np.float64)))          # feasible
    assert np.all(af > 448.0 * np.exp2(e.astype(np.float64) - 1))       # minimal
    assert np.all((e + 127 >= 1) & (e + 127 <= 254))


def test_ue8m0_exponent_equals_ceil_log2_of_fp32_quotient(oracle_mod):
    """The usual 'ceil to UE8M0' formula 2^ceil(log2(fl32(amax/448))) gives the same
    exponent everywhere on the sample (independent formula via numpy frexp)."""
    a = _scale_samples()
    a = a[a >= np.float32(1e-4)]
    q = (a / np.float32(448.0)).astype(np.float32)
    m, ex = np.frexp(q.astype(np.float64))          # q = m 2^ex, m in [0.5, 1)
    ceil_log2 = np.where(m == 0.5, ex - 1, ex)
    assert np.array_equal(oracle_mod.ue8m0_exponent(a), ceil_log2.astype(np.int32))


def test_zero_block_scale_byte(oracle_mod):
    e = oracle_mod.ue8m0_exponent([0.0, -0.0, 1e-30])
    assert list(e + 127) == [105, 105, 105]


# ---------------------------------------------------------------------------
# inverse RoPE
# ---------------------------------------------------------------------------

def test_cache_is_unit_circle_and_position0_is_identity():
    cache = di.cos_sin_cache(4096).numpy().astype(np.float64)
    c, s = cache[:, :32], cache[:, 32:]
    assert np.max(np.abs(c * c + s * s - 1.0)) < 1e-6
    assert np.all(cache[0, :32] == 1.0) and np.all(cache[0, 32:] == 0.0)


def test_inverse_pair_matches_complex_closed_form(oracle_mod):
    rng = np.random.default_rng(4)
    n = 200000
    a = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 4).to(torch.bfloat16).float().numpy()
    b = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 4).to(torch.bfloat16).float().numpy()
    th = rng.uniform(-100, 100, n)
    c = np.cos(th).astype(np.float32)
    s = np.sin(th).astype(np.float32)
    y0, y1 = oracle_mod.inv_rope_pairs(a, b, c, s)
    z = (a.astype(np.float64) + 1j * b.astype(np.float64)) * np.conj(c.astype(np.float64) + 1j * s.astype(np.float64))
    # error bound of the stated fp32 order: half an ulp of the rounded cross
    # product plus half an ulp of the result (tested with a 2x margin)
    bs = np.abs(b.astype(np.float64) * s)
    as_ = np.abs(a.astype(np.float64) * s)
    assert np.all(np.abs(y0 - z.real) <= f32_ulp(bs) + f32_ulp(z.real))
    assert np.all(np.abs(y1 - z.imag) <= f32_ulp(as_) + f32_ulp(z.imag))
    # the sign convention is the inverse: rotating a pure real by +theta then
    # inverse-rotating returns it, and the inverse of (c, s) applied to (c, s)
    # itself gives (1, 0) to rounding
    u0, u1 = oracle_mod.inv_rope_pairs(c, s, c, s)
    assert np.max(np.abs(u0 - 1.0)) < 1e-6 and np.max(np.abs(u1)) < 1e-6


def test_rotate_then_inverse_round_trip(oracle_mod):
    rng = np.random.default_rng(5)
    n = 200000
    a = rng.standard_normal(n).astype(np.float32) * 3
    b = rng.standard_normal(n).astype(np.float32) * 3
    cache = di.cos_sin_cache(65536).numpy()
    p = rng.integers(0, 65536, n)
    i = rng.integers(0, 32, n)
    c, s = cache[p, i], cache[p, 32 + i]
    f0, f1 = oracle_mod.fwd_rope_pairs(a, b, c, s)
    r0, r1 = oracle_mod.inv_rope_pairs(f0, f1, c, s)
    tol = 1e-6 * np.maximum(1.0, np.maximum(np.abs(a), np.abs(b)))
    assert np.all(np.abs(r0 - a) <= tol) and np.all(np.abs(r1 - b) <= tol)
    # pair norm preserved
    n0 = np.hypot(a.astype(np.float64), b.astype(np.float64))
    n1 = np.hypot(f0.astype(np.float64), f1.astype(np.float64))
    assert np.all(np.abs(n1 - n0) <= 4 * f32_ulp(n0) + 1e-6 * n0)


# ---------------------------------------------------------------------------
# O-1 end to end
# ---------------------------------------------------------------------------

def _quant_case(w, positions=None):
    d = di.make_inputs(w, with_wo_b=False)
    if positions is not None:
        d["positions"] = positions
    return d


def _unpack(sc, T):
    """[G, PK, T_al] int32 -> bytes [T, G, NB_total] by the little-endian reading."""
    b = sc.view(np.uint8).reshape(sc.shape[0], sc.shape[1], sc.shape[2], 4)
    b = b[:, :, :T, :].transpose(2, 0, 1, 3).reshape(T, sc.shape[0], sc.shape[1] * 4)
    return b


def test_shape_asserts_each_fail(oracle_mod):
    ok = dict(num_heads=4, head_dim=512, n_groups=2, heads_per_group=2, nope_dim=448,
              rope_dim=64, quant_group_size=128, cache_last_dim=64)
    assert oracle_mod.check_quant_shapes(**ok) == 0
    bad = [dict(num_heads=5), dict(head_dim=500), dict(head_dim=448 + 64, quant_group_size=96,
           nope_dim=448), dict(nope_dim=440, head_dim=504), dict(rope_dim=63, head_dim=511),
           dict(cache_last_dim=32)]
    for b in bad:
        assert oracle_mod.check_quant_shapes(**{**ok, **b}) == oracle_mod.ERR_SHAPE, b
    # a valid non-default split: nope 192 + rope 64 (192 % 128 == 128 - 64)
    assert oracle_mod.check_quant_shapes(**{**ok, "head_dim": 256, "nope_dim": 192}) == 0


def test_derived_sizes_match_rope_quant_layout(oracle_mod, facts):
    L = facts["rope_quant_layout"]
    D = L["heads_per_group"] * L["head_dim"]
    assert D == L["group_width"]
    assert L["num_heads"] // L["heads_per_group"] == L["n_groups"]
    NB = D // L["block"]
    assert (NB + 3) // 4 == L["scale_packs_per_group"] == L["heads_per_group"]
    for T in (1, 3, 4, 5, 16, 127, 129, 4096):
        Tal = oracle_mod.tma_aligned_tokens(T)
        assert Tal >= T and (Tal * 4) % 16 == 0 and Tal - T < 4


def test_out_of_range_position_is_an_error(oracle_mod):
    w = di.WORKLOADS["tiny"]
    d = _quant_case(w)
    pos = d["positions"].clone()
    pos[3] = w.max_pos
    with pytest.raises(oracle_mod.OracleError) as ei:
        oracle_mod.inv_rope_fp8_quant(d["o"], pos, d["cache"], 2, 2)
    assert ei.value.rc == oracle_mod.ERR_RANGE


def _bruteforce_quant(o_bf16, positions, cache, G, hpg, nope=448, rope=64):
    """Independent scalar path: fp64 closed-form rotation, exponent by search,
    codes by nearest-value search.  Returns (y64 [T,G,D], e [T,G,NB])."""
    x = o_bf16.float().numpy().astype(np.float64)
    T, H, hd = x.shape
    cache = cache.numpy().astype(np.float64)
    y = x.copy()
    half = rope // 2
    cs = cache[positions.numpy()]
    c = cs[:, None, :half]
    s = cs[:, None, half:]
    z = (x[:, :, nope::2] + 1j * x[:, :, nope + 1::2]) * (c - 1j * s)
    y[:, :, nope::2] = z.real
    y[:, :, nope + 1::2] = z.imag
    y = y.reshape(T, G, hpg * hd)
    return y


def test_tiny_bruteforce_o1(oracle_mod):
    """Every block of the tiny workload: codes decode back to within half an
    E4M3 step (plus fp32 rotation slack) of the fp64 closed form, and the
    exponent is the smallest one that fits the block's amax."""
    w = di.WORKLOADS["tiny"]
    d = _quant_case(w)
    q, sc = oracle_mod.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], w.n_groups,
                                          w.heads_per_group)
    T, G, D = w.T, w.n_groups, w.D
    y = _bruteforce_quant(d["o"], d["positions"], d["cache"], G, w.heads_per_group)
    codes = q.transpose(1, 0, 2)                        # [T, G, D]
    e = _unpack(sc, T).astype(np.int64) - 127           # [T, G, NB]
    tab = oracle_mod.e4m3_decode_table()
    dec = tab[codes] * np.exp2(np.repeat(e, 128, axis=2))
    yb = y.reshape(T, G, D // 128, 128)
    amax = np.maximum(np.abs(yb).max(axis=3), float(np.float32(1e-4)))
    # exponent: smallest feasible for the fp64 amax (the fp32 amax differs by
    # at most an ulp; allow that only where it straddles a boundary)
    feas = amax <= 448.0 * np.exp2(e) * (1 + 2 ** -22)
    minimal = amax > 448.0 * np.exp2(e - 1) * (1 - 2 ** -22)
    assert feas.all() and minimal.all()
    step = np.exp2(np.repeat(e, 128, axis=2)) * np.where(
        np.abs(y) / np.exp2(np.repeat(e, 128, axis=2)) < 2 ** -6, 2.0 ** -9,
        2.0 ** (np.floor(np.log2(np.maximum(np.abs(y) / np.exp2(np.repeat(e, 128, axis=2)), 1e-300))) - 3))
    slack = 4 * f32_ulp(y)
    assert np.all(np.abs(dec - y) <= step / 2 + slack)
    # no NaN codes, every decoded magnitude within 448 * scale
    assert not np.any((codes & 0x7F) == 0x7F)


def test_position0_reduces_to_plain_block_quant(oracle_mod):
    """With every position 0 the cache row is (1.., 0..), inverse RoPE is the
    identity, and O-1 is a plain per-token 1x128 quantisation of o: compare with
    a brute-force nearest-value quantisation (torch decode table, exponent by
    the minimality invariant)."""
    w = di.WORKLOADS["tiny"]
    d = _quant_case(w, positions=torch.zeros(16, dtype=torch.int64))
    q, sc = oracle_mod.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], w.n_groups,
                                          w.heads_per_group)
    x = d["o"].float().numpy().reshape(w.T, w.n_groups, w.D // 128, 128).astype(np.float64)
    amax = np.maximum(np.abs(x).max(axis=3), float(np.float32(1e-4)))
    e = np.ceil(np.log2(amax / 448.0))
    e = np.where(amax <= 448.0 * np.exp2(e - 1), e - 1, e)
    e = np.where(amax > 448.0 * np.exp2(e), e + 1, e)
    want_codes = _nearest_e4m3_bruteforce((x / np.exp2(e)[..., None]).ravel()).reshape(x.shape)
    got_codes = q.transpose(1, 0, 2).reshape(x.shape)
    assert np.array_equal(got_codes, want_codes)
    assert np.array_equal(_unpack(sc, w.T).astype(np.int64) - 127, e.astype(np.int64))


def test_nope_blocks_do_not_depend_on_position(oracle_mod):
    w = di.WORKLOADS["tiny"]
    d = _quant_case(w)
    q1, s1 = oracle_mod.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], 2, 2)
    pos2 = (d["positions"] + 977) % w.max_pos
    q2, s2 = oracle_mod.inv_rope_fp8_quant(d["o"], pos2, d["cache"], 2, 2)
    # blocks 0..2 of every head (lanes 0..383) are pure nope lanes
    v1 = q1.reshape(2, w.T, 2, 4, 128)
    v2 = q2.reshape(2, w.T, 2, 4, 128)
    assert np.array_equal(v1[:, :, :, :3], v2[:, :, :, :3])
    b1, b2 = _unpack(s1, w.T).reshape(w.T, 2, 2, 4), _unpack(s2, w.T).reshape(w.T, 2, 2, 4)
    assert np.array_equal(b1[..., :3], b2[..., :3])
    assert not np.array_equal(v1[:, :, :, 3], v2[:, :, :, 3])   # block 3 holds rope lanes


def test_zero_blocks_and_student_t_invariants(oracle_mod):
    w = di.WORKLOADS["quant1k"].with_tokens(64)
    d = _quant_case(w)
    q, sc = oracle_mod.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], w.n_groups,
                                          w.heads_per_group)
    x = d["o"].view(w.T, w.n_groups, w.D // 128, 128)
    zero = (x == 0).all(dim=3).numpy()
    assert zero.sum() >= 1
    codes = q.transpose(1, 0, 2).reshape(w.T, w.n_groups, w.D // 128, 128)
    bytes_ = _unpack(sc, w.T)
    assert np.all(bytes_[zero] == 105)
    assert np.all((codes[zero] & 0x7F) == 0)
    assert np.all((bytes_ >= 1) & (bytes_ <= 254))
    assert not np.any((codes & 0x7F) == 0x7F)


def test_strided_views_round_trip(oracle_mod):
    """The physical [G][T][D] / [G][PK][T_al] buffers seen through the page's
    views have strides (D, T*D, 1) and (1, PK*T_al, T_al)."""
    w = di.WORKLOADS["tiny"].with_tokens(5)
    d = _quant_case(w)
    q, sc = oracle_mod.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], 2, 2)
    qt = torch.from_numpy(q).transpose(0, 1)
    assert qt.shape == (5, 2, w.D) and qt.stride() == (w.D, 5 * w.D, 1)
    st = torch.from_numpy(sc).permute(2, 0, 1)[:5]
    PK, Tal = sc.shape[1], sc.shape[2]
    assert Tal == 8 and st.shape == (5, 2, PK) and st.stride() == (1, PK * Tal, Tal)
    assert torch.equal(qt[3, 1], torch.from_numpy(q[1, 3]))


# ---------------------------------------------------------------------------
# O-2 / O-3 GEMMs
# ---------------------------------------------------------------------------

def _scale_bytes_tgk(xs, T, G, D):
    """packed int32 [G, PK, T_al] -> int64 exponent bytes [T, G, D/128] (little-endian reading)."""
    NB = D // 128
    PK, Tal = xs.shape[1], xs.shape[2]
    b = xs.contiguous().view(torch.uint8).view(G, PK, Tal, 4)[:, :, :T]
    return b.permute(2, 0, 1, 3).reshape(T, G, PK * 4)[:, :, :NB].to(torch.int64)


def _dequant_torch(codes_u8, exps):
    return codes_u8.view(torch.float8_e4m3fn).to(torch.float64) * torch.exp2(exps.to(torch.float64))


@pytest.mark.parametrize("D", [512, 1152])
def test_grouped_gemm_matches_einsum_in_float64(oracle_mod, D):
    """The pages restate the grouped product as einsum 'tgd,grd->tgr' (sglang
    bf16 fallback) and as bmm over wo_a viewed [G, R, D] (vLLM): compare with
    torch.einsum in float64 on the dequantised operands (torch's own FP8 decode).
    D = 1152: nine scale blocks in three packed words, the last one partial."""
    T, G, R = 9, 3, 256
    Tal = oracle_mod.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=11, tma_aligned_T=Tal)
    w, ws = di.fp8_block_weight(G * R, D, seed=12)
    z, z64 = oracle_mod.grouped_gemm(x, xs, w, ws, T, G, D, R, want_fp64=True)
    ex = (_scale_bytes_tgk(xs, T, G, D) - 127).repeat_interleave(128, dim=2)
    xd = _dequant_torch(x.permute(1, 0, 2), ex)                               # [T, G, D]
    ew = (ws.to(torch.int64) - 127).repeat_interleave(128, 0).repeat_interleave(128, 1)
    wd = _dequant_torch(w, ew).view(G, R, D)
    ref = torch.einsum("tgd,grd->tgr", xd, wd).numpy()
    assert np.allclose(z64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    zb = torch.from_numpy(z.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(zb, torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()) or \
        np.max(np.abs(zb - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2 ** -8


def test_grouped_gemm_group_locality(oracle_mod):
    T, G, D, R = 4, 3, 256, 128
    Tal = oracle_mod.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=13, tma_aligned_T=Tal)
    w, ws = di.fp8_block_weight(G * R, D, seed=14)
    z = oracle_mod.grouped_gemm(x, xs, w, ws, T, G, D, R)
    w2 = w.clone()
    w2[R:] = torch.flip(w2[R:], dims=[1])     # change every row outside group 0
    z2 = oracle_mod.grouped_gemm(x, xs, w2, ws, T, G, D, R)
    assert np.array_equal(z[:, 0], z2[:, 0])
    assert not np.array_equal(z[:, 1:], z2[:, 1:])


def test_grouped_gemm_identity_weight(oracle_mod):
    """W[g*R + n, k] = 1 if k == n else 0 with unit scales: z = bf16(dq_x)."""
    T, G, D, R = 7, 2, 256, 128
    Tal = oracle_mod.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=15, tma_aligned_T=Tal)
    w = torch.zeros(G * R, D, dtype=torch.uint8)
    for g in range(G):
        w[g * R:(g + 1) * R, :R] = torch.eye(R, dtype=torch.uint8) * 0x38
    ws = torch.full((G * R // 128, D // 128), 127, dtype=torch.uint8)
    z = oracle_mod.grouped_gemm(x, xs, w, ws, T, G, D, R)
    ex = (_scale_bytes_tgk(xs, T, G, D) - 127).repeat_interleave(128, dim=2)
    xd = _dequant_torch(x.permute(1, 0, 2), ex)[:, :, :R]
    want = xd.to(torch.bfloat16).view(torch.uint16).numpy()   # exact: dq_x has 4 significant bits
    assert np.array_equal(z, want)


def test_block_quant_rows_bruteforce(oracle_mod):
    rng = np.random.default_rng(6)
    T, C = 5, 640
    x = torch.from_numpy(rng.standard_normal((T, C)).astype(np.float32) * 3).to(torch.bfloat16)
    x[2, 128:256] = 0
    q, sc = oracle_mod.block_quant_rows(x)
    xf = x.float().numpy().astype(np.float64).reshape(T, C // 128, 128)
    amax = np.maximum(np.abs(xf).max(axis=2), float(np.float32(1e-4)))
    e = np.ceil(np.log2(amax / 448.0))
    e = np.where(amax <= 448.0 * np.exp2(e - 1), e - 1, e)
    e = np.where(amax > 448.0 * np.exp2(e), e + 1, e)
    want = _nearest_e4m3_bruteforce((xf / np.exp2(e)[..., None]).ravel()).reshape(T, C)
    assert np.array_equal(q, want)
    b = sc.view(np.uint8).reshape(sc.shape[0], sc.shape[1], 4)[:, :T].transpose(1, 0, 2).reshape(T, -1)
    assert np.array_equal(b[:, :C // 128].astype(np.int64) - 127, e.astype(np.int64))
    assert np.all(b[:, C // 128:] == 0)        # unused high bytes of the last int32 are zero
    assert b[2, 1] == 105


def test_o_proj_chain_on_tiny(oracle_mod):
    """The whole chain on the tiny workload: out equals the float64 product of the
    dequantised re-quantised z with the dequantised wo_b (torch matmul)."""
    w = di.WORKLOADS["tiny"]
    d = di.make_inputs(w)
    out, out64, z = oracle_mod.o_proj(d["o"], d["positions"], d["cache"], d["wo_a"],
                                      d["wo_a_scale"], d["wo_b"], d["wo_b_scale"],
                                      n_groups=w.n_groups, heads_per_group=w.heads_per_group,
                                      o_lora_rank=w.o_lora_rank, hidden=w.hidden, want_z=True)
    zq, zs = oracle_mod.block_quant_rows(z.reshape(w.T, -1))
    C = w.n_groups * w.o_lora_rank
    zb = _scale_bytes_tgk(torch.from_numpy(zs)[None], w.T, 1, C)[:, 0]
    ez = (zb - 127).repeat_interleave(128, dim=1)
    zd = _dequant_torch(torch.from_numpy(zq), ez)
    ew = (d["wo_b_scale"].to(torch.int64) - 127).repeat_interleave(128, 0).repeat_interleave(128, 1)
    wd = _dequant_torch(d["wo_b"], ew)
    ref = (zd @ wd.T).numpy()
    assert np.allclose(out64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())



# ---------------------------------------------------------------------------
# bf16 variants (quantize=False, and the bmm fallback for a non-FP8 wo_a)
# ---------------------------------------------------------------------------

def test_inv_rope_bf16_closed_form_and_identity(oracle_mod):
    w = di.WORKLOADS["tiny"]
    d = di.make_inputs(w, with_wo_b=False)
    xb = oracle_mod.inv_rope_bf16(d["o"], d["positions"], d["cache"], w.n_groups,
                                  w.heads_per_group)
    got = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).double().numpy()
    y = _bruteforce_quant(d["o"], d["positions"], d["cache"], w.n_groups, w.heads_per_group)
    y = y.reshape(w.T, w.n_groups, w.D).transpose(1, 0, 2)          # physical [G, T, D]
    # nope lanes exact; rotated lanes within half a bf16 step (+ fp32 slack) of fp64
    lanes = np.arange(w.D) % 512
    nope = lanes < 448
    assert np.array_equal(got[:, :, nope], y[:, :, nope])
    r = got[:, :, ~nope] - y[:, :, ~nope]
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(y[:, :, ~nope]), 1e-30))) - 7)
    assert np.all(np.abs(r) <= step / 2 + 4 * f32_ulp(y[:, :, ~nope]))
    # position 0: bit-identical to o, group-major
    p0 = torch.zeros(w.T, dtype=torch.int64)
    x0 = oracle_mod.inv_rope_bf16(d["o"], p0, d["cache"], w.n_groups, w.heads_per_group)
    ref = d["o"].view(torch.uint16).reshape(w.T, w.n_groups, w.D).permute(1, 0, 2).numpy()
    assert np.array_equal(x0, ref)


def test_grouped_gemm_bf16_matches_bmm_in_float64(oracle_mod):
    """The page's own restatement: torch.bmm of x [G, T, D] with W viewed [G, R, D]
    transposed, here in float64."""
    T, G, D, R = 7, 3, 192, 64
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((G, T, D)).astype(np.float32)).to(torch.bfloat16)
    wt = torch.from_numpy(rng.standard_normal((G * R, D)).astype(np.float32) * 0.02).to(torch.bfloat16)
    z, z64 = oracle_mod.grouped_gemm_bf16(x, wt, T, G, D, R, want_fp64=True)
    ref = torch.bmm(x.double(), wt.double().view(G, R, D).transpose(1, 2)).transpose(0, 1).numpy()
    assert np.allclose(z64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    zb = torch.from_numpy(z.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(zb, torch.from_numpy(ref).to(torch.bfloat16).double().numpy()) or \
        np.max(np.abs(zb - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2 ** -8
