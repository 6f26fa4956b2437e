"""GPU parity of dsv4_grouped_wo_a and dsv4_o_proj against the CPU oracle
(through the C ABI).  Tolerance: gpu_helpers.GEMM_RTOL."""
import numpy as np
import pytest
import torch

import dsv4_inputs as di
import oracle
from gpu_helpers import (GEMM_RTOL, assert_codes_match, check_o_proj_parts, cuda_or_skip,
                         gemm_rel_err, to_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _gpu_wo_a(x, xs, w, ws, T, G, D, R, dev):
    import deepseek_v4_attention_gb300 as k
    xg = x.to(dev).view(torch.float8_e4m3fn)            # physical [G, T, D]
    sg = xs.to(dev)                                     # physical [G, PK, T_al]
    z = k.dsv4_grouped_wo_a(xg.transpose(0, 1), sg.permute(2, 0, 1)[:T], w.to(dev),
                            ws.to(dev), G, R)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    return to_bits(z)


# (1200, 4, 640, 1024) runs on CTA pairs (5 x 4 x 4 pair tiles); (128, 16, 256,
# 2560) on one SM with 256-wide tiles (T <= 128: no pairs; 10 x 16 tiles >= one
# per SM); the others on one SM with 128-wide tiles
@pytest.mark.parametrize("T,G,D,R", [(16, 2, 1024, 128), (64, 8, 4096, 1024), (1, 1, 128, 128),
                                     (3, 2, 512, 256), (129, 3, 640, 384), (200, 1, 1024, 896),
                                     (1200, 4, 640, 1024), (128, 16, 256, 2560)])
def test_grouped_wo_a_random_operands(dev, T, G, D, R):
    T_al = oracle.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=T * 7 + G, tma_aligned_T=T_al)
    w, ws = di.fp8_block_weight(G * R, D, seed=T + 1000 * G)
    zg = _gpu_wo_a(x, xs, w, ws, T, G, D, R, dev)
    zr, z64 = oracle.grouped_gemm(x, xs, w, ws, T, G, D, R, want_fp64=True)
    err = gemm_rel_err(zg, z64)
    assert err <= GEMM_RTOL, err


# Shapes of the CTA-pair kernel (more than 128 tokens, N % 256 == 0, at least
# one 256 x 256 tile per two SMs: ceil(T/256) * N/256 * G >= 76 on 152 SMs):
# the odd CTA's 128 rows all past T (T = 300) or holding one token (T = 129);
# one k-block (a single one-k-block stage); three k-blocks (a stage of two,
# then one); a dense GEMM whose last raster group has one 256-token block
# (T = 2304: groups of 8 and 1 m-blocks).
@pytest.mark.parametrize("T,G,D,R", [(300, 16, 512, 1024), (129, 16, 512, 2048),
                                     (1200, 4, 128, 1024), (1200, 4, 384, 1024),
                                     (2304, 1, 256, 2560)])
def test_grouped_wo_a_pair_kernel_edges(dev, T, G, D, R):
    assert -(-T // 256) * (R // 256) * G >= 76 and T > 128 and R % 256 == 0
    T_al = oracle.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=T * 3 + D, tma_aligned_T=T_al)
    w, ws = di.fp8_block_weight(G * R, D, seed=T + 7 * D)
    zg = _gpu_wo_a(x, xs, w, ws, T, G, D, R, dev)
    _, z64 = oracle.grouped_gemm(x, xs, w, ws, T, G, D, R, want_fp64=True)
    assert gemm_rel_err(zg, z64) <= GEMM_RTOL


@pytest.mark.parametrize("T,G,D,R", [(130, 2, 512, 256), (1200, 16, 512, 256)])
def test_grouped_wo_a_identity_weight_is_exact(dev, T, G, D, R):
    """W = I in every group with unit scales: z must equal bf16(dq_x) exactly."""
    T_al = oracle.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=5, tma_aligned_T=T_al)
    w = torch.zeros(G * R, D, dtype=torch.uint8)
    for g in range(G):
        w[g * R:(g + 1) * R, :R] = torch.eye(R, dtype=torch.uint8) * 0x38
    ws = torch.full((G * R // 128, D // 128), 127, dtype=torch.uint8)
    zg = _gpu_wo_a(x, xs, w, ws, T, G, D, R, dev)
    zr = oracle.grouped_gemm(x, xs, w, ws, T, G, D, R)
    assert np.array_equal(zg, zr)


@pytest.mark.parametrize("T,G,R", [(128, 1, 128), (1280, 16, 256)])
def test_grouped_wo_a_scale_rows(dev, T, G, R):
    """Scales that vary only by token row, by k-block and by 128-row weight
    block: catches a wrong scale-factor layout in tensor memory (exact products,
    exact sums)."""
    D = 1024
    T_al = T
    codes = torch.full((G, T, D), 0x38, dtype=torch.uint8)          # all ones
    b = torch.zeros((G, 8, T_al), dtype=torch.int64)
    row_e = torch.arange(T) % 7                                      # per-row exponent
    for kb in range(8):
        b[:, kb, :] = 120 + row_e + kb                              # + per-block exponent
    words = (b[:, 0::4] | (b[:, 1::4] << 8) | (b[:, 2::4] << 16) | (b[:, 3::4] << 24))
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)
    w = torch.full((G * R, D), 0x38, dtype=torch.uint8)
    ws = torch.full((G * R // 128, 8), 127, dtype=torch.uint8)
    ws[:, 3] = 125
    ws[1::2, 5] = 129                                                # odd 128-row blocks differ
    zg = _gpu_wo_a(codes, words, w, ws, T, G, D, R, dev)
    zr = oracle.grouped_gemm(codes, words, w, ws, T, G, D, R)
    assert np.array_equal(zg, zr)


def test_grouped_wo_a_decode_config_parity(dev):
    w = di.WORKLOADS["decode"]
    d = di.make_inputs(w, with_wo_b=False)
    x, xs = oracle.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], w.n_groups,
                                      w.heads_per_group)
    x, xs = torch.from_numpy(x), torch.from_numpy(xs)
    zg = _gpu_wo_a(x, xs, d["wo_a"], d["wo_a_scale"], w.T, w.n_groups, w.D, w.o_lora_rank, dev)
    _, z64 = oracle.grouped_gemm(x, xs, d["wo_a"], d["wo_a_scale"], w.T, w.n_groups, w.D,
                                 w.o_lora_rank, want_fp64=True)
    assert gemm_rel_err(zg, z64) <= GEMM_RTOL


def test_grouped_wo_a_prefill_config_sampled(dev):
    """T = 8192 prefill workload (all groups, all columns) checked on a seeded
    sample of 512 token rows (the product is row-independent)."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["prefill"]
    d = di.make_inputs(w, with_wo_b=False)
    q, s = k.dsv4_inv_rope_fp8_quant(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                                     w.n_groups, w.heads_per_group)
    z = k.dsv4_grouped_wo_a(q, s, d["wo_a"].to(dev), d["wo_a_scale"].to(dev), w.n_groups,
                            w.o_lora_rank)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    idx = np.sort(np.random.default_rng(0).choice(w.T, 512, replace=False))
    ti = torch.from_numpy(idx)
    xr, xsr = oracle.inv_rope_fp8_quant(d["o"][ti], d["positions"][ti], d["cache"], w.n_groups,
                                        w.heads_per_group)
    # the GPU's own quantised rows are what its GEMM consumed; they match the oracle's
    qg = to_bits(q.view(torch.uint8).transpose(0, 1))[:, idx]
    assert_codes_match(qg, xr)
    sg = s.permute(1, 2, 0).cpu().numpy()[:, :, idx]
    assert np.array_equal(sg, xsr[:, :, :len(idx)])
    _, z64 = oracle.grouped_gemm(np.ascontiguousarray(qg), xsr, d["wo_a"], d["wo_a_scale"],
                                 len(idx), w.n_groups, w.D, w.o_lora_rank, want_fp64=True)
    zg = to_bits(z)[idx]
    assert gemm_rel_err(zg, z64) <= GEMM_RTOL


def _o_proj_gpu(d, w, dev):
    """dsv4_o_proj with a caller workspace; returns (out, workspace) on the device."""
    import deepseek_v4_attention_gb300 as k
    need = k.dsv4_o_proj_workspace_bytes(w.T, w.n_groups, w.heads_per_group, w.head_dim,
                                         w.o_lora_rank)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = k.dsv4_o_proj(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                        d["wo_a"].to(dev), d["wo_a_scale"].to(dev), d["wo_b"].to(dev),
                        d["wo_b_scale"].to(dev), n_groups=w.n_groups,
                        heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank,
                        workspace=ws)
    assert k.dsv4_last_launch_count() == 3
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    return out, ws


@pytest.mark.parametrize("T", [16, 1, 5, 131])
def test_o_proj_tiny_parity(dev, T):
    w = di.WORKLOADS["tiny"].with_tokens(T, seed=T)
    d = di.make_inputs(w)
    out, ws = _o_proj_gpu(d, w, dev)
    check_o_proj_parts(d, w, out, ws)


def test_o_proj_decode_config_parity(dev):
    """The decode workload (T = 64, 8 groups, hidden 7168) through the whole
    chain, every row checked stage by stage."""
    w = di.WORKLOADS["decode"]
    d = di.make_inputs(w)
    out, ws = _o_proj_gpu(d, w, dev)
    check_o_proj_parts(d, w, out, ws)


def test_o_proj_full_config_sampled(dev):
    """Full workload (T=4096, 128 heads, R=1024, hidden 7168) in the launch
    configuration the benchmark times; 512 seeded token rows checked stage by
    stage: the quantised groups, zq and its scales against the oracle, wo_b
    against the fp64 product of the GPU's own zq (the path is row-independent)."""
    w = di.WORKLOADS["full"]
    d = di.make_inputs(w)
    out, ws = _o_proj_gpu(d, w, dev)
    idx = np.sort(np.random.default_rng(1).choice(w.T, 512, replace=False))
    check_o_proj_parts(d, w, out, ws, idx)
    out2, _ = _o_proj_gpu(d, w, dev)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "two runs differ"


@pytest.mark.parametrize("name,T", [("decode", 64), ("decode", 7), ("full", 300)])
def test_o_proj_deterministic(dev, name, T):
    """Two runs of the whole chain give bit-identical output: decode shapes take
    the split-K cluster path (partials added in a fixed order) with the 64-row
    A box, T = 300 the programmatically launched GEMMs."""
    w = di.WORKLOADS[name].with_tokens(T, seed=T + 11)
    d = di.make_inputs(w)
    og, _ = _o_proj_gpu(d, w, dev)
    og2, _ = _o_proj_gpu(d, w, dev)
    assert torch.equal(og.view(torch.int16), og2.view(torch.int16)), "two runs differ"


def test_o_proj_errors(dev):
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    w = di.WORKLOADS["tiny"]
    d = {n: t.to(dev) for n, t in di.make_inputs(w).items()}
    out = torch.empty(w.T, w.hidden, dtype=torch.bfloat16, device=dev)
    need = k.dsv4_o_proj_workspace_bytes(w.T, w.n_groups, w.heads_per_group, 512, w.o_lora_rank)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    args = [d["o"].data_ptr(), d["positions"].data_ptr(), d["cache"].data_ptr(), w.max_pos, w.T,
            w.n_groups, w.heads_per_group, 448, 64, 128, w.o_lora_rank, w.hidden,
            d["wo_a"].data_ptr(), d["wo_a_scale"].data_ptr(), d["wo_b"].data_ptr(),
            d["wo_b_scale"].data_ptr(), out.data_ptr(), ws.data_ptr(), need, None]
    assert lib.dsv4_o_proj(*args) == 0
    bad = list(args); bad[18] = need - 1
    assert lib.dsv4_o_proj(*bad) == -5
    bad = list(args); bad[17] = None
    assert lib.dsv4_o_proj(*bad) == -5
    bad = list(args); bad[17] = ws.data_ptr() + 16; bad[18] = need + 16
    assert lib.dsv4_o_proj(*bad) == -3
    bad = list(args); bad[11] = 200
    assert lib.dsv4_o_proj(*bad) == -1
    bad = list(args); bad[10] = 100
    assert lib.dsv4_o_proj(*bad) == -1
    bad = list(args); bad[4] = 0
    assert lib.dsv4_o_proj(*bad) == 0 and k.dsv4_last_launch_count() == 0
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0


def test_grouped_wo_a_on_prequantized_rope_quant_layout(dev):
    """A QuantizedActivation in the RopeQuant layout (o_proj page,
    rope_quant_attn_out: 16 group slots of 8 heads x 512, physical [group,
    token, K], scales [group, 8, T_al]) with only the first n_groups live: the
    padding groups are sliced off (deep_gemm_fp8_o_proj) and go straight into
    the grouped GEMM.  Padding slots hold NaN codes and garbage scales, which
    must not reach z."""
    import deepseek_v4_attention_gb300 as k
    T, slots, D, R, live = 48, 16, 4096, 1024, 12
    T_al = k.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, live, D, seed=77, tma_aligned_T=T_al)
    data = torch.full((slots, T, D), 0x7F, dtype=torch.uint8)        # NaN codes everywhere
    data[:live] = x
    scale = torch.full((slots, D // 512, T_al), 0x7F7F7F7F, dtype=torch.int32)
    scale[:live] = xs
    w, ws = di.fp8_block_weight(live * R, D, seed=78)
    view = data.to(dev).view(torch.float8_e4m3fn).transpose(0, 1)    # [T, 16, 4096]
    sview = scale.to(dev).permute(2, 0, 1)[:T]                        # [T, 16, 8]
    z = k.dsv4_grouped_wo_a(view[:, :live], sview[:, :live], w.to(dev), ws.to(dev), live, R)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    _, z64 = oracle.grouped_gemm(x, xs, w, ws, T, live, D, R, want_fp64=True)
    zg = to_bits(z)
    assert not np.isnan(torch.from_numpy(zg.view(np.int16)).view(torch.bfloat16).float().numpy()).any()
    assert gemm_rel_err(zg, z64) <= GEMM_RTOL



# ---------------------------------------------------------------------------
# bf16 variants: quantize=False and the bf16 grouped product (bmm path)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,T", [("tiny", 16), ("decode", 64), ("quant1k", 129)])
def test_inv_rope_bf16_parity(dev, name, T):
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS[name].with_tokens(T, seed=T + 3)
    d = di.make_inputs(w, with_wo_b=False)
    x = k.dsv4_inv_rope_bf16(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                             w.n_groups, w.heads_per_group)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    assert x.shape == (w.T, w.n_groups, w.D) and x.stride() == (w.D, w.T * w.D, 1)
    ref = oracle.inv_rope_bf16(d["o"], d["positions"], d["cache"], w.n_groups, w.heads_per_group)
    got = to_bits(x.transpose(0, 1))
    assert np.array_equal(got, ref)          # same fp32 order, same rounding: bit-exact


# CTA pairs: (1200, 4, 512, 1024) (8 k-blocks of 64), (300, 16, 192, 1024)
# (three k-blocks; the odd CTA's rows past T), (129, 16, 64, 2048) (one k-block,
# one token in the odd CTA); one SM, 256-wide: (128, 16, 256, 2560)
@pytest.mark.parametrize("T,G,D,R", [(16, 2, 1024, 128), (64, 8, 4096, 1024), (3, 1, 64, 128),
                                     (129, 3, 640, 384), (1200, 4, 512, 1024),
                                     (300, 16, 192, 1024), (129, 16, 64, 2048),
                                     (128, 16, 256, 2560)])
def test_grouped_wo_a_bf16_parity(dev, T, G, D, R):
    import deepseek_v4_attention_gb300 as k
    rng = np.random.default_rng(T + G)
    x = torch.from_numpy(rng.standard_normal((G, T, D)).astype(np.float32)).to(torch.bfloat16)
    wt = torch.from_numpy(rng.standard_normal((G * R, D)).astype(np.float32) * 0.02).to(
        torch.bfloat16)
    z = k.dsv4_grouped_wo_a_bf16(x.to(dev).transpose(0, 1), wt.to(dev), G, R)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    _, z64 = oracle.grouped_gemm_bf16(x, wt, T, G, D, R, want_fp64=True)
    assert gemm_rel_err(to_bits(z), z64) <= GEMM_RTOL


def test_bf16_path_chain_on_decode(dev):
    """grouped_input then the bmm path, as deep_gemm_fp8_o_proj runs them for a
    bf16 wo_a, against the oracle chain."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["decode"]
    d = di.make_inputs(w, with_wo_b=False)
    rng = np.random.default_rng(5)
    wt = torch.from_numpy(rng.standard_normal((w.n_groups * w.o_lora_rank, w.D)).astype(
        np.float32) * 0.02).to(torch.bfloat16)
    x = k.dsv4_inv_rope_bf16(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                             w.n_groups, w.heads_per_group)
    z = k.dsv4_grouped_wo_a_bf16(x, wt.to(dev), w.n_groups, w.o_lora_rank)
    torch.cuda.synchronize()
    xr = oracle.inv_rope_bf16(d["o"], d["positions"], d["cache"], w.n_groups, w.heads_per_group)
    _, z64 = oracle.grouped_gemm_bf16(xr, wt, w.T, w.n_groups, w.D, w.o_lora_rank, want_fp64=True)
    assert gemm_rel_err(to_bits(z), z64) <= GEMM_RTOL


def _random_o_proj_case(i):
    import dataclasses
    rng = np.random.default_rng(4242 + i)
    G = int(rng.integers(1, 5))
    hpg = int(rng.integers(1, 4))
    R = 128 * int(rng.integers(1, 4))
    hidden = 128 * int(rng.integers(1, 5))
    T = int(rng.choice([1, 2, 17, 63, 64, 65, 127, 200, 300]))
    return dataclasses.replace(di.WORKLOADS["tiny"], T=T, n_groups=G, heads_per_group=hpg,
                               o_lora_rank=R, hidden=hidden, seed=5000 + i)


@pytest.mark.parametrize("i", range(12))
def test_o_proj_random_shapes(dev, i):
    """Seeded random (T, G, hpg, R, hidden): every tile path (128 / 256 wide,
    split-K, 64-row A box, ragged T) against the oracle's whole chain."""
    w = _random_o_proj_case(i)
    d = di.make_inputs(w)
    out, ws = _o_proj_gpu(d, w, dev)
    check_o_proj_parts(d, w, out, ws)


# ---------------------------------------------------------------------------
# quantiser fused into wo_a (decode sizes)
# ---------------------------------------------------------------------------

def _fused_and_separate(w, d, dev):
    import deepseek_v4_attention_gb300 as k
    o, pos, cache = d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev)
    wa, was = d["wo_a"].to(dev), d["wo_a_scale"].to(dev)
    zf = k.dsv4_inv_rope_grouped_wo_a(o, pos, cache, wa, was, w.n_groups, w.heads_per_group,
                                      w.o_lora_rank)
    assert k.dsv4_last_launch_count() == 1
    sf = k.dsv4_device_status(clear=True)
    q, sc = k.dsv4_inv_rope_fp8_quant(o, pos, cache, w.n_groups, w.heads_per_group)
    zs = k.dsv4_grouped_wo_a(q, sc, wa, was, w.n_groups, w.o_lora_rank)
    ss = k.dsv4_device_status(clear=True)
    return to_bits(zf), to_bits(zs), sf, ss


# (T, G, hpg, R): split-K cluster tiles (even hpg, few tiles), one CTA per tile
# (hpg = 1, or 128 tiles), ragged T, a single token, column-tile counts 1-16
@pytest.mark.parametrize("T,G,hpg,R", [(1, 2, 2, 128), (7, 8, 8, 1024), (16, 2, 2, 128),
                                       (33, 4, 4, 256), (64, 8, 8, 1024), (64, 16, 8, 1024),
                                       (5, 3, 1, 384), (12, 2, 2, 512), (64, 1, 8, 2048)])
def test_fused_wo_a_equals_quant_then_gemm(dev, T, G, hpg, R):
    """The fused producer runs the quantiser's arithmetic: z is bit-identical to
    dsv4_grouped_wo_a of dsv4_inv_rope_fp8_quant's output, and within the GEMM
    tolerance of the oracle."""
    w = di.Workload("fused", T=T, n_groups=G, heads_per_group=hpg, o_lora_rank=R, hidden=256,
                    max_pos=4096, seed=T * 31 + G)
    d = di.make_inputs(w, with_wo_b=False)
    zf, zs, sf, ss = _fused_and_separate(w, d, dev)
    assert sf == 0 and ss == 0
    assert np.array_equal(zf, zs), "fused z differs from quant + grouped GEMM"
    x, xs = oracle.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], G, hpg)
    _, z64 = oracle.grouped_gemm(x, xs, d["wo_a"], d["wo_a_scale"], T, G, hpg * 512, R,
                                 want_fp64=True)
    assert gemm_rel_err(zf, z64) <= GEMM_RTOL


def test_fused_wo_a_out_of_range_position(dev):
    """A position outside [0, max_pos) is recorded (DSV4_ERR_RANGE) and that
    token's rope lanes are quantised unrotated, exactly as by the quantiser."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["decode"].with_tokens(9, seed=5)
    d = di.make_inputs(w, with_wo_b=False)
    d["positions"][3] = w.max_pos + 7
    zf, zs, sf, ss = _fused_and_separate(w, d, dev)
    assert k.STATUS[sf] == "DSV4_ERR_RANGE" and ss == sf
    assert np.array_equal(zf, zs)


# ("full", 600): the CTA-pair kernel (3 x 4 x 16 pair tiles)
@pytest.mark.parametrize("name,T", [("decode", 64), ("decode", 7), ("prefill", 300),
                                    ("full", 600)])
def test_grouped_wo_a_overlapping_the_quantiser(dev, name, T):
    """wo_a launched to overlap the kernel before it (DSV4_OVERLAP_PREVIOUS):
    the quantiser overwrites x with another token batch just before, on the
    same stream, and z must be that of the new x, bit-identical to the
    serialised launch (x is read only after the quantiser has completed)."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS[name].with_tokens(T, seed=T + 21)
    d1 = di.make_inputs(w, with_wo_b=False)
    d2 = di.make_inputs(w.with_tokens(T, seed=T + 22), with_wo_b=False)
    wa, was = d1["wo_a"].to(dev), d1["wo_a_scale"].to(dev)
    cache = d1["cache"].to(dev)
    x = torch.empty(w.n_groups, T, w.D, dtype=torch.float8_e4m3fn, device=dev)
    xs = torch.empty(w.n_groups, (w.D // 128 + 3) // 4, k.tma_aligned_tokens(T),
                     dtype=torch.int32, device=dev)

    def quant(d):
        return k.dsv4_inv_rope_fp8_quant(d["o"].to(dev), d["positions"].to(dev), cache,
                                         w.n_groups, w.heads_per_group, out_fp8=x, out_scale=xs)

    quant(d1)
    torch.cuda.synchronize()
    q, s = quant(d2)
    z_ov = k.dsv4_grouped_wo_a(q, s, wa, was, w.n_groups, w.o_lora_rank, overlap_previous=True)
    torch.cuda.synchronize()
    z_se = k.dsv4_grouped_wo_a(q, s, wa, was, w.n_groups, w.o_lora_rank)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    assert torch.equal(z_ov.view(torch.int16), z_se.view(torch.int16))
    lib = k.load_library()
    assert lib.dsv4_grouped_wo_a_ex(q.data_ptr(), s.data_ptr(), T, w.n_groups, w.D,
                                    w.o_lora_rank, wa.data_ptr(), was.data_ptr(),
                                    z_se.data_ptr(), 2, None) == -1      # unknown flag bit


def test_o_proj_all_zero_input(dev):
    """The degenerate input: o all zero.  Every 128-block of x and of zq has the
    floor scale (amax floored at 1e-4: byte 105), every code is +-0, and the
    output is exactly zero."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["full"].with_tokens(37, seed=3)
    d = di.make_inputs(w)
    d["o"] = torch.zeros_like(d["o"])
    out, ws = _o_proj_gpu(d, w, dev)
    parts = k.o_proj_workspace_views(ws, w.T, w.n_groups, w.heads_per_group, w.head_dim,
                                     w.o_lora_rank)
    assert bool((out.view(torch.int16) == 0).all())
    for name in ("x", "zq"):
        c = parts[name].cpu()
        assert bool(((c & 0x7F) == 0).all()), name
    xs = parts["xs"].cpu().numpy()[:, :, :w.T].view(np.uint8)
    assert (xs == 105).all()
    zs = parts["zs"].cpu().numpy()[:, :w.T].view(np.uint8)
    assert (zs == 105).all()            # G*R/128 = 128 blocks: every byte is a block
    check_o_proj_parts(d, w, out, ws)


@pytest.mark.parametrize("D", [65536])
def test_grouped_wo_a_largest_k(dev, D):
    """K = 65536, the largest reduction whose weight-scale words (128 packs of
    four 128-blocks) the GEMM holds per lane: every branch of the pack lookup."""
    T, G, R = 5, 1, 128
    T_al = oracle.tma_aligned_tokens(T)
    x, xs = di.random_fp8_activation(T, G, D, seed=91, tma_aligned_T=T_al)
    w, ws = di.fp8_block_weight(G * R, D, seed=92)
    zg = _gpu_wo_a(x, xs, w, ws, T, G, D, R, dev)
    _, z64 = oracle.grouped_gemm(x, xs, w, ws, T, G, D, R, want_fp64=True)
    assert gemm_rel_err(zg, z64) <= GEMM_RTOL


def test_grouped_wo_a_k_beyond_the_limit_is_rejected(dev):
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    T, D, R = 4, 65536 + 128, 128
    x = torch.zeros(T, D, dtype=torch.uint8, device=dev)
    xs = torch.zeros((D // 128 + 3) // 4, T, dtype=torch.int32, device=dev)
    w = torch.zeros(R, D, dtype=torch.uint8, device=dev)
    ws = torch.zeros(1, D // 128, dtype=torch.uint8, device=dev)
    z = torch.full((T, R), 7, dtype=torch.int16, device=dev)
    rc = lib.dsv4_grouped_wo_a(x.data_ptr(), xs.data_ptr(), T, 1, D, R, w.data_ptr(),
                               ws.data_ptr(), z.data_ptr(), None)
    assert rc == k._NAME_TO_CODE["DSV4_ERR_UNSUPPORTED"]
    torch.cuda.synchronize()
    assert bool((z == 7).all())          # nothing was launched
