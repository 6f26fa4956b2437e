"""GPU parity of the pre-quantised O-projection (dsv4_o_proj_prequant), the
group-range share (dsv4_o_proj_partial) and the sum of shares
(dsv4_sum_partials), through the C ABI.  Tolerances: gpu_helpers."""
import numpy as np
import pytest
import torch

import dsv4_inputs as di
import oracle
from deepseek_v4_attention_gb300 import tp
from gpu_helpers import (GEMM_RTOL, assert_codes_match, chain_allowance, cuda_or_skip,
                         gemm_rel_err, rel_errs, scale_bytes, to_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("n,elems", [(1, 4096 * 7 + 5), (2, 1000), (3, 8), (4, 3), (16, 777)])
def test_sum_partials_exact(dev, n, elems):
    """fp32 sum in list order, rounded to nearest even bf16: bit-exact against
    the same sum done by torch on the CPU."""
    import deepseek_v4_attention_gb300 as k
    g = torch.Generator().manual_seed(n * 1000 + elems)
    parts = [torch.randn(elems, generator=g) * (10.0 ** j) for j in range(n)]
    acc = parts[0].clone()
    for p in parts[1:]:
        acc += p
    ref = _bf16_bits(acc.to(torch.bfloat16))
    got = k.dsv4_sum_partials([p.to(dev) for p in parts])
    assert k.dsv4_last_launch_count() == 1
    torch.cuda.synchronize()
    assert np.array_equal(_bf16_bits(got.cpu()), ref)


def test_sum_partials_errors(dev):
    import ctypes
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    a = torch.zeros(64, device=dev)
    o = torch.empty(64, dtype=torch.bfloat16, device=dev)
    arr = (ctypes.c_void_p * 17)(*([a.data_ptr()] * 17))
    assert lib.dsv4_sum_partials(arr, 0, 64, o.data_ptr(), None) == -1
    assert lib.dsv4_sum_partials(arr, 17, 64, o.data_ptr(), None) == -1
    assert lib.dsv4_sum_partials(arr, 2, 0, o.data_ptr(), None) == 0
    assert lib.dsv4_sum_partials(arr, 2, 64, None, None) == -2
    bad = (ctypes.c_void_p * 2)(a.data_ptr(), a.data_ptr() + 4)
    assert lib.dsv4_sum_partials(bad, 2, 60, o.data_ptr(), None) == -3


def _zq_of(oracle_z_bits, T, C):
    return oracle.block_quant_rows(oracle_z_bits.reshape(T, C))


@pytest.mark.parametrize("name,T,world", [("full", 256, 2), ("full", 100, 4), ("decode", 64, 8),
                                          ("tiny", 13, 2)])
def test_group_range_shares_sum_to_the_output(dev, name, T, world):
    """Each group range's share on this GPU (dsv4_o_proj_partial, one after the
    other, nothing waiting on another), added by dsv4_sum_partials: zq of every
    share against the oracle's quantisation of its z, the output against the
    fp64 sum of the shares' products of their own zq (GEMM_RTOL), and against
    the oracle's whole layer (GEMM_RTOL plus the derived effect of any zq code
    one step off)."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS[name].with_tokens(T, seed=T + world)
    G, hpg, R, hidden = w.n_groups, w.heads_per_group, w.o_lora_rank, w.hidden
    d = di.make_inputs(w)
    _, full64, z_full = oracle.o_proj(d["o"], d["positions"], d["cache"], d["wo_a"],
                                      d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], n_groups=G,
                                      heads_per_group=hpg, o_lora_rank=R, hidden=hidden,
                                      want_z=True)
    dec = oracle.e4m3_decode_table()
    pos, cache = d["positions"].to(dev), d["cache"].to(dev)
    parts, own64, allow = [], np.zeros((T, hidden)), np.zeros((T, hidden))
    for r in range(world):
        s = tp.shard_weights(d["wo_a"], d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], r, world,
                             G, R)
        g0, g1 = s.groups
        Gl = g1 - g0
        o_l = tp.shard_o(d["o"], r, world, G, hpg).to(dev)
        need = k.dsv4_o_proj_workspace_bytes(T, Gl, hpg, 512, R)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        p = k.dsv4_o_proj_partial(o_l, pos, cache, s.wo_a.to(dev), s.wo_a_scale.to(dev),
                                  s.wo_b.to(dev), s.wo_b_scale.to(dev), n_groups=Gl,
                                  heads_per_group=hpg, o_lora_rank=R, workspace=ws)
        torch.cuda.synchronize()
        assert k.dsv4_device_status(clear=True) == 0
        parts.append(p)
        v = k.o_proj_workspace_views(ws, T, Gl, hpg, 512, R)
        zqg, zsg = v["zq"].cpu().numpy(), v["zs"].cpu().numpy()[:, :T]
        zqr, zsr = _zq_of(z_full[:, g0:g1], T, Gl * R)
        nb = Gl * R // 128
        assert np.array_equal(scale_bytes(zsg)[:nb], scale_bytes(zsr[:, :T])[:nb])
        assert_codes_match(zqg, zqr, f"zq of share {r}")
        zs_own = np.zeros((zsg.shape[0], oracle.tma_aligned_tokens(T)), dtype=np.int32)
        zs_own[:, :T] = zsg
        _, o64 = oracle.grouped_gemm(np.ascontiguousarray(zqg), zs_own, s.wo_b, s.wo_b_scale, T,
                                     1, Gl * R, hidden, want_fp64=True)
        own64 += o64.reshape(T, hidden)
        allow += chain_allowance(zqg, zqr, scale_bytes(zsg), s.wo_b, s.wo_b_scale, dec)
    out = k.dsv4_sum_partials(parts)
    torch.cuda.synchronize()
    og = to_bits(out)
    assert gemm_rel_err(og, own64) <= GEMM_RTOL
    err, den = rel_errs(og, full64)
    assert float((err - (GEMM_RTOL * den + allow)).max()) <= 0.0


@pytest.mark.parametrize("name,T", [("full", 300), ("decode", 64), ("tiny", 5)])
def test_single_share_equals_the_layer(dev, name, T):
    """With one group range (every group) the fp32 share rounded by
    dsv4_sum_partials is bit-identical to dsv4_o_proj: same kernels, same
    accumulators, one bf16 rounding."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS[name].with_tokens(T, seed=T + 77)
    d = {n_: t.to(dev) for n_, t in di.make_inputs(w).items()}
    args = (d["o"], d["positions"], d["cache"], d["wo_a"], d["wo_a_scale"], d["wo_b"],
            d["wo_b_scale"])
    kw = dict(n_groups=w.n_groups, heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank)
    ref = k.dsv4_o_proj(*args, **kw)
    got = k.dsv4_sum_partials([k.dsv4_o_proj_partial(*args, **kw)])
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    assert torch.equal(ref.view(torch.int16), got.view(torch.int16))


@pytest.mark.parametrize("T,live", [(48, 12), (130, 16), (7, 1)])
def test_o_proj_from_prequantised_rope_quant_output(dev, T, live):
    """A RopeQuant-layout attention output (16 slots of 8 heads x 512, live
    groups first, padding slots full of NaN codes and garbage scales) through
    dsv4_o_proj_prequant: zq and out checked stage by stage against the
    oracle, and out bit-identical to dsv4_o_proj on the o it came from."""
    import dataclasses
    import deepseek_v4_attention_gb300 as k
    slots, hpg, R, hidden = 16, 8, 1024, 7168
    w = dataclasses.replace(di.WORKLOADS["full"], T=T, n_groups=live, seed=T + live)
    d = di.make_inputs(w)
    x, xs = oracle.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], live, hpg)
    D, T_al = hpg * 512, oracle.tma_aligned_tokens(T)
    data = torch.full((slots, T, D), 0x7F, dtype=torch.uint8)
    data[:live] = torch.from_numpy(x)
    scale = torch.full((slots, D // 512, T_al), 0x7F7F7F7F, dtype=torch.int32)
    scale[:live] = torch.from_numpy(xs)
    xv = data.to(dev).view(torch.float8_e4m3fn).transpose(0, 1)
    sv = scale.to(dev).permute(2, 0, 1)[:T]
    wts = [d[n_].to(dev) for n_ in ("wo_a", "wo_a_scale", "wo_b", "wo_b_scale")]
    ws = torch.empty(k.dsv4_o_proj_prequant_workspace_bytes(T, live, R), dtype=torch.uint8,
                     device=dev)
    out = k.dsv4_o_proj_prequant(xv, sv, *wts, n_groups=live, o_lora_rank=R, workspace=ws)
    assert k.dsv4_last_launch_count() == 2
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    v = k.prequant_workspace_views(ws, T, live, R)
    zqg, zsg = v["zq"].cpu().numpy(), v["zs"].cpu().numpy()[:, :T]
    z = oracle.grouped_gemm(x, xs, d["wo_a"], d["wo_a_scale"], T, live, D, R)
    zqr, zsr = _zq_of(z, T, live * R)
    nb = live * R // 128
    assert np.array_equal(scale_bytes(zsg)[:nb], scale_bytes(zsr[:, :T])[:nb])
    assert_codes_match(zqg, zqr, "zq")
    zs_own = np.zeros((zsg.shape[0], T_al), dtype=np.int32)
    zs_own[:, :T] = zsg
    _, o64 = oracle.grouped_gemm(np.ascontiguousarray(zqg), zs_own, d["wo_b"], d["wo_b_scale"],
                                 T, 1, live * R, hidden, want_fp64=True)
    og = to_bits(out)
    assert gemm_rel_err(og, o64) <= GEMM_RTOL
    ref = k.dsv4_o_proj(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev), *wts,
                        n_groups=live, heads_per_group=hpg, o_lora_rank=R)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(ref), og)


def test_o_proj_prequant_errors(dev):
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    T, slots, D, R, hidden = 8, 4, 512, 128, 256
    x = torch.zeros(slots, T, D, dtype=torch.uint8, device=dev)
    xs = torch.zeros(slots, 1, T, dtype=torch.int32, device=dev)
    wa = torch.zeros(2 * R, D, dtype=torch.uint8, device=dev)
    was = torch.full((2 * R // 128, D // 128), 127, dtype=torch.uint8, device=dev)
    wb = torch.zeros(hidden, 2 * R, dtype=torch.uint8, device=dev)
    wbs = torch.full((hidden // 128, 2 * R // 128), 127, dtype=torch.uint8, device=dev)
    out = torch.empty(T, hidden, dtype=torch.bfloat16, device=dev)
    need = k.dsv4_o_proj_prequant_workspace_bytes(T, 2, R)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    args = [x.data_ptr(), xs.data_ptr(), T, slots, 2, D, R, hidden, wa.data_ptr(),
            was.data_ptr(), wb.data_ptr(), wbs.data_ptr(), out.data_ptr(), ws.data_ptr(), need,
            None]
    assert lib.dsv4_o_proj_prequant(*args) == 0
    bad = list(args); bad[4] = slots + 1                 # more live groups than slots
    assert lib.dsv4_o_proj_prequant(*bad) == -1
    bad = list(args); bad[5] = 500
    assert lib.dsv4_o_proj_prequant(*bad) == -1
    bad = list(args); bad[14] = need - 1
    assert lib.dsv4_o_proj_prequant(*bad) == -5
    bad = list(args); bad[0] = None
    assert lib.dsv4_o_proj_prequant(*bad) == -2
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    assert bool((out == 0).all())                        # zero codes: zero output


@pytest.mark.parametrize("T", [1024, 777])
def test_single_share_equals_the_layer_large(dev, T):
    """The fp32 share at sizes where both GEMMs take the 256-wide persistent
    tiles, rounded by dsv4_sum_partials: bit-identical to dsv4_o_proj."""
    test_single_share_equals_the_layer(dev, "full", T)
