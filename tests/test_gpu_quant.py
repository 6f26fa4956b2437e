"""GPU parity of dsv4_inv_rope_fp8_quant against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import dsv4_inputs as di
import oracle
from gpu_helpers import assert_codes_match, cuda_or_skip, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _run_gpu(d, w, dev, guard=True):
    import deepseek_v4_attention_gb300 as k
    T, G, D = w.T, w.n_groups, w.D
    PK = (D // 128 + 3) // 4
    T_al = k.tma_aligned_tokens(T)
    # outputs with guard regions: every byte outside the logical region must stay 0xA5
    fp8_buf = torch.full((G * T * D + 4096,), 0xA5, dtype=torch.uint8, device=dev)
    sc_buf = torch.full((G * PK * T_al + 1024,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    out_fp8 = fp8_buf[: G * T * D].view(torch.float8_e4m3fn).view(G, T, D)
    out_sc = sc_buf[: G * PK * T_al].view(G, PK, T_al)
    q, s = k.dsv4_inv_rope_fp8_quant(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                                     G, w.heads_per_group, out_fp8=out_fp8, out_scale=out_sc)
    assert k.dsv4_last_launch_count() == (1 if T > 0 else 0)
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    if guard:
        tail = fp8_buf[G * T * D:].cpu()
        assert torch.all(tail == 0xA5), "bytes written past the fp8 output"
        st = sc_buf.cpu().view(G * PK * T_al + 1024)
        assert torch.all(st[G * PK * T_al:] == 0x5A5A5A5A), "words written past the scale output"
        pad = out_sc[:, :, T:].cpu()
        assert torch.all(pad == 0x5A5A5A5A), "scale pad columns [T, T_al) were written"
    assert q.shape == (T, G, D) and q.stride() == (D, T * D, 1)
    assert s.shape == (T, G, PK) and s.stride() == (1, PK * T_al, T_al)
    return out_fp8, out_sc


def _compare(w, dev, sample_tokens=None, positions=None):
    d = di.make_inputs(w, with_wo_b=False)
    if positions is not None:
        d["positions"] = positions
    q, s = _run_gpu(d, w, dev)
    qg = to_bits(q.view(torch.uint8))
    sg = s.cpu().numpy()
    if sample_tokens is None:
        qr, sr = oracle.inv_rope_fp8_quant(d["o"], d["positions"], d["cache"], w.n_groups,
                                           w.heads_per_group)
        assert np.array_equal(sg[:, :, : w.T], sr[:, :, : w.T]), "scale words differ"
        return assert_codes_match(qg, qr)
    idx = torch.from_numpy(np.sort(np.random.default_rng(w.seed).choice(
        w.T, size=sample_tokens, replace=False)))
    qr, sr = oracle.inv_rope_fp8_quant(d["o"][idx], d["positions"][idx], d["cache"], w.n_groups,
                                       w.heads_per_group)
    ii = idx.numpy()
    assert np.array_equal(sg[:, :, ii], sr[:, :, : len(ii)]), "scale words differ"
    return assert_codes_match(qg[:, ii, :], qr)


@pytest.mark.parametrize("name", ["tiny", "decode", "quant1k"])
def test_quant_parity_full(dev, name):
    frac = _compare(di.WORKLOADS[name], dev)
    assert frac == 1.0


@pytest.mark.parametrize("T", [1, 3, 5, 127, 129])
def test_quant_parity_ragged(dev, T):
    w = di.WORKLOADS["quant1k"].with_tokens(T, seed=100 + T)
    _compare(w, dev)


def test_quant_parity_prefill_outliers(dev):
    _compare(di.WORKLOADS["prefill"], dev, sample_tokens=512)


@pytest.mark.parametrize("name", ["quant8k", "quant32k"])
def test_quant_parity_sweep_sampled(dev, name):
    _compare(di.WORKLOADS[name], dev, sample_tokens=512)


def test_quant_position_zero_and_max(dev):
    w = di.WORKLOADS["tiny"]
    pos = torch.zeros(w.T, dtype=torch.int64)
    pos[1::2] = w.max_pos - 1
    _compare(w, dev, positions=pos)


def test_quant_deterministic(dev):
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["quant1k"]
    d = di.make_inputs(w, with_wo_b=False)
    o, p, c = d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev)
    a = k.dsv4_inv_rope_fp8_quant(o, p, c, w.n_groups, w.heads_per_group)
    b = k.dsv4_inv_rope_fp8_quant(o, p, c, w.n_groups, w.heads_per_group)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.uint8), b[0].view(torch.uint8))
    assert torch.equal(a[1], b[1])


def test_quant_empty_and_errors(dev):
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["tiny"].with_tokens(0)
    d = di.make_inputs(w, with_wo_b=False)
    q, s = k.dsv4_inv_rope_fp8_quant(d["o"].to(dev), d["positions"].to(dev), d["cache"].to(dev),
                                     w.n_groups, w.heads_per_group)
    assert q.shape[0] == 0 and k.dsv4_last_launch_count() == 0
    lib = k.load_library()
    o = torch.zeros(4, 4, 512, dtype=torch.bfloat16, device=dev)
    pos = torch.zeros(4, dtype=torch.int64, device=dev)
    cache = torch.zeros(16, 64, dtype=torch.float32, device=dev)
    out = torch.empty(2 * 4 * 1024, dtype=torch.uint8, device=dev)
    sc = torch.empty(2 * 2 * 4, dtype=torch.int32, device=dev)
    args = [o.data_ptr(), pos.data_ptr(), cache.data_ptr(), 4, 16, 2, 2, 448, 64, 128,
            out.data_ptr(), sc.data_ptr(), None]
    assert lib.dsv4_inv_rope_fp8_quant(*args) == 0
    bad = list(args); bad[8] = 63                        # odd rope (and nope+rope != 512)
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -1
    bad = list(args); bad[9] = 32                        # nope % qgs != qgs - rope
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -1
    bad = list(args); bad[7], bad[8] = 192, 64           # valid asserts, a head the library does not serve
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -4
    bad = list(args); bad[4] = 0                         # max_pos
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -1
    bad = list(args); bad[10] = None
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -2
    bad = list(args); bad[10] = out.data_ptr() + 1
    assert lib.dsv4_inv_rope_fp8_quant(*bad) == -3
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0


def test_quant_out_of_range_position_sets_status(dev):
    """A position outside [0, max_pos) is a data error the host cannot see: the
    kernel records DSV4_ERR_RANGE (no fault, no trap) and leaves that token's
    rope lanes unrotated."""
    import deepseek_v4_attention_gb300 as k
    w = di.WORKLOADS["tiny"]
    d = di.make_inputs(w, with_wo_b=False)
    pos = d["positions"].clone()
    pos[5] = w.max_pos + 3
    pos[6] = -1
    k.dsv4_device_status(clear=True)
    k.dsv4_inv_rope_fp8_quant(d["o"].to(dev), pos.to(dev), d["cache"].to(dev), w.n_groups,
                              w.heads_per_group)
    assert k.dsv4_device_status(clear=True) == k._NAME_TO_CODE["DSV4_ERR_RANGE"]
    assert k.dsv4_device_status(clear=True) == 0


def test_pipeline_wait_timeout_is_reported_not_trapped(dev):
    """The bounded wait of the GEMM pipelines, run on a barrier nothing arrives
    on with a 2 ms limit: the kernel returns, the host reads DSV4_ERR_TIMEOUT,
    and the device keeps working (a quantisation right after is still exact)."""
    import deepseek_v4_attention_gb300 as k
    k.dsv4_device_status(clear=True)
    k.dsv4_selftest_wait_timeout(2000)
    assert k.dsv4_device_status(clear=True) == k._NAME_TO_CODE["DSV4_ERR_TIMEOUT"]
    assert k.dsv4_device_status(clear=True) == 0
    _compare(di.WORKLOADS["tiny"], dev)


@pytest.mark.parametrize("G,hpg,T", [(1, 1, 7), (1, 2, 33), (3, 1, 5), (3, 2, 130), (2, 3, 9)])
def test_quant_parity_odd_head_counts(dev, G, hpg, T):
    """H = G * hpg not a multiple of 4 (the 1- and 2-head-per-iteration paths)."""
    import dataclasses
    w = dataclasses.replace(di.WORKLOADS["tiny"], T=T, n_groups=G, heads_per_group=hpg,
                            seed=1000 + 10 * G + hpg)
    frac = _compare(w, dev)
    assert frac == 1.0
