"""Group-split tensor parallelism on CPU: the partition of deepseek_v4_attention_gb300.tp
and its exchange step, with each rank's share computed by the oracle.

A rank's share is the whole O-projection over its own groups (their heads of o,
their wo_a rows, their wo_b columns); the layer's output is the sum of the
shares, because group g's z meets only wo_b columns g*R .. (g+1)*R - 1 and the
per-128 re-quantisation of z never crosses a group.  These tests pin that claim
with the oracle and run the reduce-scatter over two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import dsv4_inputs as di
from deepseek_v4_attention_gb300 import tp


def _shape(T, G, hpg, R, hidden, seed):
    import dataclasses
    return dataclasses.replace(di.WORKLOADS["tiny"], T=T, n_groups=G, heads_per_group=hpg,
                               o_lora_rank=R, hidden=hidden, seed=seed)


def _oracle_share(oracle, d, w, rank, world):
    o = tp.shard_o(d["o"], rank, world, w.n_groups, w.heads_per_group)
    s = tp.shard_weights(d["wo_a"], d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], rank, world,
                         w.n_groups, w.o_lora_rank)
    g0, g1 = s.groups
    _, out64, _ = oracle.o_proj(o, d["positions"], d["cache"], s.wo_a, s.wo_a_scale, s.wo_b,
                                s.wo_b_scale, n_groups=g1 - g0,
                                heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank,
                                hidden=w.hidden)
    return out64


def test_partition():
    assert tp.group_range(0, 2, 16) == (0, 8) and tp.group_range(1, 2, 16) == (8, 16)
    assert tp.group_range(3, 8, 16) == (6, 8)
    with pytest.raises(ValueError):
        tp.group_range(0, 3, 16)
    with pytest.raises(ValueError):
        tp.group_range(2, 2, 16)
    for T in (1, 7, 64, 4097):
        for world in (1, 2, 4, 8):
            rows = []
            for r in range(world):
                T_pad, t0, n = tp.token_chunk(T, r, world)
                assert T_pad % world == 0 and T_pad >= T
                rows += list(range(t0, t0 + n))
            assert rows == list(range(T))          # every token owned once, in order
    w = _shape(5, 4, 2, 256, 384, 1)
    d = di.make_inputs(w)
    s = tp.shard_weights(d["wo_a"], d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], 1, 2, 4, 256)
    assert s.groups == (2, 4)
    assert torch.equal(s.wo_a, d["wo_a"][512:1024]) and s.wo_b.is_contiguous()
    assert torch.equal(s.wo_b, d["wo_b"][:, 512:1024])
    assert torch.equal(s.wo_b_scale, d["wo_b_scale"][:, 4:8])
    assert torch.equal(s.wo_a_scale, d["wo_a_scale"][4:8])
    o = tp.shard_o(d["o"], 1, 2, 4, 2)
    assert torch.equal(o, d["o"][:, 4:8]) and o.is_contiguous()


@pytest.mark.parametrize("T,G,hpg,R,hidden,world", [(9, 4, 2, 256, 384, 2), (5, 4, 1, 128, 256, 4),
                                                    (3, 2, 3, 384, 128, 2)])
def test_shares_sum_to_the_layer_output(oracle_mod, T, G, hpg, R, hidden, world):
    """The oracle's O-projection over each rank's groups, summed over the ranks,
    equals the oracle's O-projection of the whole layer (fp64, up to summation
    order: relative 1e-12)."""
    w = _shape(T, G, hpg, R, hidden, 11 * T + G)
    d = di.make_inputs(w)
    _, full64, _ = oracle_mod.o_proj(d["o"], d["positions"], d["cache"], d["wo_a"],
                                     d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], n_groups=G,
                                     heads_per_group=hpg, o_lora_rank=R, hidden=hidden)
    total = sum(_oracle_share(oracle_mod, d, w, r, world) for r in range(world))
    scale = np.abs(full64).max()
    assert np.abs(total - full64).max() <= 1e-12 * scale


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, shape, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        w = _shape(*shape)
        d = di.make_inputs(w)
        shard = tp.shard_weights(d["wo_a"], d["wo_a_scale"], d["wo_b"], d["wo_b_scale"], rank,
                                 world, w.n_groups, w.o_lora_rank)
        o_local = tp.shard_o(d["o"], rank, world, w.n_groups, w.heads_per_group)

        def partial_fn(o, pos, cache, wa, was, wb, wbs, *, n_groups, heads_per_group,
                       o_lora_rank):
            _, out64, _ = oracle.o_proj(o, pos, cache, wa, was, wb, wbs, n_groups=n_groups,
                                        heads_per_group=heads_per_group,
                                        o_lora_rank=o_lora_rank, hidden=wb.shape[0])
            return torch.from_numpy(out64)        # fp64 stands in for the kernel's fp32

        rows = tp.o_proj_tp(o_local, d["positions"], d["cache"], shard,
                            heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank,
                            partial_fn=partial_fn, finish_fn=lambda x: x.clone())
        out[rank] = rows.numpy()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shape", [(9, 4, 2, 256, 384, 5), (2, 2, 2, 128, 256, 6)])
def test_two_rank_reduce_scatter(oracle_mod, shape):
    """Two gloo ranks: each computes its share, one reduce-scatter leaves each
    rank the summed rows of its own token chunk, and together they are the
    layer's output."""
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), shape, out), nprocs=world,
                       join=True, start_method="spawn")
    w = _shape(*shape)
    d = di.make_inputs(w)
    _, full64, _ = oracle_mod.o_proj(d["o"], d["positions"], d["cache"], d["wo_a"],
                                     d["wo_a_scale"], d["wo_b"], d["wo_b_scale"],
                                     n_groups=w.n_groups, heads_per_group=w.heads_per_group,
                                     o_lora_rank=w.o_lora_rank, hidden=w.hidden)
    got = np.concatenate([out[r] for r in range(world)], axis=0)
    assert got.shape == full64.shape
    assert np.abs(got - full64).max() <= 1e-12 * np.abs(full64).max()
