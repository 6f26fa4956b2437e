"""Group-split tensor parallelism of the O-projection (host side).

The layer's groups are split into equal contiguous ranges, one per rank, as the
attention layer of sglang's deepseek_v4.py splits its heads: wo_a is
column-parallel (rank r holds the wo_a rows of its groups), wo_b row-parallel
(rank r holds the wo_b columns g*R .. (g+1)*R - 1 of each of its groups g),
and the outputs of the ranks are summed (attn_tp_all_reduce there; the vLLM
o_proj page's DeepSeek-V4.1 GEMM-RS reduce-scatters instead, leaving each rank
the sum for its own tokens).  Because group g's z meets only its own wo_b
columns and the per-128 re-quantisation of z never crosses a group, a rank's
share is the whole O-projection over its own groups
(dsv4_o_proj_partial, fp32) and the layer's output is the sum of the shares.

This module holds the partition (which groups, heads, weight rows and
columns, and which output tokens belong to a rank) and the exchange step: one
fp32 reduce-scatter over equal token chunks, then the bf16 rounding of the
rank's rows (dsv4_sum_partials with one partial).  The collective is
torch.distributed's (NCCL between GPUs); every step of the arithmetic runs in
the library's kernels.
"""
from __future__ import annotations

import dataclasses

import torch


def group_range(rank: int, world: int, n_groups: int) -> tuple[int, int]:
    """Groups [g0, g1) of `rank` when n_groups are split over `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if n_groups % world != 0:
        raise ValueError(f"{n_groups} groups do not split evenly over {world} ranks")
    per = n_groups // world
    return rank * per, (rank + 1) * per


def shard_o(o: torch.Tensor, rank: int, world: int, n_groups: int,
            heads_per_group: int) -> torch.Tensor:
    """The rank's heads of the attention output o [T, H, head_dim] (contiguous)."""
    g0, g1 = group_range(rank, world, n_groups)
    return o[:, g0 * heads_per_group:g1 * heads_per_group].contiguous()


@dataclasses.dataclass
class WeightShard:
    wo_a: torch.Tensor          # e4m3 [G_local*R, D]
    wo_a_scale: torch.Tensor    # UE8M0 [G_local*R/128, D/128]
    wo_b: torch.Tensor          # e4m3 [hidden, G_local*R], contiguous
    wo_b_scale: torch.Tensor    # UE8M0 [hidden/128, G_local*R/128]
    groups: tuple[int, int]


def shard_weights(wo_a: torch.Tensor, wo_a_scale: torch.Tensor, wo_b: torch.Tensor,
                  wo_b_scale: torch.Tensor, rank: int, world: int, n_groups: int,
                  o_lora_rank: int) -> WeightShard:
    """The rank's rows of wo_a (column-parallel) and columns of wo_b
    (row-parallel), with their 128 x 128 block scales."""
    if o_lora_rank % 128 != 0:
        raise ValueError("o_lora_rank must be a multiple of 128")
    g0, g1 = group_range(rank, world, n_groups)
    r0, r1 = g0 * o_lora_rank, g1 * o_lora_rank
    return WeightShard(
        wo_a=wo_a[r0:r1].contiguous(),
        wo_a_scale=wo_a_scale[r0 // 128:r1 // 128].contiguous(),
        wo_b=wo_b[:, r0:r1].contiguous(),
        wo_b_scale=wo_b_scale[:, r0 // 128:r1 // 128].contiguous(),
        groups=(g0, g1))


def token_chunk(num_tokens: int, rank: int, world: int) -> tuple[int, int, int]:
    """(padded token count, first row, row count) of the rank's output rows
    after the reduce-scatter over equal token chunks; rows past num_tokens are
    padding and belong to no one."""
    per = -(-num_tokens // world)
    t0 = rank * per
    return per * world, t0, max(0, min(per, num_tokens - t0))


def o_proj_tp(o_local: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
              shard: WeightShard, *, heads_per_group: int, o_lora_rank: int, group=None,
              partial_fn=None, finish_fn=None) -> torch.Tensor:
    """One rank's step of the group-split O-projection: its fp32 share of the
    output, one reduce-scatter (sum) over equal token chunks, and the bf16
    rounding of its own rows.  Returns the rank's rows [rows, hidden] (see
    token_chunk).  partial_fn / finish_fn default to the library's
    dsv4_o_proj_partial / dsv4_sum_partials."""
    import torch.distributed as dist
    if partial_fn is None or finish_fn is None:
        import deepseek_v4_attention_gb300 as k
        partial_fn = partial_fn or k.dsv4_o_proj_partial
        finish_fn = finish_fn or (lambda x: k.dsv4_sum_partials([x]))
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    T = o_local.shape[0]
    g0, g1 = shard.groups
    part = partial_fn(o_local, positions, cos_sin_cache, shard.wo_a, shard.wo_a_scale,
                      shard.wo_b, shard.wo_b_scale, n_groups=g1 - g0,
                      heads_per_group=heads_per_group, o_lora_rank=o_lora_rank)
    T_pad, t0, rows = token_chunk(T, rank, world)
    hidden = part.shape[1]
    if T_pad != T:
        padded = torch.zeros((T_pad, hidden), dtype=part.dtype, device=part.device)
        padded[:T] = part
        part = padded
    mine = torch.empty((T_pad // world, hidden), dtype=part.dtype, device=part.device)
    dist.reduce_scatter_tensor(mine, part, op=dist.ReduceOp.SUM, group=group)
    return finish_fn(mine[:rows].contiguous())
