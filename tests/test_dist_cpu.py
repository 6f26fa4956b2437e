"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with its own
token shard (weak scaling, no collective on the data path), timing reduced as the
max over ranks, whole-job throughput over all ranks' tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import dsv4_inputs as di
        w = bench.rank_workload(di.WORKLOADS["tiny"], rank)
        d = di.make_inputs(w)
        # the data path of a rank touches only its own tensors: checksum them
        chk = torch.tensor([float(d["o"].float().abs().sum()), float(d["positions"].sum())])
        gathered = [torch.zeros(2) for _ in range(world)]
        dist.all_gather(gathered, chk)
        # weights are replicated: identical on every rank
        wchk = torch.tensor([float(d["wo_a"].double().sum() + d["wo_b"].double().sum())])
        wg = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(wg, wchk.double())
        my_ms = 10.0 * (rank + 1)                       # a stand-in per-rank time
        ms = bench.reduce_max(my_ms, torch.device("cpu"))
        value = bench.job_throughput(w.T, world, 5, ms)
        out[rank] = (torch.stack(gathered).tolist(), [float(x) for x in wg], ms, value, w.T)
    finally:
        dist.destroy_process_group()


def test_two_rank_token_shards_and_max_timing():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    r0, r1 = out[0], out[1]
    assert r0[0] == r1[0]                               # both ranks saw the same gather
    assert r0[0][0] != r0[0][1]                         # ... of different token shards
    assert r0[1][0] == r0[1][1]                         # replicated weights
    assert r0[2] == r1[2] == 20.0                       # max over ranks
    T = r0[4]
    assert r0[3] == pytest.approx(T * world * 5 / 0.020)


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(4096, 1, 10, 1000.0) == pytest.approx(40960.0)
