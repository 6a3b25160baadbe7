"""The multi-GPU path is replicas only: each rank runs its own decode stream
with no exchange, and bench.py reports all ranks' work over the slowest
rank's time.  The aggregation is checked here with world_size 2 on gloo
(CPU), the same code the NCCL launch uses."""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 12.5][rank]          # rank 1 is the slower replica
        mx = bench._max_over_ranks(world, local_ms)
        thr = bench.replica_throughput(world, 1000.0, local_ms)
        dist.barrier()
        q.put((rank, mx, thr))
    finally:
        dist.destroy_process_group()


def _rank_setup(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    import synth
    devices = []
    ws, r, local = bench._dist(set_device=devices.append, backend="gloo")
    try:
        # each replica's first streaming step, from its own seed
        q_, k_, v_, pos = synth.streaming_inputs(steps=2, Hq=bench.HQ, Hkv=bench.HKV, D=bench.D,
                                                 seed=bench.replica_seed(r), device="cpu")
        mine = torch.tensor([float(q_.float().sum()), float(k_.float().abs().sum())],
                            dtype=torch.float64)
        both = [torch.zeros_like(mine) for _ in range(ws)]
        dist.all_gather(both, mine)
        q.put((r, ws, local, devices, [b.tolist() for b in both]))
    finally:
        dist.destroy_process_group()


def test_replica_setup_picks_local_rank_device_and_distinct_inputs():
    """What the NCCL launch does per rank, on gloo: the device is
    LOCAL_RANK, and the two replicas stream different synthetic inputs."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_setup, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ws, local, devices, both in got:
        assert ws == 2 and local == rank and devices == [rank]
        assert both[0] != both[1]  # rank 0's inputs differ from rank 1's
    assert got[0][4] == got[1][4]  # both ranks gathered the same pair


def test_two_replicas_report_max_time_and_summed_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, thr in got:
        assert mx == pytest.approx(12.5)
        # 2 ranks x 1000 units over the slowest rank's 12.5 ms
        assert thr == pytest.approx(2 * 1000.0 / 12.5e-3)
