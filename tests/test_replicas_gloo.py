"""The N > 1 bench path on the CPU: two gloo ranks on 127.0.0.1 agree on the
max-over-ranks step time and on the whole-job value (replicas only: every
GPU runs the full single-GPU emulation, so there is no data-path
collective, only the timing barrier and max)."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_setup()
    ms_local = 1.0 + rank          # rank 1 is the slower replica
    bench.barrier(w)
    ms = bench.barrier_max(ms_local, w)
    value = bench.replica_value(w, 1e9, ms)
    q.put((r, w, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[2] == pytest.approx(2.0) for o in out)          # max over ranks
    assert all(o[3] == pytest.approx(2 * 1e9 / 2e-3 / 1e9) for o in out)
