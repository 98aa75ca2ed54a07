"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2): the whole-job
line takes the max time over ranks and the sum of units over ranks, and the
reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(1.0 + rank, 10.0 * (rank + 1))
    ref = bench.run_reference(bench.argparse.Namespace(config=1, ref_tokens=8, warmup=0, steps=1),
                              bench.CONFIGS[1]) if rank == 1 else None
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, u, ref))


def test_aggregate_max_time_sum_units_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u, ref in res:
        assert t == pytest.approx(2.0)
        assert u == pytest.approx(30.0)
        assert ref is None  # only rank 0 runs the reference arm


def test_aggregate_single_process_is_identity():
    import bench

    assert bench.aggregate(1.5, 7.0) == (1.5, 7.0)
