"""Multi-process host logic of bench.py with the gloo backend, world size 2 (CPU).

Each rank decodes its own batches (weak scaling by sequences); the timed region's
length is the max over ranks and the work is the sum over ranks.  No GPU.
"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx, sm = bench.reduce_max_sum(10.0 + 5 * rank, 100.0 * (rank + 1))
        bench.barrier()
        seeds = bench.rank_seed(1234, rank)
        q.put((rank, mx, sm, seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]          # max over ranks
    assert [g[2] for g in got] == [300.0, 300.0]        # sum over ranks
    assert got[0][3] != got[1][3]                        # different batches per rank


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_max_sum(3.0, 4.0) == (3.0, 4.0)
    assert bench.rank_seed(1234, 0) == 1234
