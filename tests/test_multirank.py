"""Multi-process host logic of the benchmark on CPU (gloo, world size 2):
each rank runs an independent replica (the decode path has no exchange
step), ranks meet at barriers, and the timed figure is the max over ranks.
No GPU and no collective on the data path are involved."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    r, w, _ = bench.dist_info()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.reduce_max(10.0 + r, w)           # rank-local "time"
    # the reference arm runs on rank 0 only; the other ranks exit at once
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                             "--warmup", "0"])
    rc = bench.run_reference(args) if r != 0 else 0
    bench.barrier(w)
    q.put((r, mx, rc))
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [11.0, 11.0]        # max over ranks on every rank
    assert [g[2] for g in got] == [0, 0]


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)      # no process group needed for one rank
