"""bench.py's multi-rank logic (replicas: barrier, max over ranks, whole-job
throughput) with world_size 2 on the gloo backend, on CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(world)
    ms = 100.0 + 50.0 * rank                     # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world)
    out[rank] = (worst, bench.whole_job_tflops(1e12, 10, world, worst))
    dist.destroy_process_group()


def test_two_rank_replicas_on_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # both ranks see the slower rank's time; throughput counts both replicas
    assert out[0][0] == out[1][0] == 150.0
    assert abs(out[0][1] - 2 * 1e12 * 10 / 0.150 / 1e12) < 1e-9
