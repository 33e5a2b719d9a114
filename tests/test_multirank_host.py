"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend.

The attention path shards by (batch, head) with no exchange, so the only
cross-rank step is the benchmark's own timing: the step time is the maximum
over ranks and the job throughput counts every rank's work over it.
"""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 1.5 + rank  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    q.put((rank, bench.dist_env(), m, bench.job_throughput(1e12, world, m)))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, m, value in got:
        assert env[0] == rank and env[1] == 2
        assert m == 2.5                              # the slowest rank's step time
        assert abs(value - 1e12 * 2 / 2.5e-3 / 1e12) < 1e-9  # both ranks' work over it


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert abs(bench.job_throughput(2e12, 1, 4.0) - 500.0) < 1e-9
