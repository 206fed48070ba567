"""The N>1 launch of bench.py: independent replicas, one per rank, no data-path
collective. Checked on CPU with two gloo ranks: the rendezvous, the barrier
around the timed region, the max over ranks of the step time, the whole-job
value (units of all ranks / slowest rank's time), and that only rank 0 runs
the reference arm."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "DSA_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import torch
    import bench
    r, w = bench.dist_setup(world)
    bench.barrier(w)
    ms = bench.max_over_ranks(2.0 + rank, w, torch.device("cpu"))
    value = bench.job_throughput(4096, w, ms)

    class Args:
        steps, warmup, ref_rows = 1, 0, 1
    ran = bench.run_reference(Args) if rank != 0 else "skipped"   # rank != 0 returns at once
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, ms, value, ran))


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    # every rank sees the slowest rank's step time, and the value counts both ranks' rows
    assert all(g[2] == 3.0 for g in got)
    assert all(abs(g[3] - 2 * 4096 / 3.0e-3) < 1e-6 for g in got)
    assert got[1][4] is None
