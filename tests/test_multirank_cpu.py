"""bench.py's multi-rank host path on CPU.

Under torchrun every rank runs its own copy of the workload (weak scaling, no
collective on the data path); the ranks meet at a barrier around the timed
region, and the job's time is the slowest rank's. Two gloo ranks (world size 2,
rendezvous on 127.0.0.1) stand in for two GPUs here: each reports a different
step time, and both must come out with the maximum and with the job rate
world * units / max time. No GPU is used.
"""
import os
import socket
import sys
import types

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(types.SimpleNamespace(impl="reference"))  # gloo
    bench.barrier(w)
    ms, rate = bench.job_rate(w, 1000, 10.0 + 5.0 * r)  # rank 1 is the slow one
    bench.barrier(w)
    out.put((r, w, ms, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_the_summed_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    for _, w, ms, rate in res:
        assert w == 2 and ms == 15.0
        assert abs(rate - 2 * 1000 / 15e-3) < 1e-6 * rate


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_rate(1, 500, 4.0) == (4.0, 500 / 4e-3)
