"""The N>1 path of bench.py on CPU: two gloo ranks on this host.

The attention path shards into independent problems, so ranks are replicas
that exchange nothing on the data path; the only collectives are the timing
barrier and the max over ranks of the measured times.  These tests run those
helpers exactly as bench.py calls them, with world_size 2.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup()
    try:
        bench.barrier(w)
        # every rank reports its own time; all must agree on the slowest
        t_max = bench.allreduce_max(0.25 * (rank + 1), w, torch.device("cpu"))
        bench.barrier(w)
        out.put((r, w, local, dist.get_backend(), t_max))
    finally:
        dist.destroy_process_group()


def _run_ranks(world: int):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(results)


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the CPU one")
def test_two_gloo_ranks_agree_on_the_slowest_time():
    res = _run_ranks(2)
    assert [r[0] for r in res] == [0, 1]
    for rank, world, local, backend, t_max in res:
        assert world == 2 and local == rank
        assert backend == "gloo"
        assert t_max == pytest.approx(0.5)


def test_single_rank_helpers_are_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.0, 1, torch.device("cpu")) == 3.0
    bench.barrier(1)  # no process group needed with one rank
