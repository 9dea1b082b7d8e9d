"""bench.py's multi-rank host logic on CPU (gloo, world size 2): one process per
rank initialised from RANK / WORLD_SIZE / MASTER_* as under torchrun, a
barrier on both sides of the timed region, and the timing reduced as the
maximum over ranks.  The operator itself has no exchange step (replicas),
so this is all the N > 1 path needs."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    # no GPU in these ranks: bench.init_dist then takes the gloo backend
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.init_dist()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    got = bench.max_over_ranks(values[rank], w)
    bench.barrier(w)
    out.put((rank, got))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_maximum_time():
    import torch.multiprocessing as mp
    pytest.importorskip("torch.distributed")
    world, port = 2, _free_port()
    values = [3.25, 7.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: max(values), 1: max(values)}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    bench.barrier(1)
