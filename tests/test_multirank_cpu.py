"""The benchmark's multi-rank plumbing on CPU: two gloo ranks (world size 2) go through the
same process-group set-up, barrier and max-over-ranks timing reduction that bench.py uses
under torchrun, and the reference arm's rule that only rank 0 works and prints."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup(backend="gloo")
    bench.barrier(w)
    m = bench.max_over_ranks(w, 1.5 + 10.0 * r)  # rank 1 is the slow one
    out = io.StringIO()
    if r != 0:
        # The reference arm: ranks other than 0 exit 0 without work or output.
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(type("A", (), {"workload": "f32_64x768", "steps": 1,
                                                    "warmup": 0})())
    else:
        rc = 0
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((r, w, m, rc, out.getvalue()))


def test_two_gloo_ranks_share_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, m, rc, out in results:
        assert w == world
        assert m == pytest.approx(11.5)  # every rank sees the max
        assert rc == 0
    assert results[1][4] == ""  # rank 1 printed nothing
