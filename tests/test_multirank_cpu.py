"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1) check the
slowest-rank timing and the whole-job throughput of independent replicas,
and that the reference arm prints only on rank 0."""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 + rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, world)
    value = bench.job_throughput(1585.71e9, world, slowest)
    # the reference arm: only rank 0 prints its line
    buf = io.StringIO()
    args = type("A", (), dict(steps=1, warmup=0, workload="tiny"))()
    with redirect_stdout(buf):
        bench.run_reference(args)
    dist.destroy_process_group()
    q.put((rank, slowest, value, buf.getvalue()))


def test_two_gloo_ranks_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, slowest, value, text in out:
        assert slowest == 3.0
        assert value == pytest.approx(2 * 1585.71e9 / 3.0e-3 / 1e12)
        assert ('"impl": "reference"' in text) == (rank == 0)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)
