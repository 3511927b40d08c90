"""The N > 1 path of bench.py on CPU: replicas reduce their times with a
max over ranks (gloo, world size 2), the whole-job value counts every rank's
work over the slowest rank's time, and the reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench                              # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    local_ms = 10.0 * (rank + 1)                    # rank 1 is the slow replica
    m = bench.max_over_ranks(local_ms, w)
    value = bench.weak_scaling_value(100.0, 5, w, m)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, lr, m, value))


def test_replicas_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, m, value in res:
        assert m == 20.0                              # both ranks see the slowest time
        assert value == pytest.approx(100.0 * 5 * 2 / 0.020)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(10.0, 4, 1, 2000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(None) == 0       # returns before touching its arguments
    assert buf.getvalue() == ""
