"""Host logic of bench.py's multi-rank path, as two gloo ranks on CPU: the timing taken is
the maximum over ranks, the whole-job value counts every rank's work over that time, and
the reference arm prints from rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist)
        q.put((rank, ms, bench.whole_job_value(world, 1e12, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks():
    world, port = 2, _free_port()
    local_ms = [3.0, 5.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 5.0  # every rank reports the slowest rank's time
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)  # both ranks' work over it


def test_single_rank_is_identity():
    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.whole_job_value(1, 2e12, 4.0) == pytest.approx(500.0)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
