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


def test_write_aware_floor_is_a_lower_bound_of_each_kind():
    """The write-aware HBM floor is the larger of two lower bounds: written bytes at the
    write-only rate, all bytes at the copy rate; written bytes never exceed a kernel's
    algorithmic bytes."""
    import bench
    from workloads import CONFIGS
    c = CONFIGS["fwd_bf16"]
    pk = dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="test", hbm_write=4000.0)
    for k in ("gemm_up_swiglu", "gemm_down_push", "gemm_g_swiglu_bwd", "gemm_dgrad_push",
              "wgrad_w13", "wgrad_w2", "gather", "combine", "gather_bwd", "dx_reduce"):
        _, nbytes = bench.algorithmic(k, c)
        wr = bench.algorithmic_writes(k, c)
        assert 0 < wr <= nbytes, k
        r = bench.roofline_of(k, c, 1, 1.0, pk)
        floor = r["hbm_rw_floor_ms"] * 1e-3
        assert floor >= nbytes / 6800e9 - 1e-12 and floor >= wr / 4000e9 - 1e-12
        assert abs(r["frac_hbm_rw"] - floor / 1e-3) < 1e-9
    # dW13 is bound by its bf16 writes: 8.6 GB at the write-only rate
    r = bench.roofline_of("wgrad_w13", c, 1, 1.0, pk)
    assert abs(r["hbm_rw_floor_ms"] - 2.0 * c.E * 2 * c.I * c.H / 4000e9 * 1e3) < 1e-9
