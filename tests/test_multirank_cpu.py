"""Host logic of the multi-rank bench, on CPU: two gloo ranks (127.0.0.1).

Each rank is a replica of the single-GPU step; the job's time is the slowest rank's, and
the job's rate counts the units of every rank.  The reference arm runs on rank 0 only.
"""
import io
import json
import multiprocessing as mp
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


def _rank_main(rank, world, port, ms_local, q):
    sys.path.insert(0, ROOT)
    import torch
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        ms_max = bench.max_over_ranks(ms_local[rank], w, torch.device("cpu"))
        rate = bench.whole_job_rate(1e9, 10, w, ms_max, 1e9)
        q.put((r, w, ms_max, rate))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    pytest.importorskip("torch")
    world, port = 2, _free_port()
    ms_local = [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_local, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, w, ms_max, rate) in enumerate(got):
        assert rank == r and w == world
        assert ms_max == max(ms_local)  # every rank sees the slowest rank's time
        # 1e9 units per step x 10 steps x 2 ranks in 20 ms = 1e12 units/s = 1000 (x 1e9)
        assert rate == pytest.approx(1000.0)


def test_whole_job_rate_single_rank():
    import bench
    assert bench.max_over_ranks(7.0, 1, None) == 7.0
    assert bench.whole_job_rate(2.0, 5, 1, 10.0, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "3"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main() == 0
    assert buf.getvalue() == ""


def test_reference_arm_line_on_rank_zero(monkeypatch):
    """Rank 0 prints one JSON line with the reference keys (tiny sample: 1 row, 1 step)."""
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                                      "--ref-rows", "1"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main() == 0
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "TOPS" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
