"""bench.py's multi-rank accounting on CPU: two gloo ranks reduce their timings to
the maximum, the whole-job throughput counts every rank's tokens within that time,
and the reference arm's non-zero ranks exit 0 without output."""
import io
import json
import os
import sys
import contextlib

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r times step 1 + r ms, attention 5 - r ms
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.5 * rank], world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_timings_reduce_to_the_slowest_rank(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got == [2.0, 5.0, 0.5]          # max over ranks of each timing, on every rank


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_job_throughput_is_weak_scaling():
    import bench
    # 1000 tokens per rank, 2 ms per step: 0.5 M tokens/s per rank
    assert bench.job_throughput(1000, 1, 2.0) == pytest.approx(5e5)
    assert bench.job_throughput(1000, 4, 2.0) == pytest.approx(2e6)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""
