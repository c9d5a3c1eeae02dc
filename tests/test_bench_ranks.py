"""The multi-rank path of bench.py on CPU: gloo, world size 2.

Every rank runs its own replica of the workload (the path has no data
exchange), the timed region is the slowest rank's, and the job's value sums
every rank's bytes over that time.  The reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.reduce_time_max(torch, dist, 10.0 + 5.0 * rank, torch.device("cpu"))
        out[rank] = (ms, bench.whole_job_gbs(1_000_000, 100, world, ms))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_whole_job_value_gloo_world2():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        procs = [mp.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    # both ranks see the slower rank's 15 ms; value = 2 ranks x 100 steps x 1 MB / 15 ms
    for r in (0, 1):
        ms, gbs = res[r]
        assert ms == 15.0
        assert gbs == pytest.approx(2 * 100 * 1e6 / 15e-3 / 1e9)


def test_single_rank_time_is_unchanged():
    import bench
    assert bench.reduce_time_max(None, None, 3.5, None) == 3.5
    assert bench.whole_job_gbs(113_836_032, 1000, 1, 37.4) == pytest.approx(
        113_836_032 * 1000 / 37.4e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
