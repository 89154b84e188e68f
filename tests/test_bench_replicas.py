"""The bench's multi-process path on CPU: two gloo ranks run the host logic that `torchrun
--nproc-per-node N bench.py` runs on N GPUs (process group, barriers, max over ranks of the
timings, whole-job throughput), and the reference arm's non-zero ranks exit without work."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w, cuda=False)
    # each rank "took" a different time; the job's time is the slowest rank's
    ms = 10.0 * (rank + 1)
    ms_max = bench.max_over_ranks(w, ms, device="cpu")
    rate = bench.aggregate_rate(w, 8192, ms_max)
    bench.barrier(w, cuda=False)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms_max} {rate}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_aggregate(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    vals = [tuple(map(float, (tmp_path / f"rank{r}.txt").read_text().split())) for r in range(world)]
    for ms_max, rate in vals:
        assert ms_max == pytest.approx(20.0)                  # max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 8192 / 0.020)       # all ranks' tokens over the slowest time


def test_world_one_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1, 3.5, device="cpu") == 3.5
    assert bench.aggregate_rate(1, 64, 16.0) == pytest.approx(4000.0)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
