"""Multi-rank logic of bench.py on CPU: two gloo ranks, as torchrun would
launch them, run the same barrier / max-over-ranks / whole-job-rate code the
GPU bench uses. The path shards by sequence with no exchange, so a replica
per rank plus this reduction of the timings is all the multi-GPU bench does."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world), FDL_BENCH_BACKEND="gloo")
    import bench
    w, r, local = bench.dist_init()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # rank r "took" 10 + 5r ms for its steps; the job takes the slowest
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    rate = bench.whole_job_rate(64, 100, ms, w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms} {rate}")
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [tuple(map(float, (tmp_path / f"rank{r}.txt").read_text().split())) for r in range(world)]
    slowest = 10.0 + 5.0 * (world - 1)
    for ms, rate in got:
        assert ms == pytest.approx(slowest)
        # both ranks' 64 x 100 rows over the slowest rank's 15 ms
        assert rate == pytest.approx(world * 64 * 100 / (slowest * 1e-3))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(64, 10, 2.0, 1) == pytest.approx(64 * 10 / 2e-3)
