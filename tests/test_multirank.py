"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

One process per GPU runs an independent replica of the workload (weak
scaling, no collective on the data path); what crosses ranks is the barrier
around the timed region, the maximum of the ranks' times, and the whole-job
rate built from it.  No GPU is involved.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_info()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(w)
        t_max = bench.barrier_max(times[rank], w, "cpu")
        rate = bench.job_rate(1000.0, w, t_max)
        seed = bench.shard_seed(7, rank)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as fh:
            fh.write(f"{t_max} {rate} {seed}\n")
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_take_the_slowest_time_and_sum_the_work(tmp_path):
    times = [0.5, 2.0]
    mp.spawn(_rank_main, args=(2, _free_port(), times, str(tmp_path)), nprocs=2, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(2)]
    for t_max, rate, _ in rows:
        assert float(t_max) == 2.0                 # max over ranks, seen by both
        assert float(rate) == 2 * 1000.0 / 2.0     # all ranks' units / slowest time
    seeds = {int(s) for _, _, s in rows}
    assert len(seeds) == 2 and 7 in seeds          # independent problems; rank 0 unchanged


def test_single_rank_needs_no_process_group():
    assert bench.barrier_max(1.25, 1, "cpu") == 1.25
    bench.barrier(1)
    assert bench.job_rate(10.0, 1, 2.0) == 5.0
    assert bench.shard_seed(3, 0) == 3
