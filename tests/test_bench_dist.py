"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1) run the
max-over-ranks reduction of the step times and the whole-job throughput the
bench reports under torchrun (replicas, weak scaling)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)])
        env = bench.dist_env()
        value = bench.whole_job_tflops(3.0e12, env[0], times[0])
        queue.put((rank, times, env, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, env, value in results:
        assert times == [2.0, 5.0, 0.5]                  # element-wise max over the ranks
        assert env == (2, rank, rank)
        assert abs(value - 2 * 3.0e12 / 2.0e-3 / 1e12) < 1e-9   # both ranks' work / slowest time


def test_single_process_is_the_identity():
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
    assert abs(bench.whole_job_tflops(1.0e12, 1, 1.0) - 1000.0) < 1e-9
