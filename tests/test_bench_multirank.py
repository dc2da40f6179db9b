"""bench.py's multi-rank host logic on CPU with the gloo backend (world size 2): replicas time
their own steps, the slowest rank's time sets the job's, every rank sees it, and the job's
throughput counts every rank's tokens. The reference arm runs on rank 0 alone."""
import os
import socket
import types

import torch.multiprocessing as mp

import bench
from moe_inputs import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + r ms for the timed steps and 20 - r ms end to end
        q.put((rank, bench.slowest_rank_ms([10.0 + rank, 20.0 - rank], dist)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the element-wise maximum over ranks
    assert got[0] == [11.0, 20.0] and got[1] == [11.0, 20.0]


def test_whole_job_rate_counts_every_rank():
    # 2 replicas x 4096 tokens x 30 steps in the slowest rank's 60 ms
    assert bench.whole_job_rate(4096, 30, 2, 60.0) == 2 * 4096 * 30 / 0.060
    assert bench.whole_job_rate(4096, 30, 1, 60.0) == 4096 * 30 / 0.060


def test_single_process_reduction_is_identity():
    assert bench.slowest_rank_ms([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = types.SimpleNamespace(steps=1, warmup=3, gpus=2)
    assert bench.run_reference(args, WORKLOADS["tiny_fp32"], rank=1) is None
    assert capsys.readouterr().out == ""
