"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1), each
timing its own replica of the workload; rank 0 reports the maximum time over
ranks and the whole-job throughput (weak scaling, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(w)
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        worst = bench.max_over_ranks(local_ms, w, torch.device("cpu"))
        tokens_per_rank = 1000
        value = w * tokens_per_rank / (worst / 1000.0)
        # each rank draws its own independent batch
        from chunked_gated_delta_gdn_gb300 import synthetic
        inp = synthetic.workload("tiny_fp32", seed=1005 + 1000 * rank)
        digest = float(inp.q.double().sum())
        gathered = [torch.zeros(1, dtype=torch.float64) for _ in range(w)]
        dist.all_gather(gathered, torch.tensor([digest], dtype=torch.float64))
        q.put((rank, worst, value, [float(x) for x in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0, "rank exited with %s" % p.exitcode
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, worst, value, digests in res:
        assert worst == pytest.approx(15.0)                  # max over ranks
        assert value == pytest.approx(2 * 1000 / 0.015)      # whole-job tokens / max time
        assert digests[0] != digests[1]                      # independent batches per rank
