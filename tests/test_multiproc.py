"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The decode path shards by sequence with no exchange step, so N GPUs run N
independent replicas: the only cross-rank operations are the barrier around
the timed region and the max over ranks of the elapsed time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    bench.barrier(ws)
    slowest = bench.allmax(10.0 + 5.0 * rank, ws)              # rank 1 is slower
    value = bench.replica_throughput(ws, 8 * 100, slowest)
    bench.barrier(ws)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_replicas_barrier_and_max_over_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 800 / 0.015)


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "qwen32b-shaped-b8-p8192"
        layers = 0
        steps = 1
        warmup = 0
    assert bench.run_reference(A()) == 0
