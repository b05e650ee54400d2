"""Multi-GPU host logic (independent replicas) on CPU: two gloo ranks, no GPU.

The layer is data-parallel over tokens; the replicas exchange nothing but the timing
handshake, so the whole N>1 path that does not touch a GPU is exercised here.
"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from fp8_block_scaled_router_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_token_windows_partition_the_stream():
    ntok, world = 10000, 4
    offs = [replicas.token_offset(r, world, ntok) for r in range(world)]
    assert offs == [0, 2500, 5000, 7500]
    with pytest.raises(ValueError):
        replicas.token_offset(4, 4, ntok)


def test_throughput_sums_ranks_over_slowest_time():
    assert replicas.throughput(2, 100, 1, 0.5) == pytest.approx(400.0)
    with pytest.raises(ValueError):
        replicas.throughput(1, 1, 1, 0.0)
    assert replicas.slowest(0.25) == 0.25  # no process group: the local time


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 0.1 * (rank + 1)  # rank 1 is the slow one
        t = replicas.slowest(elapsed, dist)
        q.put((rank, t, replicas.throughput(world, 10, 1, t), replicas.token_offset(rank, world, 10000)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for _, t, v, _ in got:
        assert t == pytest.approx(0.2)        # max over ranks
        assert v == pytest.approx(2 * 10 / 0.2)
    assert [g[3] for g in got] == [0, 5000]   # disjoint token windows


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
