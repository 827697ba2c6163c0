"""The benchmark's multi-rank logic on CPU with the gloo backend, world size
2: the timed region's barrier and max-over-ranks reduction, the replica
aggregation of the headline value, and the reference arm running on rank 0
only. (The path itself has no cross-GPU exchange: every rank runs its own
problem.)"""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init("gloo")
    bench.barrier()
    local_ms = 10.0 * (rank + 1)
    ms = bench.reduce_max(local_ms)
    flop, steps = 2.0 * 8192 ** 3, 5
    value = flop * steps * world / (ms * 1e-3) / 1e12
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_replica_value():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]            # both ranks see the slowest time
    expect = 2.0 * 8192 ** 3 * 5 * 2 / 0.020 / 1e12
    assert all(abs(r[2] - expect) < 1e-6 * expect for r in res)


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
