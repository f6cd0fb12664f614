"""The benchmark's multi-GPU mode is N independent replicas (no data-path collective): each rank
draws its own seeded batch, and only the barrier, the max of the step time and the sum of the bytes
cross ranks. Checked here with world_size 2 on the gloo backend (CPU)."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, ROOT)
    bench = load_bench()
    d = bench.Dist()
    from paged_kv_flash_cache_gb300 import workloads as W
    # each rank's replica: its own seeded context lengths (tables only, no token data)
    gen = torch.Generator().manual_seed(1236 + 100 * rank)
    lens = torch.randint(1024, 8193, (16,), generator=gen)
    kv_bytes = float(lens.sum()) * 32 * 128 * 2 * 2
    step_ms = 1.0 + rank                  # rank 1 is the slow one
    d.barrier()
    q.put((rank, d.max(step_ms), d.sum(kv_bytes), lens.tolist()))
    d.close()


def test_replicas_max_time_sum_bytes_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, mx0, sum0, lens0), (_, mx1, sum1, lens1) = res
    assert mx0 == mx1 == 2.0                         # both ranks report the slowest rank's time
    expect = (sum(lens0) + sum(lens1)) * 32 * 128 * 4
    assert sum0 == sum1 == pytest.approx(expect)     # whole-job bytes
    assert lens0 != lens1                            # independent replicas, different batches
