"""bench.py's multi-rank host logic on CPU with the gloo backend (world size 2).

Each rank runs its own replica of the workload; the bench meets the ranks on
a barrier and reduces their times with a max (the slowest rank sets the job
time) and their work with a sum.  No GPU is involved here.
"""
from __future__ import annotations

import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank: int, world: int, port: int, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_barrier(w)
    mx = bench.dist_max(float(rank + 1) * 1.5, w)
    sm = bench.dist_sum(float(rank + 1), w)
    # the reference arm runs on rank 0 only; the other ranks return at once
    ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), r, w) if r != 0 else "skip"
    import torch.distributed as dist
    dist.destroy_process_group()
    results[rank] = (mx, sm, ref)


def test_two_rank_reductions():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    for rank in range(world):
        mx, sm, ref = results[rank]
        assert mx == 3.0          # the slowest rank's time
        assert sm == 3.0          # 1 + 2: work adds up over replicas
    assert results[1][2] is None  # non-zero ranks print nothing


def test_aggregate_throughput_formula():
    import bench
    import workloads as wl
    # replicas: value = world x per-rank work / slowest rank's time
    flops = bench.prefill_flops(wl.PREFILL_FULL_4B_B2_T8192)
    assert abs(flops - 1.0996e12) / 1.0996e12 < 1e-4
    total, full = bench.decode_kv_bytes(bench.decode_layers(36))
    assert full == 1048576 * 4096
    assert total == 9 * 1048576 * 4096 + 27 * 512 * 4096
    assert bench.visible_pairs(1024, wl.SLIDING, 512) == 393472
    assert bench.visible_pairs(65536, wl.SLIDING, 512) == 33423616
    assert bench.visible_pairs(65536, wl.FULL, 0) == 2147516416
