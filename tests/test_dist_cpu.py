"""The multi-GPU bench path on CPU: two gloo ranks agree on the max-over-ranks
time and decode independent (distinctly seeded) batches (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import sfi_workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    v = bench.aggregate_max(1.5 * (rank + 1), world)
    seed = bench.rank_seed(W.MASTER_SEED, rank)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, v, seed))


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [3.0, 3.0]
    assert res[0][2] == W.MASTER_SEED and res[1][2] != res[0][2]


def test_attention_bytes_counts_rows():
    wl = W.cfg2(n_layers=1, n_steps=3)
    import numpy as np
    import bench
    masks = np.array([[1] * 8, [0] * 8, [0] * 8], np.uint8)
    row = 2 * 8 * 128 * 2
    exp = 8 * (131072 * row + (4 + 4096 + 256) * row * 2)
    assert bench.attention_bytes(wl, masks) == exp
