"""The vocabulary-parallel exchange across two real processes (gloo, CPU):
each rank computes the oracle's partials of its ceil(V/2) vocabulary slice,
the ranks all-gather them -- the collective of hyper-parallel #269 section
3.1 -- and the combine must equal the unsplit oracle on every row."""
import math
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp


def _rank(rank, world, port, V, out):
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(9)
    N = 12
    x = rng.standard_normal((N, V)) * 3
    y = rng.integers(0, V, N)
    c = -(-V // world)
    k0, k1 = rank * c, min(V, (rank + 1) * c)
    mine = np.stack([oracle.chunk_partials(x[r], k0, k1, int(y[r])) for r in range(N)])
    gathered = [torch.zeros(N, 5, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(mine))
    parts = np.stack([g.numpy() for g in gathered], axis=1)  # (N, world, 5)
    worst = 0.0
    for r in range(N):
        lse, xy, S = oracle.combine(parts[r])
        whole = oracle.chunk_partials(x[r], 0, V, int(y[r]))
        ref = whole[0] + math.log(whole[1])
        worst = max(worst, abs(lse - ref) / abs(ref))
        assert xy == x[r, y[r]]
    out[rank] = worst
    dist.destroy_process_group()


def test_two_rank_vocab_parallel_combine():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(2, port, 1001, out), nprocs=2, join=True)
    assert out[0] <= 1e-13 and out[1] <= 1e-13
