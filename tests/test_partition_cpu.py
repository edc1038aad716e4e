"""The column partition (multi-worker path) on CPU: two gloo ranks each compute a
column slab of C with the oracle; the stitched slabs equal the whole product bit
for bit.  No GPU and no collective on the data path beyond gathering results."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from precision_gemm_gb300.partition import column_slabs, even_slabs, slab_views


def test_slabs_cover_columns_exactly():
    for n in (0, 1, 7, 100, 1500, 8191):
        for w in ([1], [1, 1], [15, 1], [3, 0, 2], [1] * 7):
            s = column_slabs(n, w)
            assert s[0][0] == 0 and s[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(s, s[1:]))
            assert all(j0 <= j1 for j0, j1 in s)
    # the lecture's Q = 15 split of 100 columns: integer formulas give 93 + 6 = 99
    assert column_slabs(100, [15, 1]) == [(0, 94), (94, 100)]
    assert even_slabs(10, 3) == [(0, 3), (3, 7), (7, 10)]
    with pytest.raises(ValueError):
        column_slabs(10, [0, 0])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from precision_gemm_gb300 import synth
        p = synth.Problem(61, 53, 37, lda=64, ldb=40, ldc=67, alpha=1.5, beta=-0.5, dist="normal", seed=3)
        A, B, C = synth.make(p)
        A, B, C = A.numpy(), B.numpy(), C.numpy()
        j0, j1 = even_slabs(p.n, world)[rank]
        b_off, c_off, width = slab_views(j0, j1, p.ldb, p.ldc)
        cref, _ = oracle.Oracle().full("N", "N", p.m, width, p.k, p.alpha, A, p.lda, B[b_off:], p.ldb, p.beta,
                                       C[c_off:], p.ldc, threads=1)
        slab = torch.from_numpy(np.ascontiguousarray(cref.T))  # (width, m)
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([width], dtype=torch.int64))
        maxw = int(max(s.item() for s in sizes))
        padded = torch.zeros((maxw, p.m), dtype=torch.float64)
        padded[:width] = slab
        gathered = [torch.zeros_like(padded) for _ in range(world)]
        dist.all_gather(gathered, padded)
        if rank == 0:
            stitched = torch.cat([g[: int(s.item())] for g, s in zip(gathered, sizes)]).numpy().T
            whole, _ = oracle.Oracle().full("N", "N", p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc,
                                            threads=1)
            q.put(bool(np.array_equal(stitched, whole)))
    finally:
        dist.destroy_process_group()


def test_two_rank_column_split_matches_whole_product():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_worker, args=(2, _free_port(), q), nprocs=2, join=True, start_method="spawn")
    assert q.get() is True
