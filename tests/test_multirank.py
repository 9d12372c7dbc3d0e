"""The N > 1 path of bench.py on CPU: two gloo ranks, timing reductions only
(every rank is an independent replica; there is no data-path collective)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        mx = bench.max_over_ranks(10.0 * (rank + 1), ws)
        sm = bench.sum_over_ranks(100.0 + rank, ws)
        # the reference arm runs on rank 0 only
        class A:  # minimal args
            steps, warmup, config, batch = 1, 0, "tiny", None
        ref = bench.run_reference(A, rank, ws) if rank else None
        q.put((rank, mx, sm, ref))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm, ref in res:
        assert mx == 20.0 and sm == 201.0
        assert ref is None
