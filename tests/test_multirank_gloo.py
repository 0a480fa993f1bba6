"""N>1 host logic of bench.py on CPU with the gloo backend (world size 2).

Sampling shards by rows with no data-path collective: rank r samples its own
batch of global rows [r*B, (r+1)*B); the only collectives are the timing
barrier and the max-over-ranks reduction of the elapsed time.
"""
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import bench
    import oracle
    from device_logits_sampling_gb300 import workloads

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, rk, local = bench.dist_setup()
    w = workloads.mixed_batch(B=8, V=2048)
    rows = list(bench.rows_of_shard(w.B, ws, rk))
    p = w.params.copy()
    p["seed"] = np.array(rows, dtype=np.uint64)
    res = oracle.sample_batch(w.logits_f32(), p)
    toks = [r.token for r in res]
    elapsed = torch.tensor([0.5 + rank])
    dist.barrier()
    dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
    q.put((rank, rows, toks, float(elapsed.item())))
    dist.destroy_process_group()


def test_two_ranks_shard_rows_and_reduce_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    (r0, rows0, tok0, t0), (r1, rows1, tok1, t1) = out
    assert rows0 == list(range(0, 8)) and rows1 == list(range(8, 16))
    assert t0 == t1 == 1.5  # max over ranks
    # greedy rows (row % 4 == 0) agree, sampled rows see different seeds
    assert tok0[0] == tok1[0] and tok0[4] == tok1[4]
    assert tok0 != tok1
