"""Host logic of the multi-rank benchmark, run as two gloo ranks on CPU.

Sequences are independent, so ranks shard the job by running their own
batches: the only cross-rank traffic is the reduction of the timing (max) and
of the token count (sum).  No GPU and no kernel is involved here.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, lr = bench.env_rank()
        elapsed = 1.0 + rank          # rank 1 is the slow one
        tokens = 10.0 * (rank + 1)
        el, tok = bench.reduce_max_sum(elapsed, tokens, torch.device("cpu"))
        cfg = bench.rank_config(rank)
        q.put((rank, r, w, lr, el, tok, cfg.seed, cfg.B, cfg.bs, cfg.L))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_by_max_and_tokens_by_sum():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, (r, env_r, w, lr, el, tok, seed, B, bs, L) in enumerate(res):
        assert (env_r, w, lr) == (rank, world, rank)
        assert el == 2.0                  # max over ranks
        assert tok == 30.0                # sum over ranks
        assert (B, bs, L) == (32, 8, 5)   # every rank runs the full batched workload (weak scaling)
    seeds = [x[6] for x in res]
    assert len(set(seeds)) == world       # ranks draw different batches


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max_sum(0.5, 7.0, torch.device("cpu")) == (0.5, 7.0)
    c = bench.rank_config(0, batch=4, layers=1)
    assert (c.B, c.L) == (4, 1)
    assert bench.rank_config(0).seed != bench.rank_config(3).seed
