"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every spin inside the library's kernels is bounded.  The test hook
dflash_debug_block_attn_wait_timeout runs the block attention's split-merge
kernel alone, over per-pair counters that nothing increments, with its wait
cut to a few milliseconds: every wait must run out, raise DEV_TIMEOUT in the
device status word and return without writing the output.  The stream and
the context stay usable: the next block attention on the same stream matches
the oracle and leaves the status word clear.
"""
import time

import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_a_bounded_wait_that_runs_out_reports_and_the_stream_stays_usable():
    seq, cap, bs = [300, 1500, 0], 2048, 8
    B = len(seq)
    g = torch.Generator().manual_seed(17)
    k = torch.randn(1, B, 8, cap, 128, generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn(1, B, 8, cap, 128, generator=g).to(torch.bfloat16).to(DEV)
    q = torch.randn(B, 32, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    kb = torch.randn(B, 8, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    vb = torch.randn(B, 8, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    cache = dfl.KVCache(k, v, torch.tensor(seq, dtype=torch.int32, device=DEV))
    stream = torch.cuda.Stream(device=DEV)
    out = torch.full_like(q, 3.0)
    dfl.read_device_status(stream)
    t0 = time.perf_counter()
    dfl.debug_block_attn_wait_timeout(cache, bs, 32, limit_us=2000, out=out, stream=stream)
    flags = dfl.read_device_status(stream)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert flags & dfl.DEV_TIMEOUT
    assert elapsed < 1.0, elapsed                   # the 2 ms limit, not the 2 s default
    assert torch.all(out == 3.0)                    # nothing written by a wait that gave up
    # the same stream, straight after: a normal call is correct and raises nothing
    out2 = dfl.block_attn(0, q, kb, vb, None, None, cache, stream=stream)
    stream.synchronize()
    assert dfl.read_device_status(stream) == 0
    ref = oracle.block_attn(np64(q), np64(kb), np64(vb), np.ones(128), np.ones(128), np64(k[0]), np64(v[0]),
                            np.asarray(seq), bf16=True)
    assert_close(out2, ref, torch.bfloat16, row=128, what="out after the timeout")
