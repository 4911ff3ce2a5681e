"""dflash_verify_noalloc: verification for callers that cannot allocate.

Callers inside a CUDA graph capture, or with an allocator that forbids late
allocation, cannot hand dflash_verify a fresh workspace; this entry point uses
the library's static device scratch instead.  Its results must equal
dflash_verify's (both are deterministic) on two calls in a row, and after a
larger call whose leftovers in the shared scratch have other strides.  Runs last (file name) and also passes alone in a fresh process.
"""
import ctypes
from dataclasses import replace

import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(lt, ld, x, T, seed, cycle):
    B, bs, V = lt.shape
    acc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    out = torch.full((B, bs), -7, dtype=torch.int32, device=DEV)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    code = dfl.lib().dflash_verify_noalloc(P(lt), P(ld), dfl.BF16 if lt.dtype == torch.bfloat16 else dfl.F32,
                                           P(x), B, bs, V, float(T), seed, cycle, P(acc), P(out),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, dfl.lib().dflash_last_error_string()
    return acc, out


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_verify_matches_workspace_verify_twice(T):
    cfg = workloads.BATCHED
    lt, ld = workloads.logits(cfg, DEV)
    x = workloads.draft_tokens(ld, T, seed=31)
    assert dfl.verify_workspace_size(cfg.B, cfg.bs, cfg.V, dfl.BF16) <= dfl.lib().dflash_verify_noalloc_max_scratch()
    for cycle in (5, 6):
        ref_acc, ref_out = dfl.verify(lt, ld, x, T, 99, cycle)
        acc, out = _noalloc(lt, ld, x, T, 99, cycle)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc) and torch.equal(out, ref_out)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_verify_after_a_larger_call(T):
    """A large call (128 sequences, V = 262144) leaves its partial sums all
    over the shared scratch; a following smaller call with other strides
    (5 sequences, block 16, V = 40000) must still equal dflash_verify with a
    fresh workspace, and so must a third, larger call again."""
    big = workloads.high_batch(8, 1.0)
    small = replace(workloads.high_batch(16, 1.0), B=5, V=40000, seed=77)
    for cfg, cycle in ((big, 3), (small, 4), (workloads.BATCHED, 5)):
        lt, ld = workloads.logits(cfg, DEV)
        x = workloads.draft_tokens(ld, T, seed=cycle)
        acc, out = _noalloc(lt, ld, x, T, 123, cycle)
        ref_acc, ref_out = dfl.verify(lt, ld, x, T, 123, cycle)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc) and torch.equal(out, ref_out), cfg.name


def test_noalloc_verify_rejects_oversized_problems():
    big_b = 4096
    assert dfl.verify_workspace_size(big_b, 16, 262144, dfl.BF16) > dfl.lib().dflash_verify_noalloc_max_scratch()
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    P = ctypes.c_void_p(dummy.data_ptr())
    code = dfl.lib().dflash_verify_noalloc(P, P, dfl.BF16, P, big_b, 16, 262144, 1.0, 0, 0, P, P, None)
    assert code == 2 and b"scratch" in dfl.lib().dflash_last_error_string()
