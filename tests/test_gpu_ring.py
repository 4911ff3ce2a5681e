"""Sliding-window draft cache kept as a ring of W rows.

Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash" -- the
released drafter attends to its latest 1024 tokens.  A ring cache of W rows
(position p in row p % W) must hold exactly the rows a linear cache holds for
its latest W positions, and block attention over the ring must equal block
attention over the linear cache with window = W (attention is a sum over keys,
so the rows' order in the ring does not matter).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
import workloads
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _filled_caches(W, steps, seed):
    cfg = replace(workloads.SINGLE_STREAM, name="ring", B=len(steps[0]), S=0, L=2, D=256, d_target=256,
                  seed=seed)
    w = workloads.weights(cfg, DEV)
    lin_cap = ((sum(max(s) for s in steps) + 63) // 64) * 64
    kl = torch.zeros(cfg.L, cfg.B, cfg.Hkv, lin_cap, 128, dtype=torch.bfloat16, device=DEV)
    kr = torch.zeros(cfg.L, cfg.B, cfg.Hkv, W, 128, dtype=torch.bfloat16, device=DEV)
    seq = torch.zeros(cfg.B, dtype=torch.int32, device=DEV)
    lin = dfl.KVCache(kl, torch.zeros_like(kl), seq)
    ring = dfl.KVCache(kr, torch.zeros_like(kr), seq, ring=True)
    for i, n_new in enumerate(steps):
        taps = workloads.taps(cfg, sum(n_new), DEV, seed_offset=i)
        cu = workloads.cu_rows(n_new, DEV)
        for cache in (lin, ring):
            dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain, cache)
        seq += torch.tensor(n_new, dtype=torch.int32, device=DEV)   # the caller advances the lengths
    assert dfl.read_device_status() == 0
    return cfg, w, lin, ring


def test_ring_rows_equal_the_latest_linear_rows():
    W = 256
    steps = [[150, 90, 256], [150, 200, 1], [150, 5, 256], [150, 256, 0], [120, 0, 3]]
    cfg, w, lin, ring = _filled_caches(W, steps, seed=21)
    n = lin.seq_len.cpu().tolist()
    for b in range(cfg.B):
        p = torch.arange(max(0, n[b] - W), n[b], device=DEV)
        for got, want in ((ring.k, lin.k), (ring.v, lin.v)):
            assert torch.equal(got[:, b][:, :, p % W], want[:, b][:, :, p]), b   # same bits, rotated rows


@pytest.mark.parametrize("bs", [8, 16])
def test_block_attn_over_a_ring_equals_the_window_of_a_linear_cache(bs):
    W = 256
    steps = [[150, 90, 256], [150, 200, 1], [150, 5, 256], [150, 256, 0], [120, 0, 3]]
    cfg, w, lin, ring = _filled_caches(W, steps, seed=22 + bs)
    cfg = replace(cfg, bs=bs)
    q, kb, vb = workloads.block(cfg, DEV, layer=1)
    out_lin = dfl.block_attn(1, q, kb, vb, w.q_gain[1], w.k_gain[1], lin, window=W)
    out_ring = dfl.block_attn(1, q, kb, vb, w.q_gain[1], w.k_gain[1], ring)
    seq = lin.seq_len.cpu().numpy()
    ref = oracle.block_attn(np64(q), np64(kb), np64(vb), np64(w.q_gain[1]), np64(w.k_gain[1]), np64(lin.k[1]),
                            np64(lin.v[1]), seq, window=W, bf16=True)
    for out in (out_lin, out_ring):
        assert_close(out, ref, torch.bfloat16, row=128, what="out")
    assert_close(out_ring, out_lin.float().cpu().numpy(), 2e-3, row=128, what="ring vs linear")
    assert dfl.read_device_status() == 0


def test_ring_scores_far_above_the_first_tile_take_the_exact_path():
    """A key scoring far above its item's first tile, in a ring whose
    sequences are longer than the ring: the combine kernel redoes the pair key
    by key, with the block at positions seq_len + j (past the ring's
    capacity), and both the ring and the linear window match the oracle."""
    W = 256
    steps = [[150, 90, 256], [150, 200, 1], [150, 5, 256], [150, 256, 0], [120, 0, 3]]
    cfg, w, lin, ring = _filled_caches(W, steps, seed=41)
    n = lin.seq_len.cpu().tolist()
    assert n[0] > W
    p = n[0] - 1                    # latest position: the second key tile of both layouts
    assert p % W >= 128 and p >= n[0] - 128
    g = torch.Generator().manual_seed(42)
    big = (200.0 * torch.randn(128, generator=g)).to(torch.bfloat16).to(DEV)
    lin.k[1, 0, 5, p] = big
    ring.k[1, 0, 5, p % W] = big
    q, kb, vb = workloads.block(cfg, DEV, layer=1)
    dfl.read_device_status()
    out_lin = dfl.block_attn(1, q, kb, vb, w.q_gain[1], w.k_gain[1], lin, window=W)
    out_ring = dfl.block_attn(1, q, kb, vb, w.q_gain[1], w.k_gain[1], ring)
    assert dfl.read_device_status() == 0
    seq = lin.seq_len.cpu().numpy()
    ref = oracle.block_attn(np64(q), np64(kb), np64(vb), np64(w.q_gain[1]), np64(w.k_gain[1]), np64(lin.k[1]),
                            np64(lin.v[1]), seq, window=W, bf16=True)
    for out in (out_lin, out_ring):
        assert torch.isfinite(out.float()).all()
        assert_close(out, ref, torch.bfloat16, row=128, what="out")


def test_ring_fusion_of_more_rows_than_the_ring_is_flagged_and_skipped():
    """One call may add at most W rows to a sequence of a W-row ring; more is
    flagged on the device and that sequence's rows are skipped (the host only
    knows the total)."""
    W = 64
    cfg = replace(workloads.SINGLE_STREAM, name="ring", B=2, S=0, L=1, D=256, d_target=256, seed=30)
    w = workloads.weights(cfg, DEV)
    k = torch.full((1, 2, cfg.Hkv, W, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    ring = dfl.KVCache(k, k.clone(), torch.zeros(2, dtype=torch.int32, device=DEV), ring=True)
    dfl.fuse_context(workloads.taps(cfg, W + 1, DEV), workloads.cu_rows([W + 1, 0], DEV), w.w_fuse, w.g_fuse,
                     w.w_kv, w.k_gain, ring)
    assert dfl.read_device_status() & dfl.DEV_CAPACITY
    assert torch.all(ring.k == 7.0) and torch.all(ring.v == 7.0)
    with pytest.raises(dfl.DFlashError):     # more rows than the whole cache holds: refused on the host
        dfl.fuse_context(workloads.taps(cfg, 2 * W + 1, DEV), workloads.cu_rows([W + 1, W], DEV), w.w_fuse,
                         w.g_fuse, w.w_kv, w.k_gain, ring)
