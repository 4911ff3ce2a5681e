"""GPU parity of dflash_fuse_context against the oracle.

Checks the fused context H_t (h_t_out) and every cache row the call writes,
with relative Frobenius error <= 2e-3 (bf16) / 1e-5 (fp32); rows the call must
not touch keep their sentinel values.  Large prefill chunks are checked on a
seeded sample of rows (fusion is row-independent).
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
import workloads
from helpers import TOL, max_abs, np64, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(cfg, n_new, seq_len, cap, layers, seed=0, rows_check=None, sentinel=7.0):
    dt = cfg.dtype
    M = int(sum(n_new))
    w = workloads.weights(cfg, DEV)
    if layers != cfg.L:
        w.w_kv = w.w_kv[: layers * 2 * cfg.Hkv * cfg.d].contiguous()
        w.k_gain = w.k_gain[:layers].contiguous()
    taps = workloads.taps(cfg, M, DEV, seed_offset=seed)
    B = len(n_new)
    k = torch.full((layers, B, cfg.Hkv, cap, cfg.d), sentinel, dtype=dt, device=DEV)
    v = torch.full_like(k, sentinel)
    seq = torch.tensor(seq_len, dtype=torch.int32, device=DEV)
    cu = workloads.cu_rows(n_new, DEV)
    ht = torch.empty(M, cfg.D, dtype=dt, device=DEV)
    cache = dfl.KVCache(k, v, seq)
    dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain, cache, h_t_out=ht)
    torch.cuda.synchronize()
    # oracle on the checked rows
    pos = np.concatenate([seq_len[b] + np.arange(n_new[b]) for b in range(B)]).astype(np.int64)
    seq_of = np.concatenate([np.full(n_new[b], b) for b in range(B)]).astype(np.int64)
    rows = np.arange(M) if rows_check is None else np.asarray(rows_check)
    H, K, V = oracle.fuse_rows([np64(t[rows]) for t in taps], np64(w.w_fuse), np64(w.g_fuse), np64(w.w_kv),
                               np64(w.k_gain), pos[rows], layers, cfg.Hkv, cfg.d, bf16=(dt == torch.bfloat16))
    tol = TOL[dt]
    assert rel_fro(ht[rows], H) <= tol, ("H_t", rel_fro(ht[rows], H), max_abs(ht[rows], H))
    kc = k[:, seq_of[rows], :, pos[rows]]        # advanced indices move to the front: [rows, L, Hkv, d]
    vc = v[:, seq_of[rows], :, pos[rows]]
    assert rel_fro(kc, K) <= tol, ("K", rel_fro(kc, K), max_abs(kc, K))
    assert rel_fro(vc, V) <= tol, ("V", rel_fro(vc, V), max_abs(vc, V))
    return k, v, pos, seq_of


def test_fuse_fp32_tiny_case():
    cfg = workloads.TINY_FP32
    k, v, pos, seq_of = _run(cfg, [64], [0], cfg.capacity, layers=1)
    assert torch.all(k[:, :, :, 64:] == 7.0) and torch.all(v[:, :, :, 64:] == 7.0)


def test_fuse_bf16_ragged_with_empty_sequence():
    cfg = workloads.SINGLE_STREAM
    n_new, seq_len, cap = [100, 0, 200], [5, 10, 0], 256
    k, v, pos, seq_of = _run(cfg, n_new, seq_len, cap, layers=2)
    written = torch.zeros(3, cap, dtype=torch.bool)
    written[0, 5:105] = True
    written[2, 0:200] = True
    untouched = ~written
    kk = k.float().cpu().permute(1, 3, 0, 2, 4)   # [B, cap, L, Hkv, d]
    assert torch.all(kk[untouched] == 7.0)


def test_fuse_bf16_cycle_batched():
    cfg = workloads.BATCHED
    seq = workloads.seq_lens(cfg).tolist()
    _run(cfg, [cfg.bs] * cfg.B, seq, cfg.capacity, layers=cfg.L)


def test_fuse_bf16_cycle_single_sequence():
    cfg = workloads.SINGLE_STREAM
    _run(cfg, [cfg.bs], [cfg.S], cfg.capacity, layers=cfg.L)


def test_fuse_bf16_prefill_chunk_sampled():
    cfg = workloads.SINGLE_STREAM
    rows = np.sort(np.random.default_rng(0).choice(2048, 48, replace=False))
    _run(cfg, [2048], [0], cfg.capacity, layers=cfg.L, rows_check=rows)


def test_fuse_bf16_long_context_chunk_sampled():
    cfg = workloads.LONG_CONTEXT
    rows = np.sort(np.random.default_rng(1).choice(4 * 2048, 64, replace=False))
    _run(cfg, [2048] * 4, [4096] * 4, 8192, layers=2, rows_check=rows)


def test_fuse_capacity_overflow_is_flagged_and_skipped():
    cfg = workloads.SINGLE_STREAM
    dt = cfg.dtype
    w = workloads.weights(cfg, DEV)
    taps = workloads.taps(cfg, 16, DEV)
    cap = 64
    k = torch.full((cfg.L, 2, cfg.Hkv, cap, cfg.d), 7.0, dtype=dt, device=DEV)
    v = torch.full_like(k, 7.0)
    seq = torch.tensor([10, cap - 3], dtype=torch.int32, device=DEV)   # sequence 1 overflows
    dfl.read_device_status()
    dfl.fuse_context(taps, workloads.cu_rows([8, 8], DEV), w.w_fuse, w.g_fuse, w.w_kv, w.k_gain,
                     dfl.KVCache(k, v, seq))
    assert dfl.read_device_status() & dfl.DEV_CAPACITY
    assert torch.all(k[:, 1] == 7.0) and torch.all(v[:, 1] == 7.0)
    assert not torch.all(k[:, 0, :, 10:18] == 7.0)
