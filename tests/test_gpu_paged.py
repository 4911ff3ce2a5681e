"""GPU parity of the paged cache layout (block table) against the linear one.

The paged layout changes only where rows live, so for the same inputs:
  * fusion writes, through the block table, exactly the rows the linear layout
    gets (bit for bit), touches no page the table does not name, and matches
    the oracle on the rows it writes (through oracle.gather_pages);
  * attention over a paged pool gives the linear layout's output bit for bit,
    never reading pages past a sequence's length (their table entries are -1,
    unreferenced pages hold NaN) and matches the oracle;
  * a block-table entry outside the pool that a new row needs raises
    DFLASH_DEV_BAD_SEQLEN and the row is skipped.
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
import workloads
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
BAD_SEQLEN = 4


def _table(B, MP, NP, used_rows, P, seed):
    """Distinct random pages; entries past each sequence's used rows are -1."""
    rng = np.random.default_rng(seed)
    t = rng.permutation(NP)[: B * MP].reshape(B, MP).astype(np.int32)
    for b, n in enumerate(used_rows):
        t[b, (n + P - 1) // P:] = -1
    return t


def _to_pool(lin, table, NP, fill):
    """Pool [L, NP, H, P, d] holding the linear cache's pages where the table says."""
    L, B, H, cap, d = lin.shape
    P = cap // table.shape[1]
    pool = torch.full((L, NP, H, P, d), fill, dtype=lin.dtype, device=lin.device)
    for b in range(B):
        for j in range(table.shape[1]):
            if table[b, j] >= 0:
                pool[:, int(table[b, j])] = lin[:, b, :, j * P:(j + 1) * P]
    return pool


def _fuse_both(n_new, seq_len, P, MP, NP, layers, seed, sentinel=7.0):
    cfg = workloads.BATCHED
    M, B, cap = int(sum(n_new)), len(n_new), MP * P
    w = workloads.weights(cfg, DEV)
    w.w_kv = w.w_kv[: layers * 2 * cfg.Hkv * cfg.d].contiguous()
    w.k_gain = w.k_gain[:layers].contiguous()
    taps = workloads.taps(cfg, M, DEV, seed_offset=seed)
    cu = workloads.cu_rows(n_new, DEV)
    seq = torch.tensor(seq_len, dtype=torch.int32, device=DEV)
    used = [s + n for s, n in zip(seq_len, n_new)]
    table = _table(B, MP, NP, used, P, seed)
    kl = torch.full((layers, B, cfg.Hkv, cap, cfg.d), sentinel, dtype=torch.bfloat16, device=DEV)
    vl = torch.full_like(kl, sentinel)
    kp = torch.full((layers, NP, cfg.Hkv, P, cfg.d), sentinel, dtype=torch.bfloat16, device=DEV)
    vp = torch.full_like(kp, sentinel)
    dfl.read_device_status()
    dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain, dfl.KVCache(kl, vl, seq))
    dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain,
                     dfl.KVCache(kp, vp, seq, block_table=torch.as_tensor(table, device=DEV)))
    torch.cuda.synchronize()
    assert dfl.read_device_status() == 0
    return cfg, w, taps, table, kl, vl, kp, vp, used


@pytest.mark.parametrize("case", ["cycle_accepted_rows", "prefill_fused_epilogue"])
def test_paged_fusion_writes_the_linear_rows(case):
    if case == "cycle_accepted_rows":   # ragged n+1 accepted rows per sequence, M <= 256
        n_new, seq_len, P, MP, NP = [3, 8, 1, 6], [300, 0, 129, 1000], 128, 9, 40
    else:                               # M > 256: the K/V epilogue fused into the GEMM
        n_new, seq_len, P, MP, NP = [300, 200], [0, 100], 256, 2, 7
    layers = 2
    cfg, w, taps, table, kl, vl, kp, vp, used = _fuse_both(n_new, seq_len, P, MP, NP, layers, seed=5)
    kg = torch.as_tensor(oracle.gather_pages(kp.float().cpu().numpy(), table, P))
    vg = torch.as_tensor(oracle.gather_pages(vp.float().cpu().numpy(), table, P))
    for b, n in enumerate(used):
        assert torch.equal(kg[:, b, :, :n], kl[:, b, :, :n].float().cpu()), b
        assert torch.equal(vg[:, b, :, :n], vl[:, b, :, :n].float().cpu()), b
    referenced = set(int(x) for x in table.reshape(-1) if x >= 0)
    for pg in range(NP):
        if pg not in referenced:
            assert torch.all(kp[:, pg] == 7.0) and torch.all(vp[:, pg] == 7.0), pg
    # the written rows against the oracle
    pos = np.concatenate([seq_len[b] + np.arange(n_new[b]) for b in range(len(n_new))]).astype(np.int64)
    seq_of = np.concatenate([np.full(n_new[b], b) for b in range(len(n_new))]).astype(np.int64)
    _, K, V = oracle.fuse_rows([np64(t) for t in taps], np64(w.w_fuse), np64(w.g_fuse), np64(w.w_kv),
                               np64(w.k_gain), pos, layers, cfg.Hkv, cfg.d, bf16=True)
    kc, vc = kg[:, seq_of, :, pos], vg[:, seq_of, :, pos]
    assert_close(kc, K, torch.bfloat16, row=cfg.d, what="K")
    assert_close(vc, V, torch.bfloat16, row=cfg.d, what="V")


def _attn_both(seq, P, MP, NP, bs, seed, layers=2, layer=1):
    B, cap = len(seq), MP * P
    g = torch.Generator().manual_seed(seed)
    kl = torch.randn(layers, B, 8, cap, 128, generator=g).to(torch.bfloat16).to(DEV)
    vl = torch.randn(layers, B, 8, cap, 128, generator=g).to(torch.bfloat16).to(DEV)
    q = torch.randn(B, 32, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    kb = torch.randn(B, 8, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    vb = torch.randn(B, 8, bs, 128, generator=g).to(torch.bfloat16).to(DEV)
    qg = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16).to(DEV)
    kgn = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16).to(DEV)
    table = _table(B, MP, NP, seq, P, seed)
    kp = _to_pool(kl, table, NP, float("nan"))
    vp = _to_pool(vl, table, NP, float("nan"))
    seq_t = torch.tensor(seq, dtype=torch.int32, device=DEV)
    dfl.read_device_status()
    out_l = dfl.block_attn(layer, q, kb, vb, qg, kgn, dfl.KVCache(kl, vl, seq_t))
    out_p = dfl.block_attn(layer, q, kb, vb, qg, kgn,
                           dfl.KVCache(kp, vp, seq_t, block_table=torch.as_tensor(table, device=DEV)))
    torch.cuda.synchronize()
    assert dfl.read_device_status() == 0
    return out_l, out_p, (q, kb, vb, qg, kgn, kl[layer], vl[layer])


@pytest.mark.parametrize("bs", [4, 8, 16])
def test_paged_attention_is_the_linear_attention(bs):
    seq = [0, 1, 128, 700, 3000]
    out_l, out_p, (q, kb, vb, qg, kgn, kl, vl) = _attn_both(seq, P=256, MP=12, NP=64, bs=bs, seed=bs)
    assert torch.equal(out_p, out_l)
    ref = oracle.block_attn(np64(q), np64(kb), np64(vb), np64(qg), np64(kgn), np64(kl), np64(vl),
                            np.asarray(seq), bf16=True)
    assert_close(out_p, ref, torch.bfloat16, row=128, what="out")


def test_paged_attention_batched_lengths():
    """32 sequences of 1024..8192 cached positions in 128-row pages (many key
    splits per sequence, splits spanning pages), bit for bit against linear."""
    rng = np.random.default_rng(9)
    seq = rng.integers(1024, 8193, size=32).tolist()
    out_l, out_p, _ = _attn_both(seq, P=128, MP=64, NP=32 * 64 + 16, bs=8, seed=9, layers=1, layer=0)
    assert torch.equal(out_p, out_l)


def test_paged_fusion_flags_a_table_entry_outside_the_pool():
    cfg = workloads.BATCHED
    n_new, seq_len, P, MP, NP, layers = [4, 4], [126, 0], 128, 2, 6, 1
    M, B = sum(n_new), len(n_new)
    w = workloads.weights(cfg, DEV)
    w.w_kv = w.w_kv[: layers * 2 * cfg.Hkv * cfg.d].contiguous()
    w.k_gain = w.k_gain[:layers].contiguous()
    taps = workloads.taps(cfg, M, DEV)
    table = np.array([[0, NP + 3], [1, -1]], dtype=np.int32)   # sequence 0's rows 128, 129 need page 1 of 2
    kp = torch.full((layers, NP, cfg.Hkv, P, cfg.d), 7.0, dtype=torch.bfloat16, device=DEV)
    vp = torch.full_like(kp, 7.0)
    seq = torch.tensor(seq_len, dtype=torch.int32, device=DEV)
    dfl.read_device_status()
    dfl.fuse_context(taps, workloads.cu_rows(n_new, DEV), w.w_fuse, w.g_fuse, w.w_kv, w.k_gain,
                     dfl.KVCache(kp, vp, seq, block_table=torch.as_tensor(table, device=DEV)))
    torch.cuda.synchronize()
    assert dfl.read_device_status() & BAD_SEQLEN
    # rows 126, 127 of sequence 0 (page 0) and rows 0..3 of sequence 1 (page 1) are written; nothing else
    assert not torch.all(kp[:, 0, :, 126:128] == 7.0)
    assert torch.all(kp[:, 0, :, :126] == 7.0)
    assert not torch.all(kp[:, 1, :, 0:4] == 7.0)
    assert torch.all(kp[:, 1, :, 4:] == 7.0)
    assert torch.all(kp[:, 2:] == 7.0) and torch.all(vp[:, 2:] == 7.0)
