"""GPU parity of dflash_block_attn against the oracle.

Relative error of the output <= 2e-3 (bf16) / 1e-5 (fp32), both over the whole
tensor (Frobenius) and for every 128-wide head row of it, on small
cases spanning several 128-key tiles, several key splits and a ragged tail, and
on sampled sequences of the full-size workloads in the launch configuration
the benchmark uses.
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


def _inputs(B, bs, cap, dtype, seed, Hq=32, Hkv=8, layers=2):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(layers, B, Hkv, cap, 128, generator=g).to(dtype)
    v = torch.randn(layers, B, Hkv, cap, 128, generator=g).to(dtype)
    q = torch.randn(B, Hq, bs, 128, generator=g).to(dtype)
    kb = torch.randn(B, Hkv, bs, 128, generator=g).to(dtype)
    vb = torch.randn(B, Hkv, bs, 128, generator=g).to(dtype)
    qg = (1 + 0.1 * torch.randn(128, generator=g)).to(dtype)
    kg = (1 + 0.1 * torch.randn(128, generator=g)).to(dtype)
    return k, v, q, kb, vb, qg, kg


def _oracle(q, kb, vb, qg, kg, k_layer, v_layer, seq, window, dtype):
    return oracle.block_attn(np64(q), np64(kb), np64(vb), np64(qg), np64(kg), np64(k_layer), np64(v_layer),
                             np.asarray(seq), window=window, bf16=(dtype == torch.bfloat16))


@pytest.mark.parametrize("bs", [1, 4, 5, 8, 16])
@pytest.mark.parametrize("window", [0, 100])
def test_block_attn_bf16_small(bs, window):
    seq = [0, 70, 700]
    cap = 768
    k, v, q, kb, vb, qg, kg = _inputs(3, bs, cap, torch.bfloat16, seed=bs * 10 + window)
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(1, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache, window=window)
    ref = _oracle(q, kb, vb, qg, kg, k[1], v[1], seq, window, torch.bfloat16)
    assert_close(out, ref, torch.bfloat16, row=128, what="out")


@pytest.mark.parametrize("bs", [8, 16])
def test_block_attn_never_reads_past_seq_len(bs):
    """Cache rows at and past seq_len (and the other layer) hold NaN: the output
    must not see them, for lengths on, just before and just after tile edges."""
    seq = [0, 1, 127, 128, 129, 255, 256, 700, 1000]
    cap = 1024
    k, v, q, kb, vb, qg, kg = _inputs(len(seq), bs, cap, torch.bfloat16, seed=40 + bs)
    kn, vn = k.clone(), v.clone()
    for b, n in enumerate(seq):
        kn[:, b, :, n:] = float("nan")
        vn[:, b, :, n:] = float("nan")
    kn[0] = float("nan")
    vn[0] = float("nan")
    cache = dfl.KVCache(kn.to(DEV), vn.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(1, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache)
    assert torch.isfinite(out.float()).all()
    ref = _oracle(q, kb, vb, qg, kg, k[1], v[1], seq, 0, torch.bfloat16)
    assert_close(out, ref, torch.bfloat16, row=128, what="out")


def test_block_attn_scores_far_above_the_first_tile_stay_exact():
    """A key scoring ~2^290 above the first tile's maximum, late in a
    three-split sequence, in a single-split sequence and (not flagged) in a
    first tile: the outputs still match the oracle."""
    seq = [700, 200, 300]
    cap = 1024
    k, v, q, kb, vb, qg, kg = _inputs(3, 8, cap, torch.bfloat16, seed=77, layers=1)
    g = torch.Generator().manual_seed(78)
    for b, pos, head in [(0, 650, 3), (1, 150, 5), (2, 10, 1)]:
        k[0, b, head, pos] = (200.0 * torch.randn(128, generator=g)).to(torch.bfloat16)
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache)
    assert torch.isfinite(out.float()).all()
    ref = _oracle(q, kb, vb, qg, kg, k[0], v[0], seq, 0, torch.bfloat16)
    assert_close(out, ref, torch.bfloat16, row=128, what="out")


@pytest.mark.parametrize("Hq,Hkv,bs", [(4, 4, 16), (8, 8, 1), (12, 4, 5), (16, 2, 3), (32, 2, 4)])
def test_block_attn_head_groupings(Hq, Hkv, bs):
    """Query heads per KV head G = 1, 3, 8 and 16 (32 and 64 query rows per
    pair): the main kernel normalises and rotates each block position's G
    query rows and its block key together; an empty cache, a ragged length
    and several tiles."""
    seq = [0, 130, 700]
    cap = 768
    k, v, q, kb, vb, qg, kg = _inputs(3, bs, cap, torch.bfloat16, seed=Hq * 31 + Hkv * 7 + bs, Hq=Hq, Hkv=Hkv)
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(1, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache)
    ref = _oracle(q, kb, vb, qg, kg, k[1], v[1], seq, 0, torch.bfloat16)
    assert_close(out, ref, torch.bfloat16, row=128, what="out")


def test_block_attn_fp32_tiny_case():
    cfg = workloads.TINY_FP32
    k, v, q, kb, vb, qg, kg = _inputs(2, cfg.bs, 128, torch.float32, seed=1, layers=1)
    seq = [64, 5]
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache)
    ref = _oracle(q, kb, vb, qg, kg, k[0], v[0], seq, 0, torch.float32)
    assert_close(out, ref, torch.float32, row=128, what="out")


def test_block_attn_null_gains_mean_ones():
    k, v, q, kb, vb, qg, kg = _inputs(2, 8, 320, torch.bfloat16, seed=5)
    seq = [300, 17]
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), torch.tensor(seq, dtype=torch.int32, device=DEV))
    out = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), None, None, cache)
    ref = _oracle(q, kb, vb, torch.ones(128), torch.ones(128), k[0], v[0], seq, 0, torch.bfloat16)
    assert_close(out, ref, torch.bfloat16, row=128, what="out")


def _full_size(cfg, layer, sample):
    """Run the whole batch on the GPU (benchmark launch), check `sample` sequences."""
    seq = workloads.seq_lens(cfg, DEV)
    k, v = workloads.cache(cfg, DEV, layers=1)
    w = workloads.weights(cfg, DEV)
    q, kb, vb = workloads.block(cfg, DEV, layer=layer)
    cache = dfl.KVCache(k, v, seq)
    dfl.read_device_status()
    out = dfl.block_attn(0, q, kb, vb, w.q_gain[layer], w.k_gain[layer], cache)
    assert dfl.read_device_status() == 0  # no bounded wait gave up, no bad length
    sel = torch.tensor(sample)
    seq_c = seq.cpu()[sel]
    nmax = int(seq_c.max())
    ref = _oracle(q[sel], kb[sel], vb[sel], w.q_gain[layer], w.k_gain[layer], k[0, sel, :, :nmax],
                  v[0, sel, :, :nmax], seq_c.numpy(), 0, cfg.dtype)
    return assert_close(out[sel], ref, cfg.dtype, row=128, what=cfg.name)[1]


def test_block_attn_batched_full_size_sampled():
    print("batched worst-row rel err %.2e" % _full_size(workloads.BATCHED, 2, [0, 5, 17, 31]))


def test_block_attn_high_batch_bs16_sampled():
    print("high_batch bs16 worst-row rel err %.2e" % _full_size(workloads.high_batch(16, 1.0), 0, [0, 63, 127]))


def test_block_attn_high_batch_bs4_sampled():
    print("high_batch bs4 worst-row rel err %.2e" % _full_size(workloads.high_batch(4, 1.0), 1, [3, 100]))


def test_block_attn_long_context_sampled():
    print("long_context worst-row rel err %.2e" % _full_size(workloads.LONG_CONTEXT, 0, [0, 3]))


def test_block_attn_single_stream():
    print("single_stream worst-row rel err %.2e" % _full_size(workloads.SINGLE_STREAM, 4, [0]))


def test_block_attn_bad_seq_len_is_flagged_not_faulted():
    k, v, q, kb, vb, qg, kg = _inputs(2, 8, 128, torch.bfloat16, seed=9)
    seq = torch.tensor([100, 5000], dtype=torch.int32, device=DEV)   # 5000 > capacity 128
    cache = dfl.KVCache(k.to(DEV), v.to(DEV), seq)
    dfl.read_device_status()
    out = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV), cache)
    assert dfl.read_device_status() & dfl.DEV_BAD_SEQLEN
    ref = _oracle(q[:1], kb[:1], vb[:1], qg, kg, k[0, :1], v[0, :1], [100], 0, torch.bfloat16)
    assert_close(out[:1], ref, torch.bfloat16, row=128, what="out")
    assert torch.isfinite(out.float()).all()


def test_block_attn_split_count_does_not_change_the_result():
    """The same 3000-token sequence attended alone (batch 1: 256-key splits,
    12 of them) and as the first of a batch of four (896-key splits, 4 of
    them): both outputs match the oracle and each other to a few bf16 ulps."""
    seq = [3000, 100, 2000, 4000]
    cap = 4096
    k, v, q, kb, vb, qg, kg = _inputs(4, 8, cap, torch.bfloat16, seed=91, layers=1)
    outs = []
    for B in (1, 4):
        cache = dfl.KVCache(k[:, :B].contiguous().to(DEV), v[:, :B].contiguous().to(DEV),
                            torch.tensor(seq[:B], dtype=torch.int32, device=DEV))
        outs.append(dfl.block_attn(0, q[:B].to(DEV), kb[:B].to(DEV), vb[:B].to(DEV), qg.to(DEV), kg.to(DEV), cache))
    ref = _oracle(q[:1], kb[:1], vb[:1], qg, kg, k[0, :1], v[0, :1], seq[:1], 0, torch.bfloat16)
    for out in outs:
        assert_close(out[:1], ref, torch.bfloat16, row=128, what="out")
    assert_close(outs[0], outs[1][:1].float().cpu().numpy(), 2e-3, row=128, what="1 vs 4 sequences")


def test_block_attn_is_invariant_to_the_order_of_cached_rows():
    """Permuting a sequence's cached (key, value) rows together leaves the
    output unchanged up to summation order."""
    seq = [900, 400]
    cap = 1024
    k, v, q, kb, vb, qg, kg = _inputs(2, 8, cap, torch.bfloat16, seed=93, layers=1)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(seq[0]))
    kp, vp = k.clone(), v.clone()
    kp[0, 0, :, :seq[0]] = k[0, 0][:, perm]
    vp[0, 0, :, :seq[0]] = v[0, 0][:, perm]
    sl = torch.tensor(seq, dtype=torch.int32, device=DEV)
    a = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV),
                       dfl.KVCache(k.to(DEV), v.to(DEV), sl))
    b = dfl.block_attn(0, q.to(DEV), kb.to(DEV), vb.to(DEV), qg.to(DEV), kg.to(DEV),
                       dfl.KVCache(kp.to(DEV), vp.to(DEV), sl))
    assert_close(a, b.float().cpu().numpy(), 2e-3, row=128, what="permuted")
    assert torch.equal(a[1], b[1])     # the other sequence is untouched bit for bit
