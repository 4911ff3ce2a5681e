"""GPU parity at the documented maximum and degenerate sizes of the calls.

Block attention at its largest bf16 batch (2048 sequences, most with short or
empty cached contexts); the layer's q/k/v and remainder at the largest model
width (4096) with one block row per sequence; the drafter head with a single
proposal row per sequence and the largest rows-per-sequence (31); fusion of a
single new row.  Each compares with the oracle under the bounds of the other
parity tests (relative 2e-3 per tensor and per row, integers exact).
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


def test_block_attn_largest_batch_short_contexts():
    """2048 sequences (the bf16 maximum), cached lengths 0..300: checked on
    a sample of 24 sequences, including empty ones and the last one."""
    B, bs, cap = 2048, 8, 320
    g = torch.Generator(device=DEV).manual_seed(61)
    seq = torch.randint(0, 301, (B,), generator=g, device=DEV, dtype=torch.int32)
    seq[::97] = 0
    k = torch.randn(1, B, 8, cap, 128, generator=g, device=DEV).to(torch.bfloat16)
    v = torch.randn(1, B, 8, cap, 128, generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn(B, 32, bs, 128, generator=g, device=DEV).to(torch.bfloat16)
    kb = torch.randn(B, 8, bs, 128, generator=g, device=DEV).to(torch.bfloat16)
    vb = torch.randn(B, 8, bs, 128, generator=g, device=DEV).to(torch.bfloat16)
    qg = (1 + 0.1 * torch.randn(128, generator=g, device=DEV)).to(torch.bfloat16)
    kg = (1 + 0.1 * torch.randn(128, generator=g, device=DEV)).to(torch.bfloat16)
    dfl.read_device_status()
    out = dfl.block_attn(0, q, kb, vb, qg, kg, dfl.KVCache(k, v, seq))
    torch.cuda.synchronize()
    assert dfl.read_device_status() == 0
    sel = np.unique(np.concatenate([np.random.default_rng(3).choice(B, 21, replace=False), [0, 97, B - 1]]))
    st = torch.as_tensor(sel, device=DEV)
    ref = oracle.block_attn(np64(q[st]), np64(kb[st]), np64(vb[st]), np64(qg), np64(kg), np64(k[0, st]),
                            np64(v[0, st]), seq.cpu().numpy()[sel], bf16=True)
    assert_close(out[st], ref, torch.bfloat16, row=128, what="out")


def test_layer_qkv_and_tail_at_the_largest_width_one_row_per_sequence():
    B, bs, Hq, Hkv, D, I = 6, 1, 4, 2, 4096, 256
    g = torch.Generator(device=DEV).manual_seed(62)
    r = lambda *s, std=1.0: (torch.randn(*s, generator=g, device=DEV) * std).to(torch.bfloat16)  # noqa: E731
    x = r(B * bs, D, std=2.0)
    g_in = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(torch.bfloat16)
    w_qkv = r((Hq + 2 * Hkv) * 128, D, std=0.02)
    q, kb, vb = dfl.draft_layer_qkv(x, g_in, w_qkv, B, Hq, Hkv)
    rq, rk, rv = oracle.draft_layer_qkv(np64(x), np64(g_in), np64(w_qkv), B, Hq, Hkv, bf16=True)
    for got, ref, what in ((q, rq, "q"), (kb, rk, "kb"), (vb, rv, "vb")):
        assert_close(got, ref, torch.bfloat16, row=128, what=what)
    o = r(B, Hq, bs, 128)
    w_o, w_gate, w_up, w_down = r(D, Hq * 128, std=0.02), r(I, D, std=0.05), r(I, D, std=0.05), r(D, I, std=0.02)
    g_post = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(torch.bfloat16)
    x2 = x.clone()
    dfl.draft_layer_tail(x2, o, w_o, g_post, dfl.interleave_gate_up(w_gate, w_up), w_down)
    torch.cuda.synchronize()
    _, ref = oracle.draft_layer_tail(np64(x), np64(o), np64(w_o), np64(g_post), np64(w_gate), np64(w_up),
                                     np64(w_down), bf16=True)
    assert_close(x2, ref, torch.bfloat16, row=D, what="x2")


@pytest.mark.parametrize("R", [1, 31])
def test_draft_head_one_and_the_most_rows_per_sequence(R):
    B, D, V = 3, 256, 1024
    g = torch.Generator(device=DEV).manual_seed(63 + R)
    x = (torch.randn(B * R, D, generator=g, device=DEV) * 2.0).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(torch.bfloat16)
    w = (torch.randn(V, D, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    logits, tok = dfl.draft_head(x, gain, w, R, 1.0, 5, 9)
    torch.cuda.synchronize()
    ref = oracle.draft_head(np64(x), np64(gain), np64(w), bf16=True)
    assert_close(logits, ref, torch.bfloat16, row=V, what="logits")
    got = logits.float().cpu().numpy().reshape(B, R, V)
    rtok, near = oracle.draft_sample(got, 1.0, 5, 9)
    assert np.all((tok.cpu().numpy().reshape(B, R) == rtok) | near)


def test_fuse_a_single_new_row():
    cfg = workloads.SINGLE_STREAM
    w = workloads.weights(cfg, DEV)
    taps = workloads.taps(cfg, 1, DEV, seed_offset=3)
    k = torch.full((cfg.L, 1, cfg.Hkv, 64, cfg.d), 7.0, dtype=torch.bfloat16, device=DEV)
    v = torch.full_like(k, 7.0)
    seq = torch.tensor([63], dtype=torch.int32, device=DEV)          # the last free position
    ht = torch.empty(1, cfg.D, dtype=torch.bfloat16, device=DEV)
    dfl.fuse_context(taps, workloads.cu_rows([1], DEV), w.w_fuse, w.g_fuse, w.w_kv, w.k_gain,
                     dfl.KVCache(k, v, seq), h_t_out=ht)
    torch.cuda.synchronize()
    assert dfl.read_device_status() == 0
    H, K, V = oracle.fuse_rows([np64(t) for t in taps], np64(w.w_fuse), np64(w.g_fuse), np64(w.w_kv),
                               np64(w.k_gain), np.array([63]), cfg.L, cfg.Hkv, cfg.d, bf16=True)
    assert_close(ht, H, torch.bfloat16, row=cfg.D, what="H_t")
    assert_close(k[:, 0, :, 63][None], K, torch.bfloat16, row=cfg.d, what="K")
    assert_close(v[:, 0, :, 63][None], V, torch.bfloat16, row=cfg.d, what="V")
    assert torch.all(k[:, :, :, :63] == 7.0) and torch.all(v[:, :, :, :63] == 7.0)
