"""A whole draft forward on the GPU against the oracle composed the same way.

Five layers, each: input RMSNorm and q/k/v projections
(dflash_draft_layer_qkv) -> non-causal block attention over the layer's
cached context plus the block (dflash_block_attn) -> output projection,
post-attention norm, SwiGLU MLP and residuals (dflash_draft_layer_tail); then
the drafter's head on the mask rows (dflash_draft_head: final norm, LM head,
draft sampling).  E4B page, "The released serving cycle" (one non-causal
multi-layer pass over the block) and "The parameter count exposes the real
cost" (q/k/v/o projections, gated MLP, two norms per layer).

Checked two ways:
  * call by call: each call against the oracle applied to the GPU's own
    inputs of that call (q/k/v from the layer's input, attention from the
    GPU's q/k/v, the layer remainder from the GPU's attention output, the
    head from the GPU's final rows) -- the relative bounds of the other parity
    tests (2e-3, per tensor and per row);
  * composed: the oracle run through all five layers and the head on its own
    outputs.  Both sides round to bf16 independently at every storage point of
    a layer (the normalised rows, q/k/v, the attention output, x1, the
    post-attention rows, the SwiGLU activations, x2); values that land one
    bf16 step apart there are carried into the next layer, so the difference
    grows with depth (measured on this case: 2.1e-3 after the first layer,
    then about 1.5e-3 more per layer, 8.1e-3 after five, 8.5e-3 in the
    logits).  The composed hidden state after layer l is held to
    4e-3 * (l + 1) relative and the logits to 2e-2 (twice the first layer's
    growth per layer), per tensor and per row.
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"

L, B, BS, HQ, HKV, D, I, V = 5, 4, 8, 32, 8, 2560, 5120, 32768
SEQ = [100, 700, 1500, 0]
CAP = 1536


def _weights(seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    r = lambda *s, std=0.02: (torch.randn(*s, generator=g, device=DEV) * std).to(torch.bfloat16)  # noqa: E731
    gain = lambda *s: (1 + 0.1 * torch.randn(*s, generator=g, device=DEV)).to(torch.bfloat16)  # noqa: E731
    w = dict(
        g_in=gain(L, D), w_qkv=r(L, (HQ + 2 * HKV) * 128, D), q_gain=gain(L, 128), k_gain=gain(L, 128),
        w_o=r(L, D, HQ * 128), g_post=gain(L, D), w_gate=r(L, I, D), w_up=r(L, I, D), w_down=r(L, D, I),
        g_final=gain(D), w_head=r(V, D, std=0.05))
    w["w_gu"] = torch.stack([dfl.interleave_gate_up(w["w_gate"][l], w["w_up"][l]) for l in range(L)])
    k = r(L, B, HKV, CAP, 128, std=1.0)
    v = r(L, B, HKV, CAP, 128, std=1.0)
    x0 = r(B * BS, D, std=1.0)
    return w, k, v, x0


def _oracle_layer(x, l, w, k, v):
    q, kb, vb = oracle.draft_layer_qkv(x, np64(w["g_in"][l]), np64(w["w_qkv"][l]), B, HQ, HKV, bf16=True)
    o = oracle.block_attn(q, kb, vb, np64(w["q_gain"][l]), np64(w["k_gain"][l]), np64(k[l]), np64(v[l]),
                          np.asarray(SEQ), bf16=True)
    _, x2 = oracle.draft_layer_tail(x, o, np64(w["w_o"][l]), np64(w["g_post"][l]), np64(w["w_gate"][l]),
                                    np64(w["w_up"][l]), np64(w["w_down"][l]), bf16=True)
    return x2


def test_five_layer_draft_forward_and_head_match_the_composed_oracle():
    w, k, v, x0 = _weights(123)
    cache = dfl.KVCache(k, v, torch.tensor(SEQ, dtype=torch.int32, device=DEV))
    x = x0.clone()
    calls = []
    for l in range(L):
        x_in = x.clone()
        q, kb, vb = dfl.draft_layer_qkv(x, w["g_in"][l], w["w_qkv"][l], B, HQ, HKV)
        o = dfl.block_attn(l, q, kb, vb, w["q_gain"][l], w["k_gain"][l], cache)
        dfl.draft_layer_tail(x, o, w["w_o"][l], w["g_post"][l], w["w_gu"][l], w["w_down"][l])
        calls.append((x_in, q.clone(), kb.clone(), vb.clone(), o.clone(), x.clone()))
    rows = torch.tensor([b * BS + j for b in range(B) for j in range(1, BS)], device=DEV)   # the mask rows
    xh = x[rows].contiguous()
    logits, tok = dfl.draft_head(xh, w["g_final"], w["w_head"], BS - 1, 1.0, 77, 5)
    torch.cuda.synchronize()
    assert dfl.read_device_status() == 0

    # call by call, each from the GPU's own inputs
    for l, (x_in, q, kb, vb, o, x_out) in enumerate(calls):
        rq, rk, rv = oracle.draft_layer_qkv(np64(x_in), np64(w["g_in"][l]), np64(w["w_qkv"][l]), B, HQ, HKV,
                                            bf16=True)
        for got, ref, what in ((q, rq, "q"), (kb, rk, "kb"), (vb, rv, "vb")):
            assert_close(got, ref, torch.bfloat16, row=128, what="layer %d %s" % (l, what))
        ro = oracle.block_attn(np64(q), np64(kb), np64(vb), np64(w["q_gain"][l]), np64(w["k_gain"][l]),
                               np64(k[l]), np64(v[l]), np.asarray(SEQ), bf16=True)
        assert_close(o, ro, torch.bfloat16, row=128, what="layer %d attention" % l)
        _, rx = oracle.draft_layer_tail(np64(x_in), np64(o), np64(w["w_o"][l]), np64(w["g_post"][l]),
                                        np64(w["w_gate"][l]), np64(w["w_up"][l]), np64(w["w_down"][l]), bf16=True)
        assert_close(x_out, rx, torch.bfloat16, row=D, what="layer %d remainder" % l)
    ref_logits = oracle.draft_head(np64(xh), np64(w["g_final"]), np64(w["w_head"]), bf16=True)
    assert_close(logits, ref_logits, torch.bfloat16, row=V, what="head")

    # composed: the oracle on its own outputs through all five layers and the head
    xr = np64(x0)
    for l in range(L):
        xr = _oracle_layer(xr, l, w, k, v)
        assert_close(calls[l][5], xr, 4e-3 * (l + 1), row=D, what="composed x after layer %d" % l)
    rows_np = rows.cpu().numpy()
    ref_logits_c = oracle.draft_head(xr[rows_np], np64(w["g_final"]), np64(w["w_head"]), bf16=True)
    assert_close(logits, ref_logits_c, 2e-2, row=V, what="composed logits")

    # the draft tokens: the oracle's race on the GPU's logits
    got = logits.float().cpu().numpy().reshape(B, BS - 1, V)
    ref_tok, near = oracle.draft_sample(got, 1.0, 77, 5)
    toks = tok.cpu().numpy().reshape(B, BS - 1)
    assert np.all((toks == ref_tok) | near), (toks, ref_tok)
