"""Calls on two streams at once, each with its own workspace and outputs.

The library keeps no per-call state outside the caller's buffers (the device
status word only collects error bits), so two independent cycles interleaved
on two streams must give exactly what each gives alone: block attention of
two caches, and verification of two batches, launched alternately.
"""
from dataclasses import replace

import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    cfg = replace(workloads.BATCHED, B=5, S=4096, S_min=512, L=1, seed=seed, name="streams_%d" % seed)
    seq = workloads.seq_lens(cfg, DEV)
    k, v = workloads.cache(cfg, DEV)
    w = workloads.weights(cfg, DEV)
    q, kb, vb = workloads.block(cfg, DEV, layer=0)
    lt, ld = workloads.logits(cfg, DEV)
    x = workloads.draft_tokens(ld, 1.0, seed=seed + 7)
    dt = dfl.BF16
    c = {
        "cfg": cfg, "cache": dfl.KVCache(k, v, seq), "w": w, "q": q, "kb": kb, "vb": vb, "lt": lt, "ld": ld, "x": x,
        "out": torch.empty_like(q),
        "acc": torch.empty(cfg.B, dtype=torch.int32, device=DEV),
        "tok": torch.empty(cfg.B, cfg.bs, dtype=torch.int32, device=DEV),
        "ws_a": torch.empty(dfl.block_attn_workspace_size(cfg.B, cfg.bs, cfg.Hq, cfg.Hkv, cfg.capacity, 0, dt),
                            dtype=torch.uint8, device=DEV),
        "ws_v": torch.empty(dfl.verify_workspace_size(cfg.B, cfg.bs, cfg.V, dt), dtype=torch.uint8, device=DEV),
    }
    return c


def _attn(c, stream):
    dfl.block_attn(0, c["q"], c["kb"], c["vb"], c["w"].q_gain[0], c["w"].k_gain[0], c["cache"], out=c["out"],
                   workspace=c["ws_a"], stream=stream)


def _verify(c, stream, cycle):
    dfl.verify(c["lt"], c["ld"], c["x"], 1.0, 99, cycle, accepted_len=c["acc"], out_tokens=c["tok"],
               workspace=c["ws_v"], stream=stream)


def test_two_streams_give_the_results_of_each_alone():
    a, b = _case(41), _case(42)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    # each alone
    ref = {}
    for name, c, s in (("a", a, s1), ("b", b, s2)):
        with torch.cuda.stream(s):
            _attn(c, s)
            _verify(c, s, 3)
        s.synchronize()
        ref[name] = (c["out"].clone(), c["acc"].clone(), c["tok"].clone())
    for c in (a, b):
        c["out"].fill_(float("nan"))
        c["acc"].fill_(-7)
        c["tok"].fill_(-7)
    torch.cuda.synchronize()
    # interleaved: every call of one stream launched between two of the other's
    for _ in range(3):
        with torch.cuda.stream(s1):
            _attn(a, s1)
        with torch.cuda.stream(s2):
            _attn(b, s2)
        with torch.cuda.stream(s1):
            _verify(a, s1, 3)
        with torch.cuda.stream(s2):
            _verify(b, s2, 3)
    torch.cuda.synchronize()
    for name, c in (("a", a), ("b", b)):
        out, acc, tok = ref[name]
        assert torch.equal(c["out"], out), name
        assert torch.equal(c["acc"], acc) and torch.equal(c["tok"], tok), name
