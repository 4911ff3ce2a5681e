"""One draft-and-verify cycle captured into a CUDA graph and replayed.

Every call of the library is stream-ordered, allocates nothing when it is
given its workspace, and never synchronises, so a serving loop can capture a
whole cycle once (context fusion, the block attention of each layer,
verification) and replay it; the kernels' programmatic dependent launches
become programmatic edges of the graph.  The replay must reproduce the eager
run bit for bit: the cache rows the fusion appends, every layer's attention
output, and the accepted lengths and tokens.
"""
from dataclasses import replace

import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(cfg, T):
    seq = workloads.seq_lens(cfg, DEV)
    k, v = workloads.cache(cfg, DEV)
    w = workloads.weights(cfg, DEV)
    M = cfg.B * cfg.bs
    taps = workloads.taps(cfg, M, DEV)
    cu = workloads.cu_rows([cfg.bs] * cfg.B, DEV)
    blocks = [workloads.block(cfg, DEV, layer=l) for l in range(cfg.L)]
    lt, ld = workloads.logits(cfg, DEV)
    x = workloads.draft_tokens(ld, T, seed=cfg.seed + 7)
    cache = dfl.KVCache(k, v, seq)
    outs = [torch.empty_like(b[0]) for b in blocks]
    acc = torch.empty(cfg.B, dtype=torch.int32, device=DEV)
    tok = torch.empty(cfg.B, cfg.bs, dtype=torch.int32, device=DEV)
    dt = dfl.BF16
    ws_f = torch.empty(dfl.fuse_context_workspace_size(M, cfg.J, cfg.d_target, cfg.D, cfg.L, cfg.Hkv, dt),
                       dtype=torch.uint8, device=DEV)
    ws_a = torch.empty(dfl.block_attn_workspace_size(cfg.B, cfg.bs, cfg.Hq, cfg.Hkv, cfg.capacity, 0, dt),
                       dtype=torch.uint8, device=DEV)
    ws_v = torch.empty(dfl.verify_workspace_size(cfg.B, cfg.bs, cfg.V, dt), dtype=torch.uint8, device=DEV)

    def cycle(stream):
        dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain, cache, workspace=ws_f, stream=stream)
        for l in range(cfg.L):
            q, kb, vb = blocks[l]
            dfl.block_attn(l, q, kb, vb, w.q_gain[l], w.k_gain[l], cache, out=outs[l], workspace=ws_a, stream=stream)
        dfl.verify(lt, ld, x, T, 1234, 5, accepted_len=acc, out_tokens=tok, workspace=ws_v, stream=stream)

    return cycle, (k, v), outs, acc, tok


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_cycle_replays_from_a_cuda_graph(T):
    cfg = replace(workloads.BATCHED, B=6, S=2048, S_min=256, L=2, name="graph_small")
    cycle, (k, v), outs, acc, tok = _setup(cfg, T)
    k0, v0 = k.clone(), v.clone()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cycle(s)
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs], acc.clone(), tok.clone(), k.clone(), v.clone()
    assert not torch.equal(ref[3], k0)  # the fusion wrote new cache rows

    def reset():
        for o in outs:
            o.fill_(float("nan"))
        acc.fill_(-7)
        tok.fill_(-7)
        k.copy_(k0)
        v.copy_(v0)
        torch.cuda.synchronize()

    reset()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cycle(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for _ in range(2):  # replays overwrite the same buffers with the same values
        reset()
        g.replay()
        torch.cuda.synchronize()
        for l, o in enumerate(outs):
            assert torch.equal(o, ref[0][l]), "layer %d attention output differs from the eager run" % l
        assert torch.equal(acc, ref[1]) and torch.equal(tok, ref[2])
        assert torch.equal(k, ref[3]) and torch.equal(v, ref[4])
