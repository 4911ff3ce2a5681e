"""Calls chained back to back on one stream give the same bytes as calls separated by host syncs.

Every call launches its kernels as programmatic dependents, so a call's first
kernel can become resident while the previous call's last kernel still runs.
Fusion -> attention -> layer remainder -> attention -> layer remainder ->
drafter head -> verification are run (a) with a host synchronisation after
every call and (b) back to back, three times; all results are deterministic,
so any read of a previous call's output before that output is complete would
show as a difference.
"""
import pytest
import torch

import block_speculative_decoding_gb300 as dfl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)

    def r(*s, std=1.0):
        return (torch.randn(*s, generator=g, device=DEV) * std).to(torch.bfloat16)
    B, bs, D, Hq, Hkv, L, I, V, J, dt, cap = 4, 8, 256, 4, 2, 2, 256, 4096, 5, 256, 512
    c = dict(B=B, bs=bs, D=D, Hq=Hq, Hkv=Hkv, L=L, I=I, V=V)
    c["taps"] = [r(B * bs, dt) for _ in range(J)]
    c["cu"] = torch.arange(0, B * bs + 1, bs, dtype=torch.int32, device=DEV)
    c["seq"] = torch.tensor([0, 100, 250, 400], dtype=torch.int32, device=DEV)
    c["w_fuse"], c["g_fuse"] = r(D, J * dt, std=0.02), (1 + 0.1 * r(D).float()).to(torch.bfloat16)
    c["w_kv"], c["k_gain"] = r(L * 2 * Hkv * 128, D, std=0.05), (1 + 0.1 * r(L, 128).float()).to(torch.bfloat16)
    c["q_gain"] = (1 + 0.1 * r(L, 128).float()).to(torch.bfloat16)
    c["blocks"] = [(r(B, Hq, bs, 128), r(B, Hkv, bs, 128), r(B, Hkv, bs, 128)) for _ in range(L)]
    c["w_o"] = [r(D, Hq * 128, std=0.02) for _ in range(L)]
    c["g_post"] = [(1 + 0.1 * r(D).float()).to(torch.bfloat16) for _ in range(L)]
    c["w_gu"] = [r(2 * I, D, std=0.05) for _ in range(L)]
    c["w_dn"] = [r(D, I, std=0.02) for _ in range(L)]
    c["x0"] = r(B * bs, D, std=2.0)
    c["g_final"] = (1 + 0.1 * r(D).float()).to(torch.bfloat16)
    c["w_head"] = r(V, D, std=0.05)
    c["lt"] = r(B, bs, V, std=3.0)
    c["ld"] = r(B, bs - 1, V, std=3.0)
    c["xt"] = torch.randint(0, V, (B, bs - 1), generator=g, device=DEV, dtype=torch.int32)
    c["cap"] = cap
    return c


def _run(c, sync):
    B, bs, L, Hkv = c["B"], c["bs"], c["L"], c["Hkv"]
    k = torch.zeros(L, B, Hkv, c["cap"], 128, dtype=torch.bfloat16, device=DEV)
    cache = dfl.KVCache(k, torch.zeros_like(k), c["seq"].clone())
    x = c["x0"].clone()
    outs = [torch.empty_like(b[0]) for b in c["blocks"]]
    logits = torch.empty(B * bs, c["V"], dtype=torch.bfloat16, device=DEV)
    toks = torch.empty(B * bs, dtype=torch.int32, device=DEV)
    # workspaces allocated up front: no allocation between the chained calls
    ws_f = torch.empty(dfl.fuse_context_workspace_size(B * bs, 5, 256, c["D"], L, Hkv, dfl.BF16),
                       dtype=torch.uint8, device=DEV)
    ws_a = torch.empty(dfl.block_attn_workspace_size(B, bs, c["Hq"], Hkv, c["cap"], 0, dfl.BF16),
                       dtype=torch.uint8, device=DEV)
    ws_t = torch.empty(dfl.draft_layer_tail_workspace_size(B, bs, c["Hq"], c["D"], c["I"]), dtype=torch.uint8,
                       device=DEV)
    ws_h = torch.empty(dfl.draft_head_workspace_size(B, bs, c["D"], c["V"]), dtype=torch.uint8, device=DEV)
    ws_v = torch.empty(dfl.verify_workspace_size(B, bs, c["V"], dfl.BF16), dtype=torch.uint8, device=DEV)
    acc = torch.empty(B, dtype=torch.int32, device=DEV)
    out_t = torch.empty(B, bs, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    step = torch.cuda.synchronize if sync else (lambda: None)
    dfl.fuse_context(c["taps"], c["cu"], c["w_fuse"], c["g_fuse"], c["w_kv"], c["k_gain"], cache, workspace=ws_f)
    step()
    for l in range(L):
        q, kb, vb = c["blocks"][l]
        dfl.block_attn(l, q, kb, vb, c["q_gain"][l], c["k_gain"][l], cache, out=outs[l], workspace=ws_a)
        step()
        dfl.draft_layer_tail(x, outs[l], c["w_o"][l], c["g_post"][l], c["w_gu"][l], c["w_dn"][l], workspace=ws_t)
        step()
    dfl.draft_head(x, c["g_final"], c["w_head"], bs, 1.0, 7, 3, logits=logits, tokens=toks, workspace=ws_h)
    step()
    dfl.verify(c["lt"], c["ld"], c["xt"], 1.0, 11, 5, accepted_len=acc, out_tokens=out_t, workspace=ws_v)
    torch.cuda.synchronize()
    return [cache.k, cache.v, *outs, x, logits, toks, acc, out_t]


def test_chained_calls_equal_synchronised_calls():
    c = _setup()
    ref = _run(c, sync=True)
    assert dfl.read_device_status() == 0
    for _ in range(3):
        got = _run(c, sync=False)
        assert dfl.read_device_status() == 0
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a, b), i
