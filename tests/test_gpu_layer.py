"""GPU parity of dflash_draft_layer_qkv and dflash_draft_layer_tail against the oracle.

dflash_draft_layer_qkv: q, kb and vb (the input norm and the projections,
bf16 storage of the normalised rows and of the outputs) within the relative
bounds of the oracle's, for block sizes 4, 8, 16 on small shapes, the batched
workload's shape (every row) and a 2048-row high-batch shape (sampled rows).

The updated residual stream x2 must match the oracle's (bf16 storage of x1, the
normalised rows, the SwiGLU activations and x2) within the relative Frobenius
bound and the per-row bound (each D-wide row), on small cases with several tiles and split-K slots and on sampled
sequences of the batched workload's shapes (D = 2560, 32 heads, I = 5120).
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, bs, Hq, D, I, seed, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed)
    r = lambda *s, std=1.0: (torch.randn(*s, generator=g, device=device) * std).to(torch.bfloat16)  # noqa: E731
    return dict(x=r(B * bs, D, std=2.0), o=r(B, Hq, bs, 128), w_o=r(D, Hq * 128, std=0.02),
                g_post=(1 + 0.1 * torch.randn(D, generator=g, device=device)).to(torch.bfloat16),
                w_gate=r(I, D, std=0.05), w_up=r(I, D, std=0.05), w_down=r(D, I, std=0.02))


def _run(c):
    x = c["x"].to(DEV).clone()
    dfl.draft_layer_tail(x, c["o"].to(DEV), c["w_o"].to(DEV), c["g_post"].to(DEV),
                         dfl.interleave_gate_up(c["w_gate"].to(DEV), c["w_up"].to(DEV)), c["w_down"].to(DEV))
    torch.cuda.synchronize()
    return x


@pytest.mark.parametrize("bs", [4, 8, 16])
def test_layer_tail_small(bs):
    c = _case(B=5, bs=bs, Hq=4, D=256, I=192, seed=bs)
    x2 = _run(c)
    _, ref = oracle.draft_layer_tail(*[np64(c[k]) for k in ("x", "o", "w_o", "g_post", "w_gate", "w_up", "w_down")],
                                     bf16=True)
    assert_close(x2, ref, torch.bfloat16, row=c["x"].shape[1], what="x2")


def test_layer_tail_zero_projections_leave_the_stream():
    """W_o = 0 and W_gate = 0 (silu(0) = 0): x2 is x, bit for bit."""
    c = _case(B=3, bs=8, Hq=4, D=256, I=128, seed=3)
    c["w_o"] = torch.zeros_like(c["w_o"])
    c["w_gate"] = torch.zeros_like(c["w_gate"])
    x2 = _run(c)
    assert torch.equal(x2.cpu(), c["x"])


def test_layer_tail_batched_shape_sampled():
    """B = 32 sequences x 8 block rows, 32 heads, D = 2560, I = 5120 (the
    batched workload's drafter layer, the configuration the benchmark times);
    six sampled sequences checked."""
    B, bs, Hq, D, I = 32, 8, 32, 2560, 5120
    c = _case(B, bs, Hq, D, I, seed=11, device=DEV)
    x2 = _run(c)
    seqs = np.sort(np.random.default_rng(2).choice(B, 6, replace=False))
    rows = (seqs[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)
    sel = torch.as_tensor(seqs, device=DEV)
    _, ref = oracle.draft_layer_tail(np64(c["x"][torch.as_tensor(rows, device=DEV)]), np64(c["o"][sel]),
                                     *[np64(c[k]) for k in ("w_o", "g_post", "w_gate", "w_up", "w_down")], bf16=True)
    got = x2[torch.as_tensor(rows, device=DEV)]
    assert_close(got, ref, torch.bfloat16, row=D, what="x2")


def _qkv_case(B, bs, Hq, Hkv, D, seed, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed)
    x = (torch.randn(B * bs, D, generator=g, device=device) * 2.0).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(D, generator=g, device=device)).to(torch.bfloat16)
    w = (torch.randn((Hq + 2 * Hkv) * 128, D, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return x, gain, w


def _check_qkv(x, gain, w, B, Hq, Hkv, seqs=None):
    q, kb, vb = dfl.draft_layer_qkv(x, gain, w, B, Hq, Hkv)
    torch.cuda.synchronize()
    bs = x.shape[0] // B
    seqs = np.arange(B) if seqs is None else np.asarray(seqs)
    rows = (seqs[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)
    xs = x[torch.as_tensor(rows, device=x.device)]
    rq, rk, rv = oracle.draft_layer_qkv(np64(xs), np64(gain), np64(w), len(seqs), Hq, Hkv, bf16=True)
    sel = torch.as_tensor(seqs, device=x.device)
    for got, ref, what in ((q[sel], rq, "q"), (kb[sel], rk, "kb"), (vb[sel], rv, "vb")):
        assert_close(got, ref, torch.bfloat16, row=128, what=what)
    return q, kb, vb


@pytest.mark.parametrize("bs", [4, 8, 16])
def test_layer_qkv_small(bs):
    x, gain, w = _qkv_case(B=5, bs=bs, Hq=4, Hkv=2, D=256, seed=bs + 40)
    _check_qkv(x.to(DEV), gain.to(DEV), w.to(DEV), 5, 4, 2)


def test_layer_qkv_null_gain_means_ones():
    x, gain, w = _qkv_case(B=3, bs=8, Hq=4, Hkv=2, D=256, seed=44)
    q, kb, vb = dfl.draft_layer_qkv(x.to(DEV), None, w.to(DEV), 3, 4, 2)
    q1, kb1, vb1 = dfl.draft_layer_qkv(x.to(DEV), torch.ones(256, dtype=torch.bfloat16, device=DEV), w.to(DEV), 3, 4, 2)
    assert torch.equal(q, q1) and torch.equal(kb, kb1) and torch.equal(vb, vb1)


def test_layer_qkv_batched_shape():
    """B = 32 sequences x 8 block rows, D = 2560, 32 query and 8 KV heads (the
    batched workload's drafter layer): every row checked."""
    x, gain, w = _qkv_case(32, 8, 32, 8, 2560, seed=45, device=DEV)
    _check_qkv(x, gain, w, 32, 32, 8)


def test_layer_qkv_high_batch_shape_sampled():
    """B = 128 x 16 block rows (2048 rows, 128-row units): sampled sequences."""
    x, gain, w = _qkv_case(128, 16, 32, 8, 2560, seed=46, device=DEV)
    _check_qkv(x, gain, w, 128, 32, 8, seqs=[0, 9, 64, 127])
