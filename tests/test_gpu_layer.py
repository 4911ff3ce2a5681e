"""GPU parity of dflash_draft_layer_tail against the oracle.

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
