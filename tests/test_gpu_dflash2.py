"""GPU parity of the DFlash2 variants (dflash_block_conv, dflash_draft_topm) against the oracle.

block_conv: bf16 output within the relative Frobenius bound and the per-row
bound (each D-wide row) of the oracle;
identity and one-step-shift kernels reproduce / shift the input bit for bit;
in place equals out of place.  draft_topm: the candidate indices equal the
oracle's exactly (the order is taken on the exact bf16 logits, ties to the
lower index, and bf16 rows carry many ties); log-probabilities, entropies and
path scores within 1e-4; uniform rows give the closed form.
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _conv_case(B, bs, D, k, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(B * bs, D, generator=g).to(torch.bfloat16)
    w = (0.5 * torch.randn(k, D, generator=g)).to(torch.bfloat16)
    bias = (0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    return h, w, bias


@pytest.mark.parametrize("bs,k", [(4, 3), (8, 3), (8, 5), (16, 5), (3, 8)])
@pytest.mark.parametrize("with_bias,residual", [(False, False), (True, True)])
def test_block_conv_matches_oracle(bs, k, with_bias, residual):
    h, w, bias = _conv_case(5, bs, 2560, k, seed=bs * 10 + k)
    b = bias if with_bias else None
    out = dfl.block_conv(h.to(DEV), w.to(DEV), b.to(DEV) if b is not None else None, bs, residual=residual)
    torch.cuda.synchronize()
    ref = oracle.round_to_bf16(oracle.block_conv(np64(h), np64(w), np64(b) if b is not None else None, bs,
                                                 residual=residual))
    assert_close(out, ref, torch.bfloat16, row=h.shape[1], what="conv")
    # in place gives the same bytes
    hd = h.to(DEV).clone()
    dfl.block_conv(hd, w.to(DEV), b.to(DEV) if b is not None else None, bs, residual=residual, out=hd)
    torch.cuda.synchronize()
    assert torch.equal(hd, out)


def test_block_conv_identity_and_shift_are_exact():
    h, _, _ = _conv_case(4, 8, 256, 3, seed=1)
    hd = h.to(DEV)
    ident = torch.zeros(3, 256, dtype=torch.bfloat16)
    ident[0] = 1.0
    assert torch.equal(dfl.block_conv(hd, ident.to(DEV), None, 8), hd)
    shift = torch.zeros(3, 256, dtype=torch.bfloat16)
    shift[1] = 1.0
    out = dfl.block_conv(hd, shift.to(DEV), None, 8).cpu()
    for r in range(h.shape[0]):
        expect = torch.zeros(256, dtype=torch.bfloat16) if r % 8 == 0 else h[r - 1]
        assert torch.equal(out[r], expect), r


def _check_topm(logits, m, T, lam, rows=None):
    idx, logp, ent, score = dfl.draft_topm(logits, m, T, lam)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    l64 = np64(logits[sel])
    ri, rl, re, rs = oracle.draft_topm(l64, m, T, lam)
    np.testing.assert_array_equal(idx[sel].cpu().numpy(), ri)
    np.testing.assert_allclose(logp[sel].cpu().numpy(), rl, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(ent[sel].cpu().numpy(), re, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(score[sel].cpu().numpy(), rs, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("m", [1, 4, 8])
def test_draft_topm_small(m):
    g = torch.Generator().manual_seed(m)
    V = 40000   # three chunks of 16384, the last one ragged; bf16 rows carry many exact ties
    logits = (3.0 * torch.randn(3, 7, V, generator=g)).to(torch.bfloat16).to(DEV)
    _check_topm(logits, m, 0.7, 0.3)


def test_draft_topm_uniform_rows_and_masked_logits():
    V, m = 16384 + 8, 5
    logits = torch.zeros(2, 3, V, dtype=torch.bfloat16, device=DEV)
    idx, logp, ent, score = dfl.draft_topm(logits, m, 1.0, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), torch.arange(m, dtype=torch.int32).expand(2, 3, m))
    np.testing.assert_allclose(logp.cpu().numpy(), -np.log(V), rtol=1e-5)
    np.testing.assert_allclose(ent.cpu().numpy(), np.log(V), rtol=1e-5)
    # -inf logits have zero probability and are chosen last
    lm = logits.clone()
    lm[:, :, : V // 2] = float("-inf")
    _check_topm(lm, m, 1.0, 0.5)


def test_draft_topm_batched_shape_sampled():
    """The batched workload's draft logits: B = 32 sequences x 7 proposal rows,
    V = 262144, m = 8; two sequences checked against the oracle."""
    g = torch.Generator(device=DEV).manual_seed(21)
    logits = (3.0 * torch.randn(32, 7, 262144, generator=g, device=DEV)).to(torch.bfloat16)
    _check_topm(logits, 8, 1.0, 0.2, rows=torch.tensor([3, 30], device=DEV))


def test_draft_topm_rows_with_fewer_finite_logits_than_m():
    """Fewer than m finite logits: the -inf logits follow them, lowest index first."""
    V, m = 16384 + 8, 8
    logits = torch.full((1, 2, V), float("-inf"), dtype=torch.bfloat16, device=DEV)
    logits[0, 0, 100] = 1.0
    logits[0, 0, 7000] = 2.0
    logits[0, 0, 16390] = 2.0
    idx, logp, ent, score = dfl.draft_topm(logits, m, 1.0, 0.0)
    torch.cuda.synchronize()
    ri, rl, re, rs = oracle.draft_topm(np64(logits), m, 1.0, 0.0)
    np.testing.assert_array_equal(idx[0, 0].cpu().numpy(), ri[0, 0])
    np.testing.assert_allclose(logp[0, 0, :3].cpu().numpy(), rl[0, 0, :3], rtol=1e-5)
    assert torch.all(torch.isinf(logp[0, 0, 3:]))
    # the all -inf row: indices in order, ln P = -inf, entropy 0 (as the oracle)
    np.testing.assert_array_equal(idx[0, 1].cpu().numpy(), ri[0, 1])
    assert torch.all(torch.isneginf(logp[0, 1])) and ent[0, 1].item() == 0.0
