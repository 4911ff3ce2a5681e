"""GPU parity of dflash_draft_head against the oracle.

The logits must match the oracle's (final RMSNorm, bf16 rows, product, bf16
rounding) within the relative Frobenius bound and the per-row bound (each
vocabulary row); the draft tokens must equal the
oracle's exponential race (argmax at T = 0) taken on the GPU's own logits --
the integer decision is taken on the same stored bf16 values on both sides --
except in rows the oracle flags as near-ties.
"""
import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle
from helpers import assert_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, R, D, V, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(B * R, D, generator=g) * 2.0).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    w = (torch.randn(V, D, generator=g) * 0.05).to(torch.bfloat16)
    return x, gain, w


def _check(x, gain, w, R, T, seed, cycle, rows=None):
    logits, tok = dfl.draft_head(x.to(DEV), gain.to(DEV), w.to(DEV), R, T, seed, cycle)
    torch.cuda.synchronize()
    M = x.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    ref = oracle.draft_head(np64(x[rows]), np64(gain), np64(w), bf16=True)
    got = logits[torch.as_tensor(rows, device=DEV)].float().cpu().numpy()
    assert_close(got, ref, torch.bfloat16, row=w.shape[0], what="logits")
    assert (got == ref).mean() > 0.98      # bf16 values agree except at rounding edges
    # the draw, taken by the oracle on the GPU's stored logits
    b, k = rows // R, rows % R
    toks = tok.cpu().numpy()[rows]
    for i, row in enumerate(rows):
        tk, nr = _race_row(got[i][None, None, :], T, seed, cycle, b[i], k[i])
        assert toks[i] == tk or nr, (row, toks[i], tk)
    return logits, tok


def _race_row(z, T, seed, cycle, b, k):
    """oracle.draft_sample for one (sequence b, proposal row k)."""
    tok, near = oracle.draft_sample(z, T, seed, cycle, seq_ids=[b], row_ids=[k])
    return int(tok[0, 0]), bool(near[0, 0])


@pytest.mark.parametrize("T", [0.0, 1.0, 0.6])
def test_draft_head_small(T):
    B, R, D, V = 3, 7, 256, 4096
    x, gain, w = _case(B, R, D, V, seed=5)
    _check(x, gain, w, R, T, seed=11, cycle=3)


def test_draft_head_ragged_rows_and_short_vocab():
    """M = 5 rows (less than one 128-row tile), V = 128 (one column tile)."""
    x, gain, w = _case(5, 1, 128, 128, seed=6)
    _check(x, gain, w, 1, 1.0, seed=2, cycle=9)


def test_draft_head_full_size_sampled():
    """B = 32 sequences x 7 proposal rows, D = 2560, V = 262144 (the batched
    workload's drafter head, the launch configuration the benchmark times);
    24 sampled rows checked."""
    B, R, D, V = 32, 7, 2560, 262144
    g = torch.Generator(device=DEV).manual_seed(7)
    x = (torch.randn(B * R, D, generator=g, device=DEV) * 2.0).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(torch.bfloat16)
    w = (torch.randn(V, D, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    rows = np.sort(np.random.default_rng(3).choice(B * R, 24, replace=False))
    logits, tok = dfl.draft_head(x, gain, w, R, 1.0, 1234, 17)
    torch.cuda.synchronize()
    ref = oracle.draft_head(np64(x[torch.as_tensor(rows, device=DEV)]), np64(gain), np64(w), bf16=True)
    got = logits[torch.as_tensor(rows, device=DEV)].float().cpu().numpy()
    assert_close(got, ref, torch.bfloat16, row=V, what="logits")
    toks = tok.cpu().numpy()
    for i, row in enumerate(rows):
        tk, nr = _race_row(got[i][None, None, :], 1.0, 1234, 17, row // R, row % R)
        assert toks[row] == tk or nr, (row, toks[row], tk)


def test_draft_head_tokens_follow_the_softmax():
    """Many cycles of a tiny vocabulary (V = 128): the GPU's draws of one row
    follow softmax(logits / T) (chi-square on the 8 most likely tokens + rest)."""
    from scipy import stats
    x, gain, w = _case(1, 1, 128, 128, seed=8)
    w = (w.float() * 20).to(torch.bfloat16)       # a peaked distribution
    T, N = 0.8, 3000
    xd, gd, wd = x.to(DEV), gain.to(DEV), w.to(DEV)
    counts = np.zeros(128)
    logits = None
    for c in range(N):
        logits, tok = dfl.draft_head(xd, gd, wd, 1, T, 99, c)
        counts[int(tok[0])] += 1
    z = logits[0].float().cpu().numpy().astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    top = np.argsort(-p)[:8]
    obs = np.append(counts[top], N - counts[top].sum())
    exp = np.append(N * p[top], N * (1 - p[top].sum()))
    keep = exp > 5
    chi2 = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-3, (obs, exp)
