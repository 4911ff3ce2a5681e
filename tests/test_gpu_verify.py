"""GPU parity of dflash_verify against the oracle.

Accepted lengths and tokens must match the oracle exactly, except in
sequences where the oracle flags a near-tie (a uniform within 1e-6 of alpha,
or a draw threshold within 1e-6 of a cumulative-mass edge); the count of such
sequences is reported.  Philox words must match bit for bit.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import block_speculative_decoding_gb300 as dfl
import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _mk_logits(B, bs, V, dtype, seed, noise=1.0, std=3.0):
    g = torch.Generator().manual_seed(seed)
    lt = torch.randn(B, bs, V, generator=g) * std
    ld = lt[:, :bs - 1] + torch.randn(B, bs - 1, V, generator=g) * noise
    return lt.to(dtype), ld.to(dtype)


def _greedy_tokens(lt, seed):
    """Draft tokens that match the target argmax for a random prefix length."""
    g = torch.Generator().manual_seed(seed)
    B, bs, V = lt.shape
    am = lt.float().argmax(-1)[:, :bs - 1]
    rnd = torch.randint(0, V, (B, bs - 1), generator=g)
    m = torch.randint(0, bs, (B, 1), generator=g)
    k = torch.arange(bs - 1)[None, :]
    return torch.where(k < m, am, rnd).to(torch.int32)


def run_and_compare(lt, ld, x, T, seed, cycle, seq_ids=None, gpu_out=None):
    if gpu_out is None:
        acc, out = dfl.verify(lt.to(DEV), None if ld is None else ld.to(DEV), x.to(DEV), T, seed, cycle)
        acc, out = acc.cpu().numpy(), out.cpu().numpy()
    else:
        acc, out = gpu_out
    ref = oracle.verify(lt.double().numpy(), None if ld is None else ld.double().numpy(), x.numpy(), T, seed,
                        cycle, seq_ids=seq_ids)
    mism = (acc != ref.accepted_len) | np.any(out != ref.out_tokens, axis=1)
    bad = mism & ~ref.near_tie
    assert not bad.any(), "mismatch at sequences %s: gpu %s %s oracle %s %s" % (
        np.nonzero(bad)[0][:5], acc[bad][:5], out[bad][:5], ref.accepted_len[bad][:5], ref.out_tokens[bad][:5])
    return int(mism.sum()), int(ref.near_tie.sum()), ref


def test_philox_matches_oracle_bit_for_bit():
    n = 1 << 20
    g = torch.Generator().manual_seed(0)
    ctr = torch.randint(-2**31, 2**31, (n, 4), generator=g, dtype=torch.int64).to(torch.int32)
    ctr[:4] = torch.tensor([[0, 0, 0, 0], [-1, -1, -1, -1], [0x243f6a88, 0x85a308d3 - 2**32, 0x13198a2e, 0x03707344],
                            [7, 1, 2, 3]], dtype=torch.int32)
    k0, k1 = 0xA4093822, 0x299F31D0
    out = dfl.philox4x32_10(ctr.to(DEV), k0, k1).cpu().numpy().view(np.uint32)
    c = ctr.numpy().view(np.uint32).astype(np.uint64)
    ref = oracle.philox4x32_10((c[:, 0], c[:, 1], c[:, 2], c[:, 3]), (k0, k1))
    for w in range(4):
        assert np.array_equal(out[:, w], ref[w])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [4096, 1000, 40000])
@pytest.mark.parametrize("bs", [1, 2, 8, 16])
@pytest.mark.parametrize("T", [0.0, 1.0, 0.7])
def test_verify_small_grid(dtype, V, bs, T):
    B = 8
    lt, ld = _mk_logits(B, bs, V, dtype, seed=V + bs)
    if T == 0.0:
        x = _greedy_tokens(lt, seed=bs)
    else:
        x = workloads.draft_tokens(ld, T, seed=7)
    run_and_compare(lt, ld, x, T, seed=1234 + bs, cycle=V)


@pytest.mark.parametrize("V", [600000, 600001])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_verify_rows_longer_than_the_register_paths(V, T):
    """Rows of more than 32 stats chunks and 256 residual segments: the
    normalisers merge through the looped path and the draw scans its segment
    masses 32 at a time; V = 600001 also takes the scalar (unvectorised) loads."""
    B, bs = 3, 4
    lt, ld = _mk_logits(B, bs, V, torch.bfloat16, seed=V % 1000 + 3)
    x = _greedy_tokens(lt, seed=5) if T == 0.0 else workloads.draft_tokens(ld, T, seed=9)
    run_and_compare(lt, ld, x, T, seed=77, cycle=2)


def test_verify_identical_rows_accept_everything():
    B, bs, V = 16, 8, 50000
    lt, _ = _mk_logits(B, bs, V, torch.bfloat16, seed=3)
    ld = lt[:, :bs - 1].clone()
    x = workloads.draft_tokens(ld, 1.0, seed=4)
    acc, out = dfl.verify(lt.to(DEV), ld.to(DEV), x.to(DEV), 1.0, 9, 0)
    assert torch.all(acc.cpu() == bs - 1)
    assert torch.all(out.cpu() >= 0)
    run_and_compare(lt, ld, x, 1.0, 9, 0)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_verify_batched_full_size(T):
    cfg = workloads.BATCHED
    lt, ld = workloads.logits(cfg, "cpu")
    x = workloads.draft_tokens(ld, T, seed=11)
    mism, ties, ref = run_and_compare(lt, ld, x, T, seed=2024, cycle=17)
    for b in workloads.all_accept_sequences(cfg):
        if T > 0:
            assert ref.accepted_len[b] == cfg.bs - 1
    print("batched T=%g: mismatches %d, near-tie sequences %d, mean tau %.3f" % (
        T, mism, ties, ref.accepted_len.mean() + 1))


@pytest.mark.parametrize("bs,sigma", [(16, 0.25), (4, 4.0)])
def test_verify_high_batch_sampled(bs, sigma):
    cfg = workloads.high_batch(bs, sigma)
    lt, ld = workloads.logits(cfg, DEV)
    x = workloads.draft_tokens(ld, 1.0, seed=5)
    acc, out = dfl.verify(lt, ld, x, 1.0, 77, 3)
    sel = np.array([0, 1, 37, 64, 90, 127])
    acc_s, out_s = acc.cpu().numpy()[sel], out.cpu().numpy()[sel]
    run_and_compare(lt[sel].cpu(), ld[sel].cpu(), x[sel].cpu(), 1.0, 77, 3, seq_ids=sel, gpu_out=(acc_s, out_s))


def test_verify_bad_token_raises_status_and_rejects():
    B, bs, V = 4, 8, 4096
    lt, ld = _mk_logits(B, bs, V, torch.float32, seed=8)
    ld[:] = lt[:, :bs - 1]                   # everything would be accepted ...
    x = workloads.draft_tokens(ld, 1.0, seed=1)
    x[2, 3] = V + 5                          # ... but sequence 2 has an invalid token at row 3
    dfl.read_device_status()
    acc, out = dfl.verify(lt.to(DEV), ld.to(DEV), x.to(DEV), 1.0, 5, 5)
    flags = dfl.read_device_status()
    assert flags & dfl.DEV_BAD_TOKEN
    acc = acc.cpu().numpy()
    assert acc[2] == 3 and all(acc[b] == bs - 1 for b in (0, 1, 3))


def test_verify_gpu_output_follows_target_distribution():
    # Many independent sequences of the same tiny problem: the emitted token at
    # each reached position must be distributed as p at that position.
    B, bs, V = 60000, 4, 16
    g = torch.Generator().manual_seed(21)
    lt1 = torch.randn(bs, V, generator=g) * 1.5
    ld1 = lt1[:bs - 1] + torch.randn(bs - 1, V, generator=g)
    lt = lt1.expand(B, bs, V).contiguous()
    ld = ld1.expand(B, bs - 1, V).contiguous()
    x = workloads.draft_tokens(ld, 1.0, seed=22)
    acc, out = dfl.verify(lt.to(DEV), ld.to(DEV), x.to(DEV), 1.0, 123, 1)
    acc, out = acc.cpu().numpy(), out.cpu().numpy()
    p = torch.softmax(lt1.double(), -1).numpy()
    for k in range(bs):
        reached = acc >= k
        obs = np.bincount(out[reached, k], minlength=V)
        assert stats.chisquare(obs, p[k] * reached.sum()).pvalue > 1e-4
