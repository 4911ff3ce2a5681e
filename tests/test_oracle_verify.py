"""Pins for the oracle's speculative verification.

The pages fix what verification must achieve, not how: the output follows the
target distribution, identical p and q accept the whole block, greedy decoding
accepts the argmax-prefix match, and the cycle emits at most bs tokens.  These
tests check those facts, plus the closed forms they imply:

  P(output = t_0..t_n, n accepted) = prod_{k<n} min(p_k, q_k)(t_k)
                                     * ((p_n - q_n)_+(t_n) if n < bs-1 else p_{bs-1}(t_n))
  E[tau] = 1 + sum_{k=1}^{bs-1} prod_{j<k} beta_j,  beta_j = sum_x min(p_j, q_j)(x)

(the accepted mass q*a = min(p, q) and the residual [p - q]_+ are stated in
"Why exact verification preserves the target" of the E4B page).
"""
import itertools

import numpy as np
import pytest
from scipy import stats

import oracle


def _softmax(l):
    e = np.exp(l - l.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def _draft_from_q(ld, T, rng):
    q = _softmax(ld / T)
    B, R, V = q.shape
    c = np.cumsum(q, -1)
    u = rng.random((B, R, 1))
    return np.minimum((c < u * c[..., -1:]).sum(-1), V - 1)


def test_identical_p_and_q_accept_whole_block():
    rng = np.random.default_rng(0)
    B, bs, V = 64, 8, 50
    lt = rng.normal(0, 3, size=(B, bs, V))
    ld = lt[:, :bs - 1].copy()
    x = _draft_from_q(ld, 1.0, rng)
    r = oracle.verify(lt, ld, x, 1.0, seed=5, cycle=0)
    assert np.all(r.accepted_len == bs - 1)
    assert np.all(r.out_tokens[:, :bs - 1] == x)
    assert np.all(r.out_tokens >= 0)           # tau = bs: all 8 slots filled


def test_greedy_constructed_prefix():
    B, bs, V = 6, 5, 9
    lt = np.zeros((B, bs, V))
    am = np.array([[1, 2, 3, 4, 5], [0, 0, 0, 0, 8], [7, 7, 7, 7, 7],
                   [3, 1, 4, 1, 5], [2, 7, 1, 8, 2], [8, 8, 8, 8, 8]])
    for b, k in itertools.product(range(B), range(bs)):
        lt[b, k, am[b, k]] = 4.0
    lt[5, 0, 2] = 4.0                          # tie: argmax of row 0 is index 2, not 8
    x = np.array([[1, 2, 3, 4], [0, 0, 0, 0], [0, 7, 7, 7], [3, 1, 0, 1], [2, 7, 1, 8], [8, 8, 8, 8]])
    r = oracle.verify(lt, None, x, 0.0, seed=1, cycle=0)
    assert r.accepted_len.tolist() == [4, 4, 0, 2, 4, 0]
    assert r.out_tokens[0].tolist() == [1, 2, 3, 4, 5]
    assert r.out_tokens[1].tolist() == [0, 0, 0, 0, 8]
    assert r.out_tokens[2].tolist() == [7, -1, -1, -1, -1]
    assert r.out_tokens[3].tolist() == [3, 1, 4, -1, -1]
    assert r.out_tokens[5].tolist() == [2, -1, -1, -1, -1]


def test_categorical_draw_bins():
    from oracle.dflash_oracle import _categorical_draw
    w = np.array([[0.2, 0.3, 0.5, 0.0], [0.2, 0.3, 0.5, 0.0], [0.2, 0.3, 0.5, 0.0], [0.0, 0.5, 0.0, 0.5]])
    y, _ = _categorical_draw(w, np.array([0.1, 0.25, 0.6, 0.5]))
    assert y.tolist() == [0, 1, 2, 3]


def test_boundary_band_is_on_the_uniforms_scale():
    """A draw is a boundary case when its uniform lies within 1e-6 of a value
    at which the drawn index would change: a bin edge C_y / S of the
    normalised cumulative mass.  With total mass S = 0.25 the edge of
    [0.125, 0.125] sits at v = 0.5: v = 0.5 - 5e-7 is flagged, v = 0.5 - 2e-6
    is not (its distance in unnormalised mass, 5e-7, is not the criterion),
    and with S = 1 the same two uniforms behave the same way."""
    from oracle.dflash_oracle import _categorical_draw
    for S in (0.25, 1.0):
        w = np.array([[S / 2, S / 2]] * 4)
        y, tie = _categorical_draw(w, np.array([0.5 - 5e-7, 0.5 - 2e-6, 0.5 + 5e-7, 0.5 + 2e-6]))
        assert y.tolist() == [0, 0, 1, 1]
        assert tie.tolist() == [True, False, True, False], S
    # the acceptance decision: |u - alpha| < 1e-6 flags the sequence
    lt = np.log(np.array([[[0.5, 0.5], [0.5, 0.5]]]))
    ld = np.log(np.array([[[0.25, 0.75]]]))               # alpha = min(1, 0.5 / 0.75) = 2/3 for token 1
    for seed in range(200):
        u = oracle.verify_uniforms(seed, 0, 0, np.array([0]))[0][0]
        r = oracle.verify(lt, ld, np.array([[1]]), 1.0, seed, 0)
        assert r.accepted_len[0] == (1 if u < 2.0 / 3.0 else 0)
        if abs(u - 2.0 / 3.0) >= 1e-6 and r.accepted_len[0] == 1:
            assert not r.near_tie[0]       # accepted, bonus draw from p = [0.5, 0.5]: edge at v = 0.5


def _mc_case(seed, B, bs, V, sharp=1.5):
    rng = np.random.default_rng(seed)
    lt1 = rng.normal(0, sharp, size=(bs, V))
    ld1 = lt1[:bs - 1] + rng.normal(0, 1.0, size=(bs - 1, V))
    lt = np.broadcast_to(lt1, (B, bs, V))
    ld = np.broadcast_to(ld1, (B, bs - 1, V))
    x = _draft_from_q(np.array(ld), 1.0, rng)
    return lt, ld, x, _softmax(lt1), _softmax(ld1)


def test_output_distribution_equals_target_per_position():
    B, bs, V = 200000, 4, 8
    lt, ld, x, p, q = _mc_case(11, B, bs, V)
    r = oracle.verify(lt, ld, x, 1.0, seed=123, cycle=9)
    assert np.all((r.accepted_len >= 0) & (r.accepted_len <= bs - 1))
    for k in range(bs):
        reached = r.accepted_len >= k
        tok = r.out_tokens[reached, k]
        assert np.all(tok >= 0)
        obs = np.bincount(tok, minlength=V)
        exp = p[k] * reached.sum()
        chi = stats.chisquare(obs, exp)
        assert chi.pvalue > 1e-3, (k, chi)


def test_exact_enumeration_small_vocab():
    B, bs, V = 300000, 3, 3
    lt, ld, x, p, q = _mc_case(12, B, bs, V, sharp=1.0)
    r = oracle.verify(lt, ld, x, 1.0, seed=77, cycle=1)
    probs, counts = [], []
    for n in range(bs):
        for toks in itertools.product(range(V), repeat=n + 1):
            pr = 1.0
            for k in range(n):
                pr *= min(p[k, toks[k]], q[k, toks[k]])
            pr *= max(0.0, p[n, toks[n]] - q[n, toks[n]]) if n < bs - 1 else p[n, toks[n]]
            sel = (r.accepted_len == n)
            for k in range(n + 1):
                sel &= r.out_tokens[:, k] == toks[k]
            probs.append(pr)
            counts.append(int(sel.sum()))
    probs = np.array(probs)
    counts = np.array(counts)
    assert abs(probs.sum() - 1.0) < 1e-12
    assert counts.sum() == B
    keep = probs > 0
    assert counts[~keep].sum() == 0
    chi = stats.chisquare(counts[keep], probs[keep] * B)
    assert chi.pvalue > 1e-3, chi


@pytest.mark.parametrize("bs", [3, 8])
def test_mean_acceptance_length_closed_form(bs):
    B, V = 100000, 12
    lt, ld, x, p, q = _mc_case(20 + bs, B, bs, V, sharp=2.0)
    r = oracle.verify(lt, ld, x, 1.0, seed=4, cycle=bs)
    tau = r.accepted_len + 1
    beta = np.minimum(p[:bs - 1], q).sum(-1)
    expect = 1.0 + sum(np.prod(beta[:k]) for k in range(1, bs))
    assert abs(tau.mean() - expect) < 4 * tau.std() / np.sqrt(B)
    assert tau.min() >= 1 and tau.max() <= bs


def test_temperature_scales_both_rows():
    # Dividing logits by T must equal running at T = 1 on logits / T.
    rng = np.random.default_rng(30)
    B, bs, V = 256, 6, 40
    lt = rng.normal(0, 3, size=(B, bs, V))
    ld = lt[:, :bs - 1] + rng.normal(0, 1, size=(B, bs - 1, V))
    x = _draft_from_q(ld, 0.7, rng)
    a = oracle.verify(lt, ld, x, 0.7, seed=9, cycle=2)
    b = oracle.verify(lt / 0.7, ld / 0.7, x, 1.0, seed=9, cycle=2)
    assert np.array_equal(a.accepted_len, b.accepted_len)
    assert np.array_equal(a.out_tokens, b.out_tokens)
