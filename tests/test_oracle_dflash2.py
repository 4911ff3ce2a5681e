"""Pins of the DFlash2-variant oracle functions: block_conv, draft_topm, path_score.

block_conv is tied to kernels whose result is known without the formula
(identity, a pure one-step shift, bias only, all-ones input giving cumulative
weight sums), to linearity and to the residual form.  draft_topm is tied to
closed forms (uniform logits, one raised logit), to invariances (adding a
constant to a row, temperature as a logit scale), to the tie rule and, for the
path score, to brute-force enumeration of every candidate path.
"""
import itertools

import numpy as np

import oracle


def _h(B=3, bs=4, D=5, seed=0):
    return np.random.default_rng(seed).standard_normal((B * bs, D))


def test_conv_identity_shift_and_bias():
    h = _h()
    D = h.shape[1]
    ident = np.zeros((3, D))
    ident[0] = 1.0
    np.testing.assert_array_equal(oracle.block_conv(h, ident, None, 4), h)
    shift = np.zeros((3, D))
    shift[1] = 1.0
    out = oracle.block_conv(h, shift, None, 4)
    for r in range(h.shape[0]):
        if r % 4 == 0:
            np.testing.assert_array_equal(out[r], 0.0)      # nothing leaks from the previous sequence
        else:
            np.testing.assert_array_equal(out[r], h[r - 1])
    bias = np.arange(D, dtype=float)
    np.testing.assert_array_equal(oracle.block_conv(h, np.zeros((5, D)), bias, 4), np.tile(bias, (h.shape[0], 1)))


def test_conv_of_ones_is_the_cumulative_weight_sum():
    bs, D = 8, 3
    w = np.random.default_rng(1).standard_normal((5, D))
    out = oracle.block_conv(np.ones((2 * bs, D)), w, None, bs)
    for r in range(2 * bs):
        t = r % bs
        np.testing.assert_allclose(out[r], w[: min(t, 4) + 1].sum(axis=0), rtol=1e-14)


def test_conv_is_linear_and_residual_adds_the_input():
    h1, h2 = _h(seed=2), _h(seed=3)
    w = np.random.default_rng(4).standard_normal((3, h1.shape[1]))
    a = oracle.block_conv(2.0 * h1 - 3.0 * h2, w, None, 4)
    b = 2.0 * oracle.block_conv(h1, w, None, 4) - 3.0 * oracle.block_conv(h2, w, None, 4)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.block_conv(h1, w, None, 4, residual=True),
                               h1 + oracle.block_conv(h1, w, None, 4), rtol=0, atol=0)


def test_topm_uniform_logits():
    V, m = 50, 4
    idx, logp, ent, best = oracle.draft_topm(np.zeros((2, 3, V)), m, 0.7, 0.25)
    np.testing.assert_array_equal(idx, np.broadcast_to(np.arange(m), idx.shape))   # ties: lower index first
    np.testing.assert_allclose(logp, -np.log(V), rtol=1e-14)
    np.testing.assert_allclose(ent, np.log(V), rtol=1e-14)
    np.testing.assert_allclose(best, 3 * (-np.log(V)) + 0.25 * 3 * np.log(V), rtol=1e-13)


def test_topm_one_raised_logit_closed_form():
    V, a, T = 20, 3.0, 1.0
    l = np.zeros((1, 1, V))
    l[0, 0, 7] = a
    idx, logp, ent, _ = oracle.draft_topm(l, 2, T, 0.0)
    z = np.exp(a) + V - 1
    p1, p0 = np.exp(a) / z, 1.0 / z
    assert idx[0, 0, 0] == 7 and idx[0, 0, 1] == 0
    np.testing.assert_allclose(logp[0, 0], [a - np.log(z), -np.log(z)], rtol=1e-13)
    np.testing.assert_allclose(ent[0, 0], -(p1 * np.log(p1) + (V - 1) * p0 * np.log(p0)), rtol=1e-13)


def test_topm_invariances():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((2, 3, 30)) * 3
    i1, lp1, e1, b1 = oracle.draft_topm(l, 5, 0.5, 0.3)
    i2, lp2, e2, b2 = oracle.draft_topm(l + 100.0, 5, 0.5, 0.3)        # a constant per row changes nothing
    i3, lp3, e3, b3 = oracle.draft_topm(l / 0.5, 5, 1.0, 0.3)          # T is a scale of the logits
    for i, lp, e, b in ((i2, lp2, e2, b2), (i3, lp3, e3, b3)):
        np.testing.assert_array_equal(i, i1)
        np.testing.assert_allclose(lp, lp1, rtol=1e-10)
        np.testing.assert_allclose(e, e1, rtol=1e-10)
        np.testing.assert_allclose(b, b1, rtol=1e-10)


def test_best_path_by_enumerating_every_path():
    rng = np.random.default_rng(6)
    B, R, V, m, lam = 2, 3, 6, 3, 0.4
    l = rng.standard_normal((B, R, V))
    idx, logp, ent, best = oracle.draft_topm(l, m, 0.8, lam)
    for b in range(B):
        scores = {c: oracle.path_score(logp[b:b + 1], ent[b:b + 1], np.array([c]), lam)[0]
                  for c in itertools.product(range(m), repeat=R)}
        top = max(scores, key=scores.get)
        assert top == (0,) * R
        np.testing.assert_allclose(scores[top], best[b], rtol=1e-13)
    # the candidates are the m largest logits of each row
    for b in range(B):
        for r in range(R):
            assert set(idx[b, r]) == set(np.argsort(-l[b, r], kind="stable")[:m])


def test_topm_zero_probability_tokens():
    """-inf logits have probability 0: they add nothing to the entropy (0 ln 0 = 0) and come last."""
    l = np.zeros((1, 1, 8))
    l[0, 0, :4] = -np.inf
    idx, logp, ent, _ = oracle.draft_topm(l, 5, 1.0, 0.0)
    np.testing.assert_allclose(ent[0, 0], np.log(4), rtol=1e-14)
    assert list(idx[0, 0]) == [4, 5, 6, 7, 0] and logp[0, 0, 4] == -np.inf


def test_topm_row_of_only_minus_inf():
    """A row without probability mass: ln P = -inf for its candidates, entropy 0, no NaN."""
    l = np.full((1, 2, 6), -np.inf)
    l[0, 0, 2] = 1.0
    idx, logp, ent, best = oracle.draft_topm(l, 3, 1.0, 0.5)
    assert list(idx[0, 1]) == [0, 1, 2] and np.all(logp[0, 1] == -np.inf) and ent[0, 1] == 0.0
    assert logp[0, 0, 0] == 0.0 and not np.isnan(best).any()
