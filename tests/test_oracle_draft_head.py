"""Pins for the oracle's drafter head: final RMSNorm + LM head, and the
exponential-race draft sampler.

Each test checks a closed form, an invariant, a constructed case or a
distribution, not the oracle's own formula retyped.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def test_draft_head_matches_loops_and_the_norm_closed_form():
    rng = np.random.default_rng(0)
    R, D, V = 3, 8, 11
    x = rng.normal(size=(R, D)) * 3.0
    g = 1 + 0.1 * rng.normal(size=D)
    w = rng.normal(size=(V, D))
    z = oracle.draft_head(x, g, w, eps=1e-6)
    for r in range(R):
        ms = sum(v * v for v in x[r]) / D
        h = [x[r][i] / np.sqrt(ms + 1e-6) * g[i] for i in range(D)]
        for t in range(V):
            assert abs(z[r, t] - sum(h[i] * w[t, i] for i in range(D))) < 1e-10
    # constant gain c: every normalised row has root-mean-square |c|; with the
    # identity as head the logits are that row
    c = -1.7
    zi = oracle.draft_head(x, np.full(D, c), np.eye(D), eps=0.0)
    np.testing.assert_allclose(np.sqrt((zi ** 2).mean(axis=1)), abs(c), rtol=1e-12)
    # bf16 storage points: the logits are bfloat16 values
    zb = oracle.draft_head(x, g, w, bf16=True)
    np.testing.assert_array_equal(zb, oracle.round_to_bf16(zb))


def test_greedy_draft_is_the_first_argmax():
    z = np.zeros((1, 2, 7))
    z[0, 0, [2, 5]] = 3.0           # tie: lowest index
    z[0, 1, 6] = 1.0
    tok, near = oracle.draft_sample(z, 0.0, seed=1, cycle=0)
    assert tok.tolist() == [[2, 6]]
    assert near.tolist() == [[True, False]]


def test_temperature_scales_the_logits():
    z = np.random.default_rng(2).normal(size=(2, 3, 50)) * 4
    for T in (0.3, 1.0, 2.5):
        a, _ = oracle.draft_sample(z, T, seed=9, cycle=4)
        b, _ = oracle.draft_sample(z / T, 1.0, seed=9, cycle=4)
        np.testing.assert_array_equal(a, b)


def test_race_uniforms_are_in_the_open_unit_interval_and_distinct_per_row():
    u = oracle.draft_race_uniforms(seed=5, cycle=11, b=3, k=2, V=4096)
    assert u.min() > 0.0 and u.max() <= 1.0
    assert abs(u.mean() - 0.5) < 0.02 and abs(u.var() - 1 / 12) < 0.01
    v = oracle.draft_race_uniforms(seed=5, cycle=11, b=3, k=1, V=4096)
    w = oracle.draft_race_uniforms(seed=5, cycle=12, b=3, k=2, V=4096)
    assert not np.array_equal(u, v) and not np.array_equal(u, w)
    # a prefix of the vocabulary draws the same uniforms as the whole row
    np.testing.assert_array_equal(oracle.draft_race_uniforms(5, 11, 3, 2, 10), u[:10])


def test_race_draws_follow_the_softmax():
    """Many cycles of one row: the empirical distribution of the drawn token
    is softmax(logits / T) (chi-square)."""
    V, T, N = 6, 0.7, 6000
    z = np.array([0.3, -1.0, 1.2, 0.0, 2.0, -0.4])
    p = np.exp(z / T - (z / T).max())
    p /= p.sum()
    counts = np.zeros(V)
    zz = np.broadcast_to(z, (1, 1, V))
    for c in range(N):
        tok, _ = oracle.draft_sample(zz, T, seed=77, cycle=c)
        counts[tok[0, 0]] += 1
    chi2 = ((counts - N * p) ** 2 / (N * p)).sum()
    assert stats.chi2.sf(chi2, V - 1) > 1e-3, (counts, N * p)


def test_a_subset_of_rows_draws_what_the_whole_batch_draws():
    z = np.random.default_rng(4).normal(size=(3, 4, 40))
    full, _ = oracle.draft_sample(z, 0.9, seed=3, cycle=8)
    part, _ = oracle.draft_sample(z[2:3, 1:3], 0.9, seed=3, cycle=8, seq_ids=[2], row_ids=[1, 2])
    np.testing.assert_array_equal(part, full[2:3, 1:3])


def _tail_case(seed, B=2, Hq=4, bs=3, hd=4, D=8, I=6):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(B * bs, D)), o=rng.normal(size=(B, Hq, bs, hd)),
                w_o=rng.normal(size=(D, Hq * hd)) * 0.3, g_post=1 + 0.1 * rng.normal(size=D),
                w_gate=rng.normal(size=(I, D)), w_up=rng.normal(size=(I, D)), w_down=rng.normal(size=(D, I)) * 0.3)


def test_layer_tail_matches_loops():
    c = _tail_case(0)
    x1, x2 = oracle.draft_layer_tail(**c)
    B, Hq, bs, hd = c["o"].shape
    D, I = c["w_o"].shape[0], c["w_gate"].shape[0]
    for b in range(B):
        for j in range(bs):
            r = b * bs + j
            ox = [c["o"][b, h, j, e] for h in range(Hq) for e in range(hd)]   # head-major flattening
            y1 = [c["x"][r, i] + sum(ox[t] * c["w_o"][i, t] for t in range(Hq * hd)) for i in range(D)]
            assert np.allclose(x1[r], y1, atol=1e-12)
            ms = sum(v * v for v in y1) / D
            h = [y1[i] / np.sqrt(ms + 1e-6) * c["g_post"][i] for i in range(D)]
            a = []
            for u in range(I):
                g = sum(h[i] * c["w_gate"][u, i] for i in range(D))
                up = sum(h[i] * c["w_up"][u, i] for i in range(D))
                a.append(g / (1 + np.exp(-g)) * up)
            y2 = [y1[i] + sum(a[u] * c["w_down"][i, u] for u in range(I)) for i in range(D)]
            assert np.allclose(x2[r], y2, atol=1e-10)


def test_layer_tail_special_cases():
    c = _tail_case(1)
    # a zero output projection leaves the residual stream; a zero gate zeroes the MLP (silu(0) = 0)
    z = dict(c, w_o=np.zeros_like(c["w_o"]), w_gate=np.zeros_like(c["w_gate"]))
    x1, x2 = oracle.draft_layer_tail(**z)
    np.testing.assert_array_equal(x1, c["x"])
    np.testing.assert_array_equal(x2, c["x"])
    # silu: closed values and the limit z * sigmoid(z) -> z
    np.testing.assert_allclose(oracle.silu([0.0, 1.0, -1.0, 40.0]),
                               [0.0, 1 / (1 + np.exp(-1)), -1 / (1 + np.e), 40.0], rtol=1e-12)
    # bf16 storage points
    x1b, x2b = oracle.draft_layer_tail(**c, bf16=True)
    np.testing.assert_array_equal(x2b, oracle.round_to_bf16(x2b))


def test_layer_qkv_matches_loops():
    """The input norm and the q/k/v projections, element by element: row
    b * bs + j of x, query head h at output row h * hd + e of w_qkv, key head g
    at (Hq + g) * hd + e, value head g at (Hq + Hkv + g) * hd + e."""
    rng = np.random.default_rng(21)
    B, bs, D, Hq, Hkv, hd = 2, 3, 8, 4, 2, 4
    x = rng.normal(size=(B * bs, D)) * 2.0
    g = 1 + 0.1 * rng.normal(size=D)
    w = rng.normal(size=((Hq + 2 * Hkv) * hd, D))
    q, kb, vb = oracle.draft_layer_qkv(x, g, w, B, Hq, Hkv, head_dim=hd, eps=1e-6)
    assert q.shape == (B, Hq, bs, hd) and kb.shape == (B, Hkv, bs, hd) and vb.shape == (B, Hkv, bs, hd)
    for b in range(B):
        for j in range(bs):
            row = x[b * bs + j]
            r = (sum(v * v for v in row) / D + 1e-6) ** 0.5
            h = [row[i] / r * g[i] for i in range(D)]
            dot = lambda o: sum(h[i] * w[o, i] for i in range(D))  # noqa: E731
            for e in range(hd):
                for hh in range(Hq):
                    assert abs(q[b, hh, j, e] - dot(hh * hd + e)) < 1e-10
                for gg in range(Hkv):
                    assert abs(kb[b, gg, j, e] - dot((Hq + gg) * hd + e)) < 1e-10
                    assert abs(vb[b, gg, j, e] - dot((Hq + Hkv + gg) * hd + e)) < 1e-10


def test_layer_qkv_selection_weights_place_each_head():
    """A weight whose output row o reads input column pi(o) (a selection
    matrix) puts the normalised row's column pi(o) at o's head position: this
    catches a transposed layout or a wrong head order; zero weights give zero
    heads; bf16 outputs are bfloat16 values."""
    rng = np.random.default_rng(22)
    B, bs, D, Hq, Hkv, hd = 2, 4, 16, 4, 2, 8
    N = (Hq + 2 * Hkv) * hd
    x = rng.normal(size=(B * bs, D))
    pi = rng.integers(0, D, size=N)
    w = np.zeros((N, D))
    w[np.arange(N), pi] = 1.0
    q, kb, vb = oracle.draft_layer_qkv(x, np.ones(D), w, B, Hq, Hkv, head_dim=hd, eps=0.0)
    hn = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True))
    full = np.concatenate([q, kb, vb], axis=1)        # [B, Hq + 2 Hkv, bs, hd]
    for o in range(N):
        np.testing.assert_allclose(full[:, o // hd, :, o % hd], hn[:, pi[o]].reshape(B, bs), rtol=1e-12)
    z = oracle.draft_layer_qkv(x, np.ones(D), np.zeros((N, D)), B, Hq, Hkv, head_dim=hd)
    assert all(np.all(t == 0) for t in z)
    qb, _, _ = oracle.draft_layer_qkv(x, 1 + 0.1 * rng.normal(size=D), rng.normal(size=(N, D)), B, Hq, Hkv,
                                      head_dim=hd, bf16=True)
    np.testing.assert_array_equal(qb, oracle.round_to_bf16(qb))
