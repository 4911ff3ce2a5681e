"""Pins for the oracle's context fusion, K/V injection and block attention.

Each test checks a closed form, an invariant or a constructed case whose
answer is known without running the oracle's own formula.
"""
import itertools

import numpy as np
import pytest

import oracle

J, DT, D, L, HKV, HD = 5, 16, 32, 2, 2, 8     # reduced widths for CPU pins


def _perm(n, seed):
    return np.random.default_rng(seed).permutation(n)


def test_rms_norm_closed_form():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(7, 64)) * rng.uniform(0.1, 10, size=(7, 1))
    y = oracle.rms_norm(x, 2.5, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 2.5, rtol=1e-12)
    # scale invariance and sign of the gain
    np.testing.assert_allclose(oracle.rms_norm(3.0 * x, -1.0, 0.0), -oracle.rms_norm(x, 1.0, 0.0), rtol=1e-12)
    # eps only matters for tiny inputs: zero stays zero
    assert np.all(oracle.rms_norm(np.zeros((1, 8)), 1.0, 1e-6) == 0.0)


def test_rope_is_complex_rotation_of_paired_halves():
    rng = np.random.default_rng(1)
    d, theta = 128, 1e6
    x = rng.normal(size=(5, d))
    pos = np.array([0, 1, 17, 4096, 131071])
    y = oracle.rope(x, pos, theta)
    # pair e with e + d/2 as one complex number and turn it by pos * theta^(-2e/d)
    for r in range(5):
        for e in range(d // 2):
            z = complex(x[r, e], x[r, e + d // 2]) * np.exp(1j * pos[r] * theta ** (-2.0 * e / d))
            assert abs(z.real - y[r, e]) < 1e-9 and abs(z.imag - y[r, e + d // 2]) < 1e-9
    np.testing.assert_allclose(oracle.rope(x, np.zeros(5), theta), x, rtol=0, atol=0)


def test_rope_relative_position_property():
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=(2, 128))
    dots = [oracle.rope(q, m + s, 1e6) @ oracle.rope(k, n + s, 1e6)
            for (m, n) in [(10, 3)] for s in (0, 5, 1000, 70000)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(oracle.rope(q, 12345, 1e6)), np.linalg.norm(q), rtol=1e-12)


@pytest.mark.parametrize("j", range(J))
def test_fusion_selects_tap_through_permutation(j):
    # W_c in R^{D x J*d_t}: a block permutation that reads only tap j must
    # reproduce a permutation of that tap (up to the RMSNorm scale).
    rng = np.random.default_rng(10 + j)
    M = 3
    taps = [rng.normal(size=(M, DT)) for _ in range(J)]
    pi = _perm(DT, j)
    w = np.zeros((D, J * DT))
    for n in range(DT):
        w[n, j * DT + pi[n]] = 1.0
    H, _, _ = oracle.fuse_rows(taps, w, 1.0, rng.normal(size=(L * 2 * HKV * HD, D)), np.ones((L, HD)),
                               np.zeros(M), L, HKV, HD, eps=0.0)
    expect = np.zeros((M, D))
    expect[:, :DT] = taps[j][:, pi]
    expect /= np.sqrt(np.mean(expect ** 2, axis=1, keepdims=True))
    np.testing.assert_allclose(H, expect, rtol=1e-12, atol=1e-12)


def test_fusion_brute_force_loops():
    rng = np.random.default_rng(4)
    M, j, dt, dm = 2, 2, 3, 4
    taps = [rng.normal(size=(M, dt)) for _ in range(j)]
    w = rng.normal(size=(dm, j * dt))
    g = rng.normal(size=dm)
    H, _, _ = oracle.fuse_rows(taps, w, g, rng.normal(size=(2 * 1 * 1 * dm, dm)), np.ones((1, dm)),
                               np.zeros(M), 1, 1, dm, eps=1e-6)
    for m in range(M):
        feat = [taps[t][m, i] for t in range(j) for i in range(dt)]
        y = [sum(w[n][c] * feat[c] for c in range(j * dt)) for n in range(dm)]
        ms = sum(v * v for v in y) / dm
        for n in range(dm):
            assert abs(H[m, n] - y[n] / (ms + 1e-6) ** 0.5 * g[n]) < 1e-12


def test_kv_column_layout_and_key_norm():
    # w_kv column ((l*2 + s)*Hkv + h)*d + e reads H_t component pi(column).
    rng = np.random.default_rng(5)
    M = 4
    taps = [rng.normal(size=(M, DT)) for _ in range(J)]
    w_fuse = rng.normal(size=(D, J * DT))
    N = L * 2 * HKV * HD
    pi = rng.integers(0, D, size=N)
    w_kv = np.zeros((N, D))
    w_kv[np.arange(N), pi] = 1.0
    kg = rng.normal(size=(L, HD))
    pos = np.array([0, 3, 9, 100])
    H, K, V = oracle.fuse_rows(taps, w_fuse, 1.0, w_kv, kg, pos, L, HKV, HD, eps=0.0)
    for l, s, h, e in itertools.product(range(L), range(2), range(HKV), range(HD)):
        col = ((l * 2 + s) * HKV + h) * HD + e
        if s == 1:
            np.testing.assert_allclose(V[:, l, h, e], H[:, pi[col]], rtol=1e-12)
    # keys: constant gain c => the rotated, normalised head vector has rms |c|
    _, K2, _ = oracle.fuse_rows(taps, w_fuse, 1.0, w_kv, np.full((L, HD), -3.0), pos, L, HKV, HD, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(K2 ** 2, axis=-1)), 3.0, rtol=1e-12)
    # at position 0 the key is the normalised projection itself
    raw = H[0, pi[:N]].reshape(L, 2, HKV, HD)[:, 0]
    np.testing.assert_allclose(K[0], raw / np.sqrt(np.mean(raw ** 2, -1, keepdims=True)) * kg[:, None, :], rtol=1e-12)


def test_fuse_context_scatters_to_positions():
    rng = np.random.default_rng(6)
    B, cap = 3, 12
    n_new = [2, 0, 3]
    cu = np.concatenate([[0], np.cumsum(n_new)])
    seq_len = np.array([4, 7, 9])
    taps = [rng.normal(size=(cu[-1], DT)) for _ in range(J)]
    w_fuse = rng.normal(size=(D, J * DT))
    w_kv = rng.normal(size=(L * 2 * HKV * HD, D))
    kg = np.ones((L, HD))
    ck = np.full((L, B, HKV, cap, HD), 7.0)
    cv = np.full((L, B, HKV, cap, HD), 7.0)
    oracle.fuse_context(taps, cu, seq_len, w_fuse, 1.0, w_kv, kg, ck, cv)
    written = np.zeros((B, cap), bool)
    written[0, 4:6] = True
    written[2, 9:12] = True
    for b in range(B):
        for p in range(cap):
            changed = not np.all(ck[:, b, :, p] == 7.0)
            assert changed == written[b, p], (b, p)
    with pytest.raises(ValueError):
        oracle.fuse_context(taps, cu, np.array([4, 7, 10]), w_fuse, 1.0, w_kv, kg, ck, cv)


def _attn_case(seed, B=2, Hq=8, Hkv=2, bs=4, d=16, cap=20, seq_len=(9, 0)):
    rng = np.random.default_rng(seed)
    return dict(
        q=rng.normal(size=(B, Hq, bs, d)), kb=rng.normal(size=(B, Hkv, bs, d)),
        vb=rng.normal(size=(B, Hkv, bs, d)), q_gain=1 + 0.1 * rng.normal(size=d),
        k_gain=1 + 0.1 * rng.normal(size=d), cache_k=rng.normal(size=(B, Hkv, cap, d)),
        cache_v=rng.normal(size=(B, Hkv, cap, d)), seq_len=np.array(seq_len))


def test_attention_zero_query_is_mean_of_window_values():
    c = _attn_case(0)
    c["q"][:] = 0.0                       # RMSNorm(0) = 0 => every score is 0
    for window in (0, 4):
        o = oracle.block_attn(**c, window=window)
        for b in range(2):
            n = c["seq_len"][b]
            lo = max(0, n - window) if window else 0
            for h in range(8):
                g = h // 4
                vals = np.concatenate([c["cache_v"][b, g, lo:n], c["vb"][b, g]])
                np.testing.assert_allclose(o[b, h], np.broadcast_to(vals.mean(0), o[b, h].shape), rtol=1e-12)


def test_attention_gqa_head_mapping():
    c = _attn_case(1)
    const = np.array([[1.0] * 16, [-2.0] * 16])
    c["cache_v"][:] = const[None, :, None, :]
    c["vb"][:] = const[None, :, None, :]
    o = oracle.block_attn(**c)
    for h in range(8):
        np.testing.assert_allclose(o[:, h], np.broadcast_to(const[h // 4], o[:, h].shape), rtol=1e-12)  # h // (Hq/Hkv), not h % Hkv


def test_attention_dominant_key_returns_its_value():
    c = _attn_case(2)
    b, h, j = 0, 5, 1
    g = h // 4
    n = c["seq_len"][b]
    qh = oracle.rope(oracle.rms_norm(c["q"][b, h, j], c["q_gain"], 1e-6), n + j, 1e6)
    c["cache_k"][b, g, 3] = 200.0 * qh / np.linalg.norm(qh)
    o = oracle.block_attn(**c)
    np.testing.assert_allclose(o[b, h, j], c["cache_v"][b, g, 3], rtol=1e-6, atol=1e-6)


def test_attention_is_non_causal_and_ignores_stale_cache():
    c = _attn_case(3)
    base = oracle.block_attn(**c)
    # the last block value influences the first block row (no causal mask)
    c2 = {k: v.copy() for k, v in c.items()}
    c2["vb"][0, 1, -1] += 5.0
    o2 = oracle.block_attn(**c2)
    assert np.abs(o2[0, 4:8, 0] - base[0, 4:8, 0]).max() > 1e-3
    # positions >= seq_len and positions outside the window are never read
    c3 = {k: v.copy() for k, v in c.items()}
    c3["cache_k"][0, :, 9:] = 1e3
    c3["cache_v"][0, :, 9:] = 1e3
    c3["cache_k"][1] = 1e3      # sequence 1 has an empty cached context
    np.testing.assert_array_equal(oracle.block_attn(**c3), base)
    c4 = {k: v.copy() for k, v in c.items()}
    c4["cache_v"][0, :, :5] = 1e3
    np.testing.assert_array_equal(oracle.block_attn(**c4, window=4), oracle.block_attn(**c, window=4))
    assert np.abs(oracle.block_attn(**c4, window=5) - oracle.block_attn(**c, window=5)).max() > 1.0


def test_attention_is_invariant_to_the_order_of_cached_rows():
    """Softmax attention is a sum over keys: permuting the cached (key, value)
    rows of a sequence together leaves the output unchanged; permuting the keys
    alone (values left in place) does not."""
    c = _attn_case(4)
    base = oracle.block_attn(**c)
    n = c["seq_len"][0]
    perm = _perm(n, 11)
    c2 = {k: v.copy() for k, v in c.items()}
    c2["cache_k"][0, :, :n] = c["cache_k"][0][:, perm]
    c2["cache_v"][0, :, :n] = c["cache_v"][0][:, perm]
    np.testing.assert_allclose(oracle.block_attn(**c2), base, rtol=1e-12, atol=1e-12)
    c3 = {k: v.copy() for k, v in c.items()}
    c3["cache_k"][0, :, :n] = c["cache_k"][0][:, perm]
    assert np.abs(oracle.block_attn(**c3)[0] - base[0]).max() > 1e-3


@pytest.mark.parametrize("gain0", [0.5, 1.5, 3.0])
def test_attention_closed_form_pins_scale_and_block_positions(gain0):
    """A case whose output is written out by hand, without the oracle's own
    formula.  Every query head vector is c_h * e_0, so the per-head RMSNorm
    leaves c_h / sqrt(c_h^2 / d + eps) * gain[0] in element 0 and zeros
    elsewhere; element pair (0, d/2) has inverse frequency theta^0 = 1, so RoPE
    turns it by exactly the row's position in radians.  Two cached keys (the
    cache holds keys already normalised and rotated) lie in that same pair at
    angles phi_1 = n (where block row 0 sits when rows start at seq_len = n)
    and phi_2 = 0 (where it would sit if rows started at 0), with lengths a_1,
    a_2.  The block keys are zero, so RMSNorm keeps them zero and they score 0.
    Score of key i for block row j: s_i = qn * a_i * cos(n + j - phi_i) / sqrt(d).
    Output: (sum_i e^{s_i} v_i + sum_j' vb_j') / (sum_i e^{s_i} + bs).
    An oracle without the 1/sqrt(d) scale, with 1/d, or with block row j at
    position j fails this test."""
    import math
    d, bs, n, eps, theta = 128, 3, 2, 1e-6, 1e6
    rng = np.random.default_rng(31)
    c = [1000.0, -1000.0, 250.0, 4000.0]          # one per query head (GQA 4:1 onto one KV head)
    q = np.zeros((1, 4, bs, d))
    for h in range(4):
        q[0, h, :, 0] = c[h]
    q_gain = 1.0 + 0.1 * rng.normal(size=d)
    q_gain[0] = gain0
    k_gain = 1.0 + 0.1 * rng.normal(size=d)
    a = [4.0, 3.0]
    phi = [float(n), 0.0]
    cache_k = np.zeros((1, 1, 4, d))
    cache_v = rng.normal(size=(1, 1, 4, d))
    for i in range(2):
        cache_k[0, 0, i, 0] = a[i] * math.cos(phi[i])
        cache_k[0, 0, i, d // 2] = a[i] * math.sin(phi[i])
    cache_k[0, 0, 2:] = 50.0                       # rows at and past seq_len: never read
    kb = np.zeros((1, 1, bs, d))
    vb = rng.normal(size=(1, 1, bs, d))
    o = oracle.block_attn(q, kb, vb, q_gain, k_gain, cache_k, cache_v, np.array([n]), theta=theta, eps=eps)
    for h in range(4):
        qn = c[h] / math.sqrt(c[h] ** 2 / d + eps) * gain0
        for j in range(bs):
            s = [qn * a[i] * math.cos(n + j - phi[i]) / math.sqrt(d) for i in range(2)]
            w = [math.exp(x) for x in s]
            num = w[0] * cache_v[0, 0, 0] + w[1] * cache_v[0, 0, 1] + vb[0, 0].sum(axis=0)
            np.testing.assert_allclose(o[0, h, j], num / (w[0] + w[1] + bs), rtol=1e-12, atol=1e-14)


def test_attention_brute_force_loops():
    """Scalar loops over the definition for a few (sequence, head, row)
    outputs: per-head RMSNorm with the gain, RoPE as a complex rotation of the
    pair (e, e + d/2) by pos * theta^(-2e/d), scores q.k / sqrt(d) over the
    window's cached keys followed by the block's keys, an explicit exp / sum
    softmax, and the weighted sum of the values."""
    import cmath
    import math
    d, theta, eps = 16, 1e4, 1e-6
    c = _attn_case(7, d=d, cap=20, seq_len=(9, 3))

    def norm_rot(x, gain, pos):
        r = math.sqrt(sum(t * t for t in x) / d + eps)
        y = [x[e] / r * gain[e] for e in range(d)]
        out = [0.0] * d
        for e in range(d // 2):
            z = complex(y[e], y[e + d // 2]) * cmath.exp(1j * pos * theta ** (-2.0 * e / d))
            out[e], out[e + d // 2] = z.real, z.imag
        return out

    for window in (0, 4):
        o = oracle.block_attn(**c, theta=theta, eps=eps, window=window)
        for b, h, j in [(0, 0, 0), (0, 5, 3), (1, 7, 2), (1, 2, 1)]:
            n = int(c["seq_len"][b])
            g = h // 4
            qv = norm_rot(list(c["q"][b, h, j]), c["q_gain"], n + j)
            keys, vals = [], []
            for t in range(max(0, n - window) if window else 0, n):
                keys.append(list(c["cache_k"][b, g, t]))
                vals.append(list(c["cache_v"][b, g, t]))
            for jj in range(4):
                keys.append(norm_rot(list(c["kb"][b, g, jj]), c["k_gain"], n + jj))
                vals.append(list(c["vb"][b, g, jj]))
            s = [sum(qv[e] * k[e] for e in range(d)) / math.sqrt(d) for k in keys]
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            tot = sum(w)
            ref = [sum(w[i] * vals[i][e] for i in range(len(w))) / tot for e in range(d)]
            np.testing.assert_allclose(o[b, h, j], ref, rtol=1e-12, atol=1e-13)
