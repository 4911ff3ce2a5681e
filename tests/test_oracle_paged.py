"""Pins of oracle.gather_pages (the paged cache layout's linear view).

Tied to the layout's definition element by element (brute force), to the
linear layout it generalises (one page per sequence, identity table), and to
the rule that out-of-pool entries read as zero rows.
"""
import numpy as np

import oracle


def test_identity_table_of_whole_sequence_pages_is_the_linear_layout():
    rng = np.random.default_rng(0)
    L, B, H, cap, d = 2, 3, 2, 8, 4
    lin = rng.standard_normal((L, B, H, cap, d))
    # one page per sequence holding all of its rows: page b = sequence b
    pool = np.empty((L, B, H, cap, d))
    for l in range(L):
        for b in range(B):
            for h in range(H):
                for p in range(cap):
                    pool[l, b, h, p] = lin[l, b, h, p]
    table = np.arange(B).reshape(B, 1)
    np.testing.assert_array_equal(oracle.gather_pages(pool, table, cap), lin)


def test_every_element_follows_the_block_table():
    rng = np.random.default_rng(1)
    L, NP, H, P, d = 2, 11, 3, 4, 5
    B, MP = 3, 3
    pool = rng.standard_normal((L, NP, H, P, d))
    table = rng.permutation(NP)[: B * MP].reshape(B, MP)
    out = oracle.gather_pages(pool, table, P)
    assert out.shape == (L, B, H, MP * P, d)
    for l in range(L):
        for b in range(B):
            for h in range(H):
                for p in range(MP * P):
                    for e in range(d):
                        assert out[l, b, h, p, e] == pool[l, table[b, p // P], h, p % P, e]


def test_out_of_pool_entries_read_zero_rows():
    rng = np.random.default_rng(2)
    pool = rng.standard_normal((1, 4, 1, 2, 3))
    table = np.array([[3, -1], [4, 0]])
    out = oracle.gather_pages(pool, table, 2)
    np.testing.assert_array_equal(out[0, 0, 0, 0:2], pool[0, 3, 0])
    np.testing.assert_array_equal(out[0, 0, 0, 2:4], 0.0)
    np.testing.assert_array_equal(out[0, 1, 0, 0:2], 0.0)
    np.testing.assert_array_equal(out[0, 1, 0, 2:4], pool[0, 0, 0])
