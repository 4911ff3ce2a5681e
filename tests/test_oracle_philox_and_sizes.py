"""Pins for the oracle's random numbers, bf16 rounding and size arithmetic.

Every check compares the oracle with something other than itself: published
known-answer vectors, numpy's own Philox implementation, torch's bfloat16
conversion, and numbers printed on the DFlash pages.
"""
import os

import numpy as np
import pytest
import torch

import oracle


def _read_kat(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox_kat.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            name, rounds, *words = lhs.split()
            rows.append((name, int(rounds), [int(w, 16) for w in words], [int(w, 16) for w in rhs.split()]))
    return rows


def test_philox_known_answer_vectors(golden_dir):
    rows = _read_kat(golden_dir)
    assert len(rows) == 6
    for name, rounds, inp, expect in rows:
        width = 32 if name == "philox4x32" else 64
        out = oracle.philox4(inp[:4], inp[4:], width=width, rounds=rounds)
        assert [int(w[0]) for w in out] == expect, name


@pytest.mark.parametrize("key", [0, 1, 0xDEADBEEF12345678, (1 << 64) - 1])
def test_philox4x64_matches_numpy_stream(key):
    # numpy.random.Philox is Philox-4x64-10; it advances the 256-bit counter
    # before producing each block of four words.
    g = np.random.Philox(counter=0, key=key)
    raw = g.random_raw(4 * 6)
    for blk in range(6):
        c = blk + 1
        out = oracle.philox4((c, 0, 0, 0), (key & ((1 << 64) - 1), 0), width=64)
        assert [int(w[0]) for w in out] == [int(v) for v in raw[4 * blk:4 * blk + 4]]


def test_philox4x32_vectorised_equals_scalar():
    rng = np.random.default_rng(3)
    ctr = rng.integers(0, 2**32, size=(4, 64), dtype=np.uint64)
    key = (0x12345678, 0x9ABCDEF0)
    vec = oracle.philox4x32_10(tuple(ctr), key)
    for i in range(64):
        one = oracle.philox4x32_10(tuple(int(c[i]) for c in ctr), key)
        assert [int(w[0]) for w in one] == [int(w[i]) for w in vec]


def test_verify_uniforms_range_and_float32_exact():
    b = np.arange(4096)
    u, v = oracle.verify_uniforms(7, 3, 2, b)
    for x in (u, v):
        assert np.all(x >= 0.0) and np.all(x < 1.0)
        assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    # roughly uniform: mean 1/2 within 5 sigma
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / b.size)
    # different words, different cycles, different seeds give different streams
    u2, _ = oracle.verify_uniforms(7, 4, 2, b)
    u3, _ = oracle.verify_uniforms(8, 3, 2, b)
    assert not np.array_equal(u, v) and not np.array_equal(u, u2) and not np.array_equal(u, u3)


def test_round_to_bf16_matches_torch():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(100000, generator=g, dtype=torch.float64) * torch.exp(torch.randn(100000, generator=g) * 4)
    ours = oracle.round_to_bf16(x.numpy())
    ref = x.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def _page_numbers(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "page_numbers.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_size_arithmetic_reproduces_page_numbers(golden_dir):
    pg = _page_numbers(golden_dir)
    # E4B drafter: vocab 262144, width 2560, 5 taps of width 2560, 5 layers,
    # GQA 32/8, head 128; MLP width 5120 is the only one that closes the count.
    n = oracle.draft_param_count(262144, 2560, 5, 2560, 5, 32, 8, 128, 5120)
    assert n == int(pg["draft_params"])
    head = 262144 * 2560
    assert round(100 * head / n, 1) == pg["head_share_pct"]
    assert round(n * 0.5 / 2**20, 1) == pg["codes_4bit_mib"]
    assert head * 0.5 / 2**20 == pg["head_codes_4bit_mib"]
    assert head * 2 / 2**30 == pg["embedding_bf16_gib"]
    per_seq = oracle.kv_cache_payload_bytes(5, 8, 1024, 128, 2)
    assert per_seq / 2**20 == pg["cache_payload_mib_per_seq"]
    assert 64 * per_seq / 2**30 == pg["cache_payload_gib_64_seqs"]
    assert round(oracle.fusion_weight_bytes(2048, 5, 2) / 1e6, 2) == pg["wc_mb_d2048"]
