"""Boundary cases of dflash_verify, counted over a sweep of full-vocabulary cycles.

Every case is a workload's logits at V = 262144, verified by the GPU in the
launch configuration of its own batch size (B = 1, 4, 32, 128) and by the
oracle, for several cycles, each with fresh logits, draft tokens, seed and
cycle counter.

T = 1 (2400 sequence-cycles): the accepted lengths and tokens equal the
oracle's in every sequence the oracle does not flag as a boundary case (a
Philox uniform within 1e-6 of a value at which the decision would change:
alpha for an acceptance, a normalised cumulative-mass edge for a draw).
Flagged sequences that differ are counted, and must stay within 1 % of the
sweep.  T = 0: every sequence equals the oracle's, with no flag.  The
per-case counts are printed (run with -s to see them).
"""
import multiprocessing
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import block_speculative_decoding_gb300 as dfl
import oracle_pool
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [   # (workload, cycles)
    (workloads.SINGLE_STREAM, 32),
    (workloads.LONG_CONTEXT, 16),
    (workloads.BATCHED, 16),
    (workloads.high_batch(8, 0.25), 4),
    (workloads.high_batch(8, 1.0), 4),
    (workloads.high_batch(8, 4.0), 4),
    (workloads.high_batch(16, 1.0), 1),
    (workloads.high_batch(4, 1.0), 1),
]
CHUNK = 8          # sequences per oracle task


@pytest.fixture(scope="module")
def pool():
    # spawned (not forked) workers: this process already holds a CUDA context
    ctx = multiprocessing.get_context("spawn")
    with ctx.Pool(max(1, min(16, os.cpu_count() or 1))) as p:
        yield p


def _sweep(pool, tmp_path, temperature):
    rows, totals = [], dict(seqs=0, flagged=0, mismatched=0, unflagged=0)
    for cfg0, cycles in CASES:
        n_seq = n_flag = n_mis = n_bad = 0
        for c in range(cycles):
            cfg = replace(cfg0, seed=cfg0.seed * 100 + c)
            lt, ld = workloads.logits(cfg, DEV)
            x = workloads.draft_tokens(ld, temperature, seed=500 + c)
            seed, cycle = 7000 + 13 * c, 3 * c + 1
            acc, out = dfl.verify(lt, ld, x, temperature, seed, cycle)
            acc, out = acc.cpu().numpy(), out.cpu().numpy()
            paths = [str(tmp_path / n) for n in ("lt.npy", "ld.npy", "x.npy")]
            np.save(paths[0], lt.view(torch.int16).cpu().numpy())
            if temperature > 0:
                np.save(paths[1], ld.view(torch.int16).cpu().numpy())
            np.save(paths[2], x.cpu().numpy())
            del lt, ld
            B = cfg.B
            tasks = [(*paths, lo, min(B, lo + CHUNK), temperature, seed, cycle) for lo in range(0, B, CHUNK)]
            for lo, r_acc, r_out, r_near in pool.starmap(oracle_pool.verify_chunk, tasks):
                hi = lo + len(r_acc)
                mism = (acc[lo:hi] != r_acc) | np.any(out[lo:hi] != r_out, axis=1)
                n_seq += hi - lo
                n_flag += int(r_near.sum())
                n_mis += int(mism.sum())
                n_bad += int((mism & ~r_near).sum())
        rows.append((cfg0.name, cfg0.B, cfg0.bs, cycles, n_seq, n_flag, n_mis, n_bad))
        for k, v in zip(("seqs", "flagged", "mismatched", "unflagged"), (n_seq, n_flag, n_mis, n_bad)):
            totals[k] += v
    print("\nverification sweep at T = %g (V = 262144)" % temperature)
    print("%-26s %4s %3s %6s %6s %8s %10s %9s" % ("case", "B", "bs", "cycles", "seqs", "flagged", "mismatched",
                                                 "unflagged"))
    for r in rows:
        print("%-26s %4d %3d %6d %6d %8d %10d %9d" % r)
    print("%-26s %4s %3s %6s %6d %8d %10d %9d" % ("total", "", "", "", totals["seqs"], totals["flagged"],
                                                  totals["mismatched"], totals["unflagged"]))
    return rows, totals


def test_verify_sweep_sampled_boundary_cases(pool, tmp_path):
    rows, tot = _sweep(pool, tmp_path, 1.0)
    assert tot["seqs"] >= 2000
    assert tot["unflagged"] == 0, rows
    assert tot["mismatched"] <= 0.01 * tot["seqs"], rows


def test_verify_sweep_greedy_is_exact(pool, tmp_path):
    rows, tot = _sweep(pool, tmp_path, 0.0)
    assert tot["mismatched"] == 0 and tot["flagged"] == 0, rows
