"""The oracle's verification over chunks of a saved batch, for worker processes.

Test infrastructure: the sweep in test_gpu_verify_sweep.py saves a batch's
bf16 logits (as raw 16-bit words) and draft tokens to .npy files, and spawned
workers run oracle.verify on slices of it, each slice with its own sequence
indices so that the random-number counters are those of the whole batch.
Marshalling only: no method arithmetic here.
"""
import numpy as np

import oracle


def bf16_bits_to_f64(bits):
    """bf16 values stored as uint16 words -> the same values as float64."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def verify_chunk(lt_path, ld_path, x_path, lo, hi, temperature, seed, cycle):
    lt = bf16_bits_to_f64(np.load(lt_path, mmap_mode="r")[lo:hi])
    ld = None if temperature == 0 else bf16_bits_to_f64(np.load(ld_path, mmap_mode="r")[lo:hi])
    x = np.array(np.load(x_path, mmap_mode="r")[lo:hi])
    r = oracle.verify(lt, ld, x, temperature, seed, cycle, seq_ids=np.arange(lo, hi))
    return lo, r.accepted_len, r.out_tokens, r.near_tie
