"""The C ABI library loads, exports every declared symbol, and validates
arguments on the host -- all without a GPU (no compute call is made)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def L():
    from block_speculative_decoding_gb300 import _build
    path = _build.build()
    import block_speculative_decoding_gb300 as dfl
    return dfl.lib(), path


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    syms = declared_symbols()
    for s in ("dflash_fuse_context", "dflash_block_attn", "dflash_verify"):
        assert s in syms
    assert len(syms) == 22


def test_library_exports_every_declared_symbol(L):
    lib, path = L
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(dflash_\w+)", out))
    for s in declared_symbols():
        assert s in exported, s
        assert hasattr(lib, s)
    # nothing else leaks out of the library under the dflash_ prefix
    assert exported == set(declared_symbols())


def test_workspace_queries(L):
    import block_speculative_decoding_gb300 as dfl
    assert dfl.verify_workspace_size(32, 8, 262144, dfl.BF16) > 32 * 15 * 16 * 8
    assert dfl.verify_workspace_size(0, 8, 262144, dfl.BF16) == 0
    assert dfl.block_attn_workspace_size(32, 8, 32, 8, 8256, 0, dfl.BF16) > 0
    assert dfl.block_attn_workspace_size(0, 8, 32, 8, 8256, 0, dfl.BF16) == 0
    assert dfl.fuse_context_workspace_size(256, 5, 2560, 2560, 5, 8, dfl.BF16) >= 256 * 2560 * 2
    assert dfl.version() == (1 << 16) | 3


def _cache(**kw):
    import block_speculative_decoding_gb300 as dfl
    d = dict(num_layers=5, batch=2, num_kv_heads=8, head_dim=128, capacity=64, dtype=dfl.BF16,
             k=16, v=16, seq_len=16, ring=0, block_table=None, page_size=0, num_pages=0, max_pages=0)
    d.update(kw)
    return dfl._KVCacheDesc(d["num_layers"], d["batch"], d["num_kv_heads"], d["head_dim"], d["capacity"],
                            d["dtype"], d["k"], d["v"], d["seq_len"], d["ring"], d["block_table"], d["page_size"],
                            d["num_pages"], d["max_pages"])


def test_host_validation_rejects_bad_arguments_before_any_launch(L):
    lib, _ = L
    import block_speculative_decoding_gb300 as dfl
    P = ctypes.c_void_p
    # verify: block size out of range, negative temperature, NULL outputs
    assert lib.dflash_verify(P(16), P(16), 1, P(16), 2, 0, 100, 1.0, 0, 0, P(16), P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_verify(P(16), P(16), 1, P(16), 2, 8, 100, -1.0, 0, 0, P(16), P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_verify(P(16), P(16), 1, P(16), 2, 8, 100, 1.0, 0, 0, None, P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_verify(P(16), P(16), 7, P(16), 2, 8, 100, 1.0, 0, 0, P(16), P(16), P(256), 1 << 20, None) == 2
    # verify: workspace too small / misaligned
    assert lib.dflash_verify(P(16), P(16), 1, P(16), 2, 8, 100, 1.0, 0, 0, P(16), P(16), P(256), 8, None) == 5
    assert lib.dflash_verify(P(16), P(16), 1, P(16), 2, 8, 100, 1.0, 0, 0, P(16), P(16), P(16), 1 << 20, None) == 5
    assert b"workspace" in lib.dflash_last_error_string()
    # an empty batch is a no-op
    assert lib.dflash_verify(None, None, 1, None, 0, 8, 100, 1.0, 0, 0, None, None, None, 0, None) == 0
    # block attention: head_dim, GQA divisibility, block size, cache NULL, layer range
    c = _cache(head_dim=64)
    assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(c), 0, P(16), P(256), 1 << 30, None) == 2
    c = _cache()
    assert lib.dflash_block_attn(0, 2, 8, 30, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(c), 0, P(16), P(256), 1 << 30, None) == 1
    assert lib.dflash_block_attn(0, 2, 17, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(c), 0, P(16), P(256), 1 << 30, None) == 2
    assert lib.dflash_block_attn(5, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(c), 0, P(16), P(256), 1 << 30, None) == 1
    assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, None, 0, P(16), P(256), 1 << 30, None) == 1
    assert lib.dflash_block_attn(0, 2, 8, 32, P(17), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(c), 0, P(16), P(256), 1 << 30, None) == 1
    # a ring cache is its own window; the ring flag is 0 or 1
    r = _cache(ring=1)
    assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(r), 5, P(16), P(256), 1 << 30, None) == 2
    r = _cache(ring=2)
    assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(r), 0, P(16), P(256), 1 << 30, None) == 1
    # paged layout: page size a multiple of 128, capacity = max_pages * page_size, bf16 only, no ring,
    # window 0
    pg = dict(block_table=16, page_size=128, num_pages=4, max_pages=2, capacity=256)
    ok = _cache(**pg)
    for bad, code in ((dict(pg, page_size=64, capacity=128), 2), (dict(pg, capacity=255), 1),
                      (dict(pg, num_pages=0), 1), (dict(pg, ring=1), 2), (dict(pg, dtype=dfl.F32), 2)):
        b = _cache(**bad)
        assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(b), 0, P(16), P(256), 1 << 30, None) == code, bad
    assert lib.dflash_block_attn(0, 2, 8, 32, P(16), P(16), P(16), None, None, 1e6, 1e-6, ctypes.byref(ok), 64, P(16), P(256), 1 << 30, None) == 2
    # layer q/k/v: d_model multiple of 128 and <= 4096, alignment, workspace; empty batch is a no-op
    assert lib.dflash_draft_layer_qkv(P(16), 2, 8, 32, 8, 2500, None, 1e-6, P(16), P(16), P(16), P(16), P(256), 1 << 30, None) == 2
    assert lib.dflash_draft_layer_qkv(P(16), 2, 8, 32, 8, 8192, None, 1e-6, P(16), P(16), P(16), P(16), P(256), 1 << 30, None) == 2
    assert lib.dflash_draft_layer_qkv(P(16), 2, 8, 32, 8, 2560, None, 1e-6, P(16), P(8), P(16), P(16), P(256), 1 << 30, None) == 1
    assert lib.dflash_draft_layer_qkv(P(16), 2, 8, 32, 8, 2560, None, 1e-6, P(16), P(16), P(16), P(16), P(256), 8, None) == 5
    assert lib.dflash_draft_layer_qkv(P(16), 2, 8, 32, 8, 2560, None, -1.0, P(16), P(16), P(16), P(16), P(256), 1 << 30, None) == 1
    assert lib.dflash_draft_layer_qkv(None, 0, 8, 32, 8, 2560, None, 1e-6, None, None, None, None, None, 0, None) == 0
    assert lib.dflash_draft_layer_qkv_workspace_size(32, 8, 32, 8, 2560) > 256 * 2560 * 2
    # the bounded-wait probe: bf16 only, a limit of 1 .. 100000 us
    assert lib.dflash_debug_block_attn_wait_timeout(2, 8, 32, ctypes.byref(c), P(16), P(256), 1 << 30, 0, None) == 1
    assert lib.dflash_debug_block_attn_wait_timeout(2, 8, 32, ctypes.byref(c), P(16), P(256), 1 << 30, 200000, None) == 1
    f = _cache(dtype=dfl.F32)
    assert lib.dflash_debug_block_attn_wait_timeout(2, 8, 32, ctypes.byref(f), P(16), P(256), 1 << 30, 100, None) == 2
    assert lib.dflash_debug_block_attn_wait_timeout(2, 8, 32, ctypes.byref(c), P(16), P(256), 8, 100, None) == 5
    # DFlash2: block convolution sizes and flags; top-m m, temperature, vocabulary and workspace
    assert lib.dflash_block_conv(P(16), 2, 17, 256, 3, P(16), None, 0, P(16), None) == 1
    assert lib.dflash_block_conv(P(16), 2, 8, 256, 9, P(16), None, 0, P(16), None) == 1
    assert lib.dflash_block_conv(P(16), 2, 8, 256, 3, P(16), None, 2, P(16), None) == 1
    assert lib.dflash_block_conv(P(16), 2, 8, 258, 3, P(16), None, 0, P(16), None) == 2
    assert lib.dflash_block_conv(P(16), 2, 8, 256, 3, P(12), None, 0, P(16), None) == 1
    assert lib.dflash_block_conv(None, 0, 8, 256, 3, None, None, 0, None, None) == 0
    assert lib.dflash_draft_topm(P(16), 2, 7, 4096, 9, 1.0, 0.1, P(16), P(16), P(16), P(16), P(256), 1 << 20, None) == 2
    assert lib.dflash_draft_topm(P(16), 2, 7, 4096, 8, 0.0, 0.1, P(16), P(16), P(16), P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_draft_topm(P(16), 2, 7, 4100, 8, 1.0, 0.1, P(16), P(16), P(16), P(16), P(256), 1 << 20, None) == 2
    assert lib.dflash_draft_topm(P(16), 2, 17, 4096, 8, 1.0, 0.1, P(16), P(16), P(16), P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_draft_topm(P(16), 2, 7, 4096, 8, 1.0, 0.1, P(16), P(16), P(16), P(16), P(256), 8, None) == 5
    assert lib.dflash_draft_topm(P(8), 2, 7, 4096, 8, 1.0, 0.1, P(16), P(16), P(16), P(16), P(256), 1 << 20, None) == 1
    assert lib.dflash_draft_topm_workspace_size(2, 7, 4096, 8) > 0
    # fusion: tap count, widths, capacity visible on the host
    taps = (ctypes.c_void_p * 5)(16, 16, 16, 16, 16)
    assert lib.dflash_fuse_context(0, taps, 2560, P(16), 2, 8, P(16), None, 2560, P(16), None, 1e6, 1e-6, ctypes.byref(c), None, P(256), 1 << 30, None) == 2
    assert lib.dflash_fuse_context(5, taps, 2500, P(16), 2, 8, P(16), None, 2560, P(16), None, 1e6, 1e-6, ctypes.byref(c), None, P(256), 1 << 30, None) == 2
    assert lib.dflash_fuse_context(5, taps, 2560, P(16), 2, 1000, P(16), None, 2560, P(16), None, 1e6, 1e-6, ctypes.byref(c), None, P(256), 1 << 30, None) == 3
    assert lib.dflash_fuse_context(5, taps, 2560, P(16), 2, 0, P(16), None, 2560, P(16), None, 1e6, 1e-6, ctypes.byref(c), None, P(256), 1 << 30, None) == 0
