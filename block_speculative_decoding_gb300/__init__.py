"""DFlash draft-and-verify hot path on GB300: Python binding of libdflash.so.

Argument marshalling only.  Every step of the path runs in the CUDA kernels of
libdflash.so (sm_103a); torch supplies device memory and streams.  If the
library is missing this module raises on first use: there is no CPU fallback.

Functions (same names as the C ABI in include/dflash.h, without the prefix):
    fuse_context(taps, cu_new, w_fuse, g_fuse, w_kv, k_gain, cache, ...)
    block_attn(layer, q, kb, vb, q_gain, k_gain, cache, ...)
    verify(target_logits, draft_logits, draft_tokens, temperature, seed, cycle, ...)
plus the *_workspace_size queries, philox4x32_10 and read_device_status.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "KVCache", "DFlashError", "lib", "fuse_context", "block_attn", "verify", "draft_head", "draft_layer_tail",
    "interleave_gate_up", "draft_layer_tail_workspace_size", "draft_layer_qkv", "draft_layer_qkv_workspace_size",
    "fuse_context_workspace_size", "block_attn_workspace_size", "verify_workspace_size", "draft_head_workspace_size",
    "philox4x32_10", "read_device_status", "debug_block_attn_wait_timeout", "version", "LIB_PATH",
    "DEV_CAPACITY", "DEV_BAD_TOKEN", "DEV_BAD_SEQLEN", "DEV_TIMEOUT",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdflash.so")

F32, BF16 = 0, 1
DEV_CAPACITY, DEV_BAD_TOKEN, DEV_BAD_SEQLEN, DEV_TIMEOUT = 1, 2, 4, 8
_STATUS = {0: "OK", 1: "INVALID_ARGUMENT", 2: "UNSUPPORTED", 3: "CAPACITY", 4: "CUDA", 5: "WORKSPACE"}


class DFlashError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("dflash status %d (%s): %s" % (code, _STATUS.get(code, "?"), msg))
        self.code = code


class _KVCacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int), ("batch", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("capacity", ctypes.c_int), ("dtype", ctypes.c_int),
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
        ("ring", ctypes.c_int), ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int), ("max_pages", ctypes.c_int),
    ]


_lib = None


def lib():
    """Load libdflash.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdflash.so is not built (%s); run __graft_entry__.build() or "
                           "python -m block_speculative_decoding_gb300._build" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32, u32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float,
                                  ctypes.c_uint32, ctypes.c_uint64)
    P = ctypes.POINTER
    L.dflash_fuse_context_workspace_size.argtypes = [i32] * 6 + [i32]
    L.dflash_fuse_context_workspace_size.restype = sz
    L.dflash_fuse_context.argtypes = [i32, P(vp), i32, vp, i32, i32, vp, vp, i32, vp, vp, f32, f32,
                                      P(_KVCacheDesc), vp, vp, sz, vp]
    L.dflash_fuse_context.restype = i32
    L.dflash_block_attn_workspace_size.argtypes = [i32] * 7
    L.dflash_block_attn_workspace_size.restype = sz
    L.dflash_block_attn.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, f32, f32,
                                    P(_KVCacheDesc), i32, vp, vp, sz, vp]
    L.dflash_block_attn.restype = i32
    L.dflash_verify_workspace_size.argtypes = [i32] * 4
    L.dflash_verify_workspace_size.restype = sz
    L.dflash_verify.argtypes = [vp, vp, i32, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp, sz, vp]
    L.dflash_verify.restype = i32
    L.dflash_draft_head_workspace_size.argtypes = [i32] * 4
    L.dflash_draft_head_workspace_size.restype = sz
    L.dflash_draft_head.argtypes = [vp, i32, i32, i32, vp, f32, vp, i32, f32, u64, u64, vp, vp, vp, sz, vp]
    L.dflash_draft_head.restype = i32
    L.dflash_draft_layer_qkv_workspace_size.argtypes = [i32] * 5
    L.dflash_draft_layer_qkv_workspace_size.restype = sz
    L.dflash_draft_layer_qkv.argtypes = [vp, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp, vp, vp, sz, vp]
    L.dflash_draft_layer_qkv.restype = i32
    L.dflash_draft_layer_tail_workspace_size.argtypes = [i32] * 5
    L.dflash_draft_layer_tail_workspace_size.restype = sz
    L.dflash_draft_layer_tail.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, f32, vp, sz, vp]
    L.dflash_draft_layer_tail.restype = i32
    L.dflash_block_conv.argtypes = [vp, i32, i32, i32, i32, vp, vp, i32, vp, vp]
    L.dflash_block_conv.restype = i32
    L.dflash_draft_topm_workspace_size.argtypes = [i32] * 4
    L.dflash_draft_topm_workspace_size.restype = sz
    L.dflash_draft_topm.argtypes = [vp, i32, i32, i32, i32, f32, f32, vp, vp, vp, vp, vp, sz, vp]
    L.dflash_draft_topm.restype = i32
    L.dflash_verify_noalloc_max_scratch.argtypes = []
    L.dflash_verify_noalloc_max_scratch.restype = sz
    L.dflash_verify_noalloc.argtypes = [vp, vp, i32, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp]
    L.dflash_verify_noalloc.restype = i32
    L.dflash_debug_block_attn_wait_timeout.argtypes = [i32, i32, i32, P(_KVCacheDesc), vp, vp, sz, u32, vp]
    L.dflash_debug_block_attn_wait_timeout.restype = i32
    L.dflash_philox4x32_10.argtypes = [vp, u32, u32, vp, i32, vp]
    L.dflash_philox4x32_10.restype = i32
    L.dflash_read_device_status.argtypes = [P(u32), vp]
    L.dflash_read_device_status.restype = i32
    L.dflash_last_error_string.argtypes = []
    L.dflash_last_error_string.restype = ctypes.c_char_p
    L.dflash_version.argtypes = []
    L.dflash_version.restype = i32
    _lib = L
    return L


def _check(code):
    if code != 0:
        raise DFlashError(code, lib().dflash_last_error_string().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("dflash tensors must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("dflash tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, device, ws):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small: need %d bytes" % nbytes)
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


@dataclass
class KVCache:
    """Caller-owned draft cache: k, v [L, B, Hkv, cap, 128], seq_len int32 [B].

    ring=True makes it the drafter's sliding window: position p lives in row
    p % cap, seq_len may exceed cap, attention sees the latest min(seq_len,
    cap) positions (block_attn's window must then be 0).

    block_table (int32 [B, max_pages]) makes it paged: k, v are then
    [L, num_pages, Hkv, page_size, 128] and position p of sequence b lives in
    page block_table[b, p // page_size], row p % page_size (page_size a
    multiple of 128, bf16, window 0)."""
    k: torch.Tensor
    v: torch.Tensor
    seq_len: torch.Tensor
    ring: bool = False
    block_table: torch.Tensor | None = None

    def desc(self) -> _KVCacheDesc:
        if self.seq_len.dtype != torch.int32:
            raise TypeError("seq_len must be int32")
        if self.block_table is None:
            L, B, H, cap, d = self.k.shape
            return _KVCacheDesc(L, B, H, d, cap, _dt(self.k), self.k.data_ptr(), self.v.data_ptr(),
                                self.seq_len.data_ptr(), int(bool(self.ring)), None, 0, 0, 0)
        if self.block_table.dtype != torch.int32 or self.block_table.dim() != 2:
            raise TypeError("block_table must be int32 [batch, max_pages]")
        L, NP, H, P, d = self.k.shape
        B, MP = self.block_table.shape
        return _KVCacheDesc(L, B, H, d, MP * P, _dt(self.k), self.k.data_ptr(), self.v.data_ptr(),
                            self.seq_len.data_ptr(), int(bool(self.ring)), self.block_table.data_ptr(), P, NP, MP)


def version() -> int:
    return lib().dflash_version()


def fuse_context_workspace_size(total_new, num_taps, d_target, d_model, num_layers, num_kv_heads, dtype):
    return lib().dflash_fuse_context_workspace_size(total_new, num_taps, d_target, d_model, num_layers,
                                                    num_kv_heads, dtype)


def block_attn_workspace_size(batch, block_size, num_q_heads, num_kv_heads, capacity, window, dtype):
    return lib().dflash_block_attn_workspace_size(batch, block_size, num_q_heads, num_kv_heads, capacity,
                                                  window, dtype)


def verify_workspace_size(batch, block_size, vocab, dtype):
    return lib().dflash_verify_workspace_size(batch, block_size, vocab, dtype)


def fuse_context(taps, cu_new, w_fuse, g_fuse, w_kv, k_gain, cache: KVCache, rope_theta=1e6, eps=1e-6,
                 h_t_out=None, workspace=None, stream=None):
    """Fuse J tap tensors [M, d_t] and append K/V rows to every layer of `cache`."""
    J = len(taps)
    M, d_t = taps[0].shape
    D = w_fuse.shape[0]
    desc = cache.desc()
    L, B, Hkv = desc.num_layers, desc.batch, desc.num_kv_heads
    dt = _dt(taps[0])
    nbytes = fuse_context_workspace_size(M, J, d_t, D, L, Hkv, dt)
    ws = _workspace(nbytes, taps[0].device, workspace)
    arr = (ctypes.c_void_p * J)(*[t.data_ptr() for t in taps])
    for t in taps:
        _ptr(t)
    _check(lib().dflash_fuse_context(J, arr, d_t, _ptr(cu_new), B, M, _ptr(w_fuse), _ptr(g_fuse), D,
                                     _ptr(w_kv), _ptr(k_gain), rope_theta, eps, ctypes.byref(desc),
                                     _ptr(h_t_out), _ptr(ws), nbytes, _stream(stream)))
    return h_t_out


def block_attn(layer, q, kb, vb, q_gain, k_gain, cache: KVCache, window=0, rope_theta=1e6, eps=1e-6,
               out=None, workspace=None, stream=None):
    """One layer's non-causal block attention; returns out [B, Hq, bs, 128]."""
    B, Hq, bs, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    desc = cache.desc()
    nbytes = block_attn_workspace_size(B, bs, Hq, desc.num_kv_heads, desc.capacity, window, desc.dtype)
    ws = _workspace(nbytes, q.device, workspace)
    _check(lib().dflash_block_attn(layer, B, bs, Hq, _ptr(q), _ptr(kb), _ptr(vb), _ptr(q_gain),
                                   _ptr(k_gain), rope_theta, eps, ctypes.byref(desc), window, _ptr(out),
                                   _ptr(ws), nbytes, _stream(stream)))
    return out


def debug_block_attn_wait_timeout(cache: KVCache, block_size, num_q_heads, limit_us, out, workspace=None,
                                  stream=None):
    """Test hook: the block attention's split-merge kernel alone, over counters
    nothing increments, with its bounded wait cut to limit_us; every wait runs
    out and raises DEV_TIMEOUT (see include/dflash.h)."""
    desc = cache.desc()
    nbytes = block_attn_workspace_size(desc.batch, block_size, num_q_heads, desc.num_kv_heads, desc.capacity, 0,
                                       desc.dtype)
    ws = _workspace(nbytes, out.device, workspace)
    _check(lib().dflash_debug_block_attn_wait_timeout(desc.batch, block_size, num_q_heads, ctypes.byref(desc),
                                                      _ptr(out), _ptr(ws), nbytes, int(limit_us), _stream(stream)))


def verify(target_logits, draft_logits, draft_tokens, temperature, seed, cycle, accepted_len=None,
           out_tokens=None, workspace=None, stream=None):
    """Exact speculative verification; returns (accepted_len [B], out_tokens [B, bs])."""
    B, bs, V = target_logits.shape
    dev = target_logits.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, bs, dtype=torch.int32, device=dev)
    dt = _dt(target_logits)
    nbytes = verify_workspace_size(B, bs, V, dt)
    ws = _workspace(nbytes, dev, workspace)
    _check(lib().dflash_verify(_ptr(target_logits), _ptr(draft_logits), dt, _ptr(draft_tokens), B, bs, V,
                               float(temperature), int(seed), int(cycle), _ptr(accepted_len),
                               _ptr(out_tokens), _ptr(ws), nbytes, _stream(stream)))
    return accepted_len, out_tokens


def draft_layer_qkv_workspace_size(B, bs, Hq, Hkv, D):
    return lib().dflash_draft_layer_qkv_workspace_size(B, bs, Hq, Hkv, D)


def draft_layer_qkv(x, g_in, w_qkv, batch, num_q_heads, num_kv_heads, eps=1e-6, q=None, kb=None, vb=None,
                    workspace=None, stream=None):
    """Input RMSNorm and q/k/v projections of the block rows x [B*bs, D];
    returns (q [B, Hq, bs, 128], kb [B, Hkv, bs, 128], vb [B, Hkv, bs, 128])."""
    M, D = x.shape
    bs = M // batch
    dev = x.device
    if q is None:
        q = torch.empty(batch, num_q_heads, bs, 128, dtype=x.dtype, device=dev)
    if kb is None:
        kb = torch.empty(batch, num_kv_heads, bs, 128, dtype=x.dtype, device=dev)
    if vb is None:
        vb = torch.empty(batch, num_kv_heads, bs, 128, dtype=x.dtype, device=dev)
    nbytes = draft_layer_qkv_workspace_size(batch, bs, num_q_heads, num_kv_heads, D)
    ws = _workspace(nbytes, dev, workspace)
    _check(lib().dflash_draft_layer_qkv(_ptr(x), batch, bs, num_q_heads, num_kv_heads, D, _ptr(g_in), eps,
                                        _ptr(w_qkv), _ptr(q), _ptr(kb), _ptr(vb), _ptr(ws), nbytes, _stream(stream)))
    return q, kb, vb


def interleave_gate_up(w_gate, w_up):
    """[2I, D] rows in the layer tail's order: 64 gate rows, then the same 64 up rows."""
    I, D = w_gate.shape
    return torch.stack([w_gate.view(I // 64, 64, D), w_up.view(I // 64, 64, D)], dim=1).reshape(2 * I, D)


def block_conv(h, w, bias, block_size, residual=False, out=None, stream=None):
    """DFlash2 local depthwise convolution along each sequence's block rows:
    out_t = sum_j w[j] * h_{t-j} + bias (+ h_t with residual).  h [B * bs, D]
    bf16, w [k, D] bf16, bias [D] or None; out may be h (in place)."""
    R, D = h.shape
    if R % block_size:
        raise ValueError("rows must be a multiple of block_size")
    if out is None:
        out = torch.empty_like(h)
    _check(lib().dflash_block_conv(_ptr(h), R // block_size, block_size, D, w.shape[0], _ptr(w), _ptr(bias),
                                   int(bool(residual)), _ptr(out), _stream(stream)))
    return out


def draft_topm_workspace_size(batch, rows_per_seq, vocab, m):
    return lib().dflash_draft_topm_workspace_size(batch, rows_per_seq, vocab, m)


def draft_topm(logits, m, temperature, lam, workspace=None, stream=None):
    """DFlash2 candidate path selector inputs for draft logits [B, R, V] bf16:
    returns (idx [B, R, m] int32, logp [B, R, m], entropy [B, R], path_score [B])."""
    B, R, V = logits.shape
    dev = logits.device
    idx = torch.empty(B, R, m, dtype=torch.int32, device=dev)
    logp = torch.empty(B, R, m, dtype=torch.float32, device=dev)
    ent = torch.empty(B, R, dtype=torch.float32, device=dev)
    score = torch.empty(B, dtype=torch.float32, device=dev)
    nbytes = draft_topm_workspace_size(B, R, V, m)
    ws = _workspace(nbytes, dev, workspace)
    _check(lib().dflash_draft_topm(_ptr(logits), B, R, V, m, float(temperature), float(lam), _ptr(idx), _ptr(logp),
                                   _ptr(ent), _ptr(score), _ptr(ws), nbytes, _stream(stream)))
    return idx, logp, ent, score


def draft_layer_tail_workspace_size(batch, block_size, num_q_heads, d_model, mlp_dim):
    return lib().dflash_draft_layer_tail_workspace_size(batch, block_size, num_q_heads, d_model, mlp_dim)


def draft_layer_tail(x, attn_out, w_o, g_post, w_gate_up, w_down, eps=1e-6, workspace=None, stream=None):
    """x [B * bs, D] (updated in place to x2), attn_out [B, Hq, bs, 128], w_gate_up from interleave_gate_up."""
    B, Hq, bs, _ = attn_out.shape
    D = x.shape[1]
    I = w_down.shape[1]
    nbytes = draft_layer_tail_workspace_size(B, bs, Hq, D, I)
    ws = _workspace(nbytes, x.device, workspace)
    _check(lib().dflash_draft_layer_tail(_ptr(x), _ptr(attn_out), B, bs, Hq, D, I, _ptr(w_o), _ptr(g_post),
                                         _ptr(w_gate_up), _ptr(w_down), float(eps), _ptr(ws), nbytes,
                                         _stream(stream)))
    return x


def draft_head_workspace_size(batch, rows_per_seq, d_model, vocab):
    return lib().dflash_draft_head_workspace_size(batch, rows_per_seq, d_model, vocab)


def draft_head(x, g_final, w_head, rows_per_seq, temperature, seed, cycle, eps=1e-6, logits=None, tokens=None,
               workspace=None, stream=None):
    """The drafter's head: final RMSNorm, LM head, draft sampling.

    x [B * rows_per_seq, D] bf16 (row b * rows_per_seq + k), w_head [V, D] bf16;
    returns (logits [B * rows_per_seq, V] bf16, tokens [B * rows_per_seq] int32)."""
    M, D = x.shape
    V = w_head.shape[0]
    if M % rows_per_seq:
        raise ValueError("rows must be a multiple of rows_per_seq")
    B = M // rows_per_seq
    dev = x.device
    if logits is None:
        logits = torch.empty(M, V, dtype=torch.bfloat16, device=dev)
    if tokens is None:
        tokens = torch.empty(M, dtype=torch.int32, device=dev)
    nbytes = draft_head_workspace_size(B, rows_per_seq, D, V)
    ws = _workspace(nbytes, dev, workspace)
    _check(lib().dflash_draft_head(_ptr(x), B, rows_per_seq, D, _ptr(g_final), float(eps), _ptr(w_head), V,
                                   float(temperature), int(seed), int(cycle), _ptr(logits), _ptr(tokens),
                                   _ptr(ws), nbytes, _stream(stream)))
    return logits, tokens


def philox4x32_10(ctr: torch.Tensor, key0: int, key1: int, stream=None) -> torch.Tensor:
    """Philox-4x32-10 of int32 counters ctr [n, 4] (bit patterns) on the GPU."""
    out = torch.empty_like(ctr)
    _check(lib().dflash_philox4x32_10(_ptr(ctr), key0 & 0xFFFFFFFF, key1 & 0xFFFFFFFF, _ptr(out),
                                      ctr.shape[0], _stream(stream)))
    return out


def read_device_status(stream=None) -> int:
    """Synchronise, return and clear the library's device status bits."""
    v = ctypes.c_uint32(0)
    _check(lib().dflash_read_device_status(ctypes.byref(v), _stream(stream)))
    return int(v.value)
