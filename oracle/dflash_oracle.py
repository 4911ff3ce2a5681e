"""Plain float64 reference for the three steps of one DFlash draft-and-verify cycle.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module.

Sources (the DFlash pages, cited by title and section):
  [E4B]  "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash"
         (flozi.net, English) -- sections "The released serving cycle",
         "Five target states become persistent draft context",
         "Why exact verification preserves the target",
         "The parameter count exposes the real cost",
         "Cache and latency have separate break-even points".
  [DF2]  "DFlash & DFlash2: Block-Diffusion LLM-Speedup" (xencorenexus.com,
         German) -- section 4.1 (fusion formula H_t = RMSNorm(W_c[...]) and
         the K/V injection formulas), section 4.4 (acceptance probability,
         residual distribution, greedy rule), section 9 FAQ Q3 (temperature).
  [PHX]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
         1, 2, 3", SC'11 -- the Philox-4xW-R counter-based generator.

Readings taken where the pages are silent or garbled (each one is listed in
the design notes too):
  * RMSNorm after the fusion projection: yes ([DF2] 4.1 is the only surviving
    formula); eps is a parameter (1e-6 by default); the gain g is an input.
  * W_c is used in the pages' orientation, W_c in R^{D x J*d_t}:
    Y = concat(taps) @ W_c^T.  Tap order = ascending target layer id.
  * Per-head Q/K RMSNorm ([E4B] "Five target states...") applies to every key,
    cached context keys and block keys alike; V is not normalised.
  * RoPE: rotate-half pairing (e, e + d/2), inverse frequency
    theta^(-2e/d), theta = 1e6 by default; angle formed in float64.
  * Positions: cached context row t of a sequence sits at position t; block
    row j sits at position seq_len + j (the anchor at seq_len).
  * Attention scale 1/sqrt(d); the block is non-causal (every block row sees
    every block key and every cached key in the window).
  * Row alignment of verification: target row k and draft row k score draft
    token x_{k+1}; target row bs-1 gives the bonus token.
  * Temperature: both logit rows are divided by T before the softmax
    ([DF2] FAQ Q3 prints the 1/T power on probabilities, which is garbled);
    T = 0 selects the greedy rule.
  * Acceptance: accept iff u < alpha ([DF2] 4.4 rejects when r > alpha; the
    two differ only at u == alpha).
  * Sampling from the normalised residual (and the bonus draw from p):
    inverse CDF in vocabulary order -- the first index y whose cumulative
    mass exceeds v * S.  If the residual mass S is 0 (possible only through
    rounding), the draw is taken from p instead.
  * Ties in greedy argmax go to the lowest index.
  * Uniforms: one Philox-4x32-10 block per (row k, sequence b, cycle):
    counter = (k, b, cycle_lo, cycle_hi), key = (seed_lo, seed_hi);
    word 0 -> acceptance uniform, word 1 -> draw uniform;
    uniform(w) = (w >> 8) * 2^-24 in [0, 1).
  * bfloat16 storage points (bf16 workloads only): the fused context H_t, the
    cache K/V, the block prologue outputs q^, k^_b and the attention output.
    Rounding is round-to-nearest-even of the float32 value.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F64 = np.float64

# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------


def round_to_bf16(x):
    """Round to bfloat16 (round-to-nearest-even of the float32 value).

    Returns float64 holding exactly representable bfloat16 values.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x32.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(F64)


# --------------------------------------------------------------------------
# Philox-4xW-R  [PHX]
# --------------------------------------------------------------------------

# Round multipliers and Weyl key increments, as published in [PHX].
_PHILOX = {
    32: dict(mult=(0xD2511F53, 0xCD9E8D57), weyl=(0x9E3779B9, 0xBB67AE85)),
    64: dict(mult=(0xD2E7470EE14C6C93, 0xCA5A826395121157),
             weyl=(0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)),
}


def _u64(v):
    return np.atleast_1d(np.asarray(v, dtype=np.uint64))


def _mulhilo(a, b, width):
    """(hi, lo) words of the 2*width-bit product a*b."""
    if width == 32:
        p = a * b  # < 2^64, exact in uint64
        return p >> np.uint64(32), p & np.uint64(0xFFFFFFFF)
    m32 = np.uint64(0xFFFFFFFF)
    s32 = np.uint64(32)
    a0, a1 = a & m32, a >> s32
    b0, b1 = b & m32, b >> s32
    p00, p01, p10, p11 = a0 * b0, a0 * b1, a1 * b0, a1 * b1
    mid = (p00 >> s32) + (p01 & m32) + (p10 & m32)
    lo = (p00 & m32) | ((mid & m32) << s32)
    hi = p11 + (p01 >> s32) + (p10 >> s32) + (mid >> s32)
    return hi, lo


def philox4(ctr, key, width=32, rounds=10):
    """Philox-4xW-R of [PHX], vectorised over arrays of counters.

    ctr: 4 arrays (or scalars) of W-bit words; key: 2 of them.  Each round maps
    (c0, c1, c2, c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1,
    lo(M0*c0)); the key is bumped by the Weyl constants between rounds.
    Returns 4 uint64 arrays holding W-bit words.
    """
    const = _PHILOX[width]
    mask = np.uint64((1 << width) - 1)
    m0, m1 = (np.uint64(v) for v in const["mult"])
    w0, w1 = (np.uint64(v) for v in const["weyl"])
    c0, c1, c2, c3 = np.broadcast_arrays(*[_u64(c) for c in ctr])
    c0, c1, c2, c3 = (np.array(c, dtype=np.uint64) for c in (c0, c1, c2, c3))
    k0, k1 = (_u64(k) for k in key)
    with np.errstate(over="ignore"):
        for r in range(rounds):
            if r > 0:
                k0 = (k0 + w0) & mask
                k1 = (k1 + w1) & mask
            hi0, lo0 = _mulhilo(m0, c0, width)
            hi1, lo1 = _mulhilo(m1, c2, width)
            c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & mask, lo1 & mask, (hi0 ^ c3 ^ k1) & mask, lo0 & mask
    return c0, c1, c2, c3


def philox4x32_10(ctr, key):
    """Philox-4x32-10 of [PHX]; returns 4 uint32 arrays."""
    return tuple(w.astype(np.uint32) for w in philox4(ctr, key, width=32, rounds=10))


def _uniform24(w):
    """(w >> 8) * 2^-24: a float32-exact uniform in [0, 1)."""
    return (np.asarray(w, dtype=np.uint64) >> np.uint64(8)).astype(F64) * (2.0 ** -24)


def verify_uniforms(seed, cycle, k, b):
    """(acceptance uniform, draw uniform) for row k of sequence b in a cycle.

    Counter = (k, b, cycle_lo, cycle_hi), key = (seed_lo, seed_hi); the first
    two output words become the two uniforms (reading taken: the pages give no
    random-number convention).
    """
    seed = int(seed)
    cycle = int(cycle)
    w = philox4x32_10((k, b, cycle & 0xFFFFFFFF, (cycle >> 32) & 0xFFFFFFFF),
                      (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    return _uniform24(w[0]), _uniform24(w[1])


# --------------------------------------------------------------------------
# normalisation and rotary position embedding
# --------------------------------------------------------------------------


def rms_norm(x, gain, eps):
    """x / sqrt(mean(x^2) + eps) * gain over the last axis ([DF2] 4.1 RMSNorm;
    [E4B] per-head Q/K RMS normalisation)."""
    x = np.asarray(x, dtype=F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gain, F64)


def rope_inv_freq(d, theta):
    """Inverse frequencies theta^(-2e/d), e = 0 .. d/2-1 (reading: standard RoPE)."""
    e = np.arange(d // 2, dtype=F64)
    return float(theta) ** (-2.0 * e / d)


def rope(x, pos, theta):
    """Rotate pairs (e, e + d/2) of x[..., d] by angle pos * theta^(-2e/d).

    pos broadcasts against x[..., 0].  [E4B]: RoPE is applied after the
    per-head Q/K RMS normalisation.
    """
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=F64)[..., None] * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------
# step 1: context fusion and K/V injection  ([E4B] "Five target states...",
#         [DF2] 4.1)
# --------------------------------------------------------------------------


def fuse_rows(taps, w_fuse, g_fuse, w_kv, k_gain, positions, num_layers, num_kv_heads,
              head_dim, theta=1e6, eps=1e-6, bf16=False):
    """Fuse context rows and project them into per-layer K/V entries.

    taps      : list of J arrays [M, d_t]  (captured target hidden states; the
                pages' E4B drafter uses layers 5, 11, 17, 23, 35)
    w_fuse    : [D, J*d_t]  W_c of [DF2] 4.1
    g_fuse    : [D]         RMSNorm gain
    w_kv      : [L*2*Hkv*d, D]; output column ((l*2 + s)*Hkv + h)*d + e,
                s = 0 for K, 1 for V  (the K/V projections of all layers as one
                matrix, [E4B] "...fuse unquantized K/V projections...")
    k_gain    : [L, d]      per-layer key-norm gain
    positions : [M]         cache position of each row
    Returns (H_t [M, D], K [M, L, Hkv, d], V [M, L, Hkv, d]).

    H_t = RMSNorm(concat(taps) @ W_c^T) ([DF2] 4.1); K_i = W_i^K H_t and
    V_i = W_i^V H_t ([DF2] 4.1, context half of the K/V injection); every key
    then gets the per-head RMSNorm and RoPE of [E4B].
    """
    X = np.concatenate([np.asarray(t, dtype=F64) for t in taps], axis=1)
    Y = X @ np.asarray(w_fuse, dtype=F64).T
    H = rms_norm(Y, g_fuse, eps)
    if bf16:
        H = round_to_bf16(H)
    KV = H @ np.asarray(w_kv, dtype=F64).T
    M = KV.shape[0]
    KV = KV.reshape(M, num_layers, 2, num_kv_heads, head_dim)
    K = KV[:, :, 0]
    V = KV[:, :, 1]
    pos = np.asarray(positions, dtype=F64)
    Kn = rms_norm(K, np.asarray(k_gain, F64)[None, :, None, :], eps)
    Kr = rope(Kn, pos[:, None, None], theta)
    if bf16:
        Kr, V = round_to_bf16(Kr), round_to_bf16(V)
    return H, Kr, V


def fuse_context(taps, cu_new, seq_len, w_fuse, g_fuse, w_kv, k_gain, cache_k, cache_v,
                 theta=1e6, eps=1e-6, bf16=False):
    """Fuse the new context rows of every sequence and append them to the cache.

    cu_new [B+1] row offsets (rows of sequence b are cu_new[b] .. cu_new[b+1]-1),
    seq_len [B]; cache_k / cache_v [L, B, Hkv, cap, d] are updated in place at
    positions seq_len[b] + t.  seq_len itself is not advanced.
    Returns H_t [M, D].
    """
    cu_new = np.asarray(cu_new, dtype=np.int64)
    seq_len = np.asarray(seq_len, dtype=np.int64)
    L, B, Hkv, cap, d = cache_k.shape
    M = int(cu_new[-1])
    positions = np.empty(M, dtype=np.int64)
    seq_of_row = np.empty(M, dtype=np.int64)
    for b in range(B):
        n = int(cu_new[b + 1] - cu_new[b])
        if seq_len[b] + n > cap:
            raise ValueError("sequence %d: seq_len + n_new exceeds the cache capacity" % b)
        positions[cu_new[b]:cu_new[b + 1]] = seq_len[b] + np.arange(n)
        seq_of_row[cu_new[b]:cu_new[b + 1]] = b
    H, K, V = fuse_rows(taps, w_fuse, g_fuse, w_kv, k_gain, positions, L, Hkv, d, theta, eps, bf16)
    for m in range(M):
        b, p = seq_of_row[m], positions[m]
        cache_k[:, b, :, p, :] = K[m]
        cache_v[:, b, :, p, :] = V[m]
    return H


# --------------------------------------------------------------------------
# step 2: non-causal draft-block attention  ([E4B] "The released serving
#         cycle" step 3 and "Five target states..."; [DF2] 4.1 K/V injection)
# --------------------------------------------------------------------------


def block_attn(q, kb, vb, q_gain, k_gain, cache_k, cache_v, seq_len, theta=1e6, eps=1e-6,
               window=0, bf16=False):
    """One draft layer's block attention.

    q  [B, Hq, bs, d], kb / vb [B, Hkv, bs, d]: the block's projections
    cache_k / cache_v [B, Hkv, cap, d]: this layer's cache (already normed and
    rotated); seq_len [B]; window 0 = the whole cached context, else the latest
    `window` cached positions.
    Query head h reads KV head h // (Hq / Hkv).  Block row j sits at position
    seq_len[b] + j; every block row attends to every key of the window and to
    all bs block keys (non-causal inside the block).
    Returns O [B, Hq, bs, d].
    """
    q = np.asarray(q, F64)
    kb = np.asarray(kb, F64)
    vb = np.asarray(vb, F64)
    B, Hq, bs, d = q.shape
    Hkv = kb.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, bs, d), dtype=F64)
    for b in range(B):
        n = int(seq_len[b])
        pos = n + np.arange(bs)
        qh = rope(rms_norm(q[b], q_gain, eps), pos, theta)
        kh = rope(rms_norm(kb[b], k_gain, eps), pos, theta)
        if bf16:
            qh, kh = round_to_bf16(qh), round_to_bf16(kh)
        lo = max(0, n - window) if window > 0 else 0
        for g in range(Hkv):
            keys = np.concatenate([np.asarray(cache_k[b, g, lo:n], F64), kh[g]], axis=0)
            vals = np.concatenate([np.asarray(cache_v[b, g, lo:n], F64), vb[b, g]], axis=0)
            Q = qh[g * G:(g + 1) * G].reshape(G * bs, d)
            s = Q @ keys.T / np.sqrt(d)
            s = s - s.max(axis=-1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=-1, keepdims=True)
            out[b, g * G:(g + 1) * G] = (p @ vals).reshape(G, bs, d)
    if bf16:
        out = round_to_bf16(out)
    return out


# --------------------------------------------------------------------------
# step 3: exact speculative verification  ([E4B] "Why exact verification
#         preserves the target"; [DF2] 4.4 and FAQ Q3)
# --------------------------------------------------------------------------

BOUNDARY_EPS = 1e-6


@dataclass
class VerifyResult:
    accepted_len: np.ndarray   # [B] int32 in [0, bs-1]
    out_tokens: np.ndarray     # [B, bs] int32; accepted_len+1 valid, rest -1
    near_tie: np.ndarray       # [B] bool: some decision was within BOUNDARY_EPS


def _log_softmax(l):
    m = l.max(axis=-1, keepdims=True)
    return l - (m + np.log(np.exp(l - m).sum(axis=-1, keepdims=True)))


def _categorical_draw(weights, v):
    """Inverse-CDF draw per row: first index y with cumsum(w)[y] > v * sum(w).

    Returns (index, near_tie) where near_tie flags rows whose uniform v lies
    within BOUNDARY_EPS of either edge of the chosen bin, the edges taken on
    the uniform's own scale: cumulative mass divided by the total, the values
    of v at which the draw would change.
    """
    C = np.cumsum(weights, axis=-1)
    S = C[:, -1]
    t = v * S
    y = np.argmax(C > t[:, None], axis=-1)
    rows = np.arange(weights.shape[0])
    upper = C[rows, y]
    lower = np.where(y > 0, C[rows, np.maximum(y - 1, 0)], 0.0)
    tie = ((t - lower) < BOUNDARY_EPS * S) | ((upper - t) < BOUNDARY_EPS * S)
    return y, tie


def verify(target_logits, draft_logits, draft_tokens, temperature, seed, cycle, seq_ids=None):
    """Speculative verification of one drafted block per sequence.

    target_logits [B, bs, V]: row k is the target's scores for the position of
    draft token x_{k+1} (row bs-1 scores the bonus position);
    draft_logits [B, bs-1, V]: row k is the drafter's q for x_{k+1};
    draft_tokens [B, bs-1]; seq_ids [B] optional sequence indices used in the
    random-number counter (default 0 .. B-1), so that a subset of a batch can
    be checked on its own.

    T > 0, row k = 0 .. bs-2 in order ([DF2] 4.4, [E4B] "Why exact
    verification..."):  p = softmax(l_t / T), q = softmax(l_d / T);
    alpha = min(1, p(x) / q(x)); accept iff u < alpha.  At the first rejection
    emit a draw from max(0, p - q) normalised, and stop.  If every draft is
    accepted, emit a draw from p of row bs-1 (the bonus token; the maximum
    acceptance length is bs tokens including it).
    T == 0: accept while x equals argmax of the target row; at the first
    mismatch emit that argmax; the bonus is the argmax of row bs-1.
    """
    lt = np.asarray(target_logits, dtype=F64)
    B, bs, V = lt.shape
    x = np.asarray(draft_tokens, dtype=np.int64).reshape(B, bs - 1)
    if np.any((x < 0) | (x >= V)):
        raise ValueError("draft token out of range")
    T = float(temperature)
    n = np.full(B, bs - 1, dtype=np.int64)      # accepted count
    alive = np.ones(B, dtype=bool)
    near = np.zeros(B, dtype=bool)
    rows_b = np.arange(B)
    ids = rows_b if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    if T == 0.0:
        tmax = lt.argmax(axis=-1)                # [B, bs], lowest index on ties
        for k in range(bs - 1):
            acc = tmax[:, k] == x[:, k]
            n[alive & ~acc] = k
            alive &= acc
        corr = tmax[rows_b, n]
    else:
        ld = np.asarray(draft_logits, dtype=F64).reshape(B, bs - 1, V)
        u = np.empty((B, bs))
        v = np.empty((B, bs))
        for k in range(bs):
            u[:, k], v[:, k] = verify_uniforms(seed, cycle, k, ids)
        for k in range(bs - 1):
            lp = _log_softmax(lt[:, k] / T)
            lq = _log_softmax(ld[:, k] / T)
            alpha = np.minimum(1.0, np.exp(lp[rows_b, x[:, k]] - lq[rows_b, x[:, k]]))
            # the decision is taken on alpha rounded to float32 (the kernel's
            # precision); u is float32-exact
            acc = u[:, k] < alpha.astype(np.float32).astype(F64)
            near |= alive & (np.abs(u[:, k] - alpha) < BOUNDARY_EPS)
            n[alive & ~acc] = k
            alive &= acc
        # correction (first rejected row) or bonus (row bs-1)
        W = np.empty((B, V))
        for b in range(B):
            k = n[b]
            p = np.exp(_log_softmax(lt[b, k] / T))
            if k < bs - 1:
                q = np.exp(_log_softmax(ld[b, k] / T))
                r = np.maximum(0.0, p - q)
                W[b] = r if r.sum() > 0.0 else p
            else:
                W[b] = p
        corr, tie = _categorical_draw(W, v[rows_b, n])
        near |= tie
    out = np.full((B, bs), -1, dtype=np.int64)
    for b in range(B):
        out[b, :n[b]] = x[b, :n[b]]
        out[b, n[b]] = corr[b]
    return VerifyResult(n.astype(np.int32), out.astype(np.int32), near)


# --------------------------------------------------------------------------
# step 4: the drafter's head -- final RMSNorm, LM head, draft sampling
#         ([E4B] "The released serving cycle": the drafter proposes the block's
#         tokens from its final hidden states through the LM head; "The
#         parameter count exposes the real cost": the head is V x D)
# --------------------------------------------------------------------------

def silu(z):
    """z * sigmoid(z)."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def draft_layer_qkv(x, g_in, w_qkv, batch, num_q_heads, num_kv_heads, head_dim=128, eps=1e-6, bf16=False):
    """The start of one draft layer: its input RMSNorm and the block rows' q, k
    and v projections (Qwen3-style layer, [E4B] "The parameter count exposes
    the real cost": q/k/v/o projections and two RMSNorms per layer).

    x [M, D] residual stream of the block rows (row b * bs + j, M = batch * bs),
    g_in [D] the input norm's gain, w_qkv [(Hq + 2 Hkv) * hd, D] whose output
    rows are the Hq query heads, then the Hkv key heads, then the Hkv value
    heads, head h's element e at row h * hd + e:
      h   = RMSNorm(x) * g_in
      y   = h w_qkv^T
      q[b, h, j, e]  = y[b*bs + j, h*hd + e]
      kb[b, g, j, e] = y[b*bs + j, (Hq + g)*hd + e]
      vb[b, g, j, e] = y[b*bs + j, (Hq + Hkv + g)*hd + e]
    The per-head Q/K norms and RoPE belong to the block attention.  Returns
    (q [B, Hq, bs, hd], kb [B, Hkv, bs, hd], vb [B, Hkv, bs, hd]).  bf16: the
    normalised rows and the three outputs are stored as bfloat16.
    """
    rnd = round_to_bf16 if bf16 else (lambda v: v)
    x = np.asarray(x, dtype=F64)
    M = x.shape[0]
    bs = M // batch
    h = rnd(rms_norm(x, np.asarray(g_in, dtype=F64), eps))
    y = h @ np.asarray(w_qkv, dtype=F64).T
    heads = y.reshape(batch, bs, num_q_heads + 2 * num_kv_heads, head_dim).transpose(0, 2, 1, 3)
    q = rnd(heads[:, :num_q_heads])
    kb = rnd(heads[:, num_q_heads:num_q_heads + num_kv_heads])
    vb = rnd(heads[:, num_q_heads + num_kv_heads:])
    return q, kb, vb


def draft_layer_tail(x, o, w_o, g_post, w_gate, w_up, w_down, eps=1e-6, bf16=False):
    """The rest of one draft layer after its attention (Qwen3-style layer,
    [E4B] "The parameter count exposes the real cost": q/k/v/o projections, a
    gated MLP of intermediate size I, two RMSNorms per layer).

    x [M, D] residual stream of the block rows (row b * bs + j), o [B, Hq, bs,
    hd] the attention output, w_o [D, Hq*hd], g_post [D], w_gate / w_up [I, D],
    w_down [D, I]:
      x1 = x + o_flat w_o^T          (o_flat row b*bs + j = o[b, :, j, :] flattened)
      h  = RMSNorm(x1) * g_post
      a  = silu(h w_gate^T) * (h w_up^T)
      x2 = x1 + a w_down^T
    Returns (x1, x2).  bf16: x1, h, a and x2 are stored as bfloat16.
    """
    rnd = round_to_bf16 if bf16 else (lambda v: v)
    x = np.asarray(x, dtype=F64)
    o = np.asarray(o, dtype=F64)
    B, Hq, bs, hd = o.shape
    o_flat = o.transpose(0, 2, 1, 3).reshape(B * bs, Hq * hd)
    x1 = rnd(x + o_flat @ np.asarray(w_o, dtype=F64).T)
    h = rnd(rms_norm(x1, np.asarray(g_post, dtype=F64), eps))
    a = rnd(silu(h @ np.asarray(w_gate, dtype=F64).T) * (h @ np.asarray(w_up, dtype=F64).T))
    x2 = rnd(x1 + a @ np.asarray(w_down, dtype=F64).T)
    return x1, x2


DRAFT_TAG = 0x80000000  # top bit of the fourth counter word: draft sampling


def draft_head(x, g_final, w_head, eps=1e-6, bf16=False):
    """Draft logits of the proposal rows.

    x [R, D] final hidden states, g_final [D], w_head [V, D] (row v = token v):
    logits = RMSNorm(x) * g_final @ w_head^T.  bf16: the normalised rows are
    stored as bfloat16 before the product and the logits are rounded to
    bfloat16 (the kernel's storage points).
    """
    h = rms_norm(np.asarray(x, dtype=F64), np.asarray(g_final, dtype=F64), eps)
    if bf16:
        h = round_to_bf16(h)
    z = h @ np.asarray(w_head, dtype=F64).T
    return round_to_bf16(z) if bf16 else z


def draft_race_uniforms(seed, cycle, b, k, V):
    """U(0,1] for every vocabulary index y of proposal row k of sequence b.

    One Philox-4x32-10 block per 4 consecutive indices: counter =
    (y >> 2, (b << 5) | k, cycle_lo, cycle_hi | DRAFT_TAG), key = (seed_lo,
    seed_hi); index y takes word y & 3; U = ((w >> 8) + 1) * 2^-24.  The tag
    bit keeps these counters apart from the verification's (k, b, cycle_lo,
    cycle_hi) for cycles below 2^63 (reading taken: the pages give no
    random-number convention).
    """
    seed, cycle = int(seed), int(cycle)
    nb = (V + 3) // 4
    w = philox4x32_10((np.arange(nb, dtype=np.uint64), (int(b) << 5) | int(k), cycle & 0xFFFFFFFF,
                       ((cycle >> 32) & 0x7FFFFFFF) | DRAFT_TAG),
                      (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    words = np.stack([np.asarray(x, dtype=np.uint64) for x in w], axis=1).reshape(-1)[:V]
    return ((words >> np.uint64(8)) + np.uint64(1)).astype(F64) * (2.0 ** -24)


DRAFT_TIE_EPS = 1e-4


def draft_sample(logits, temperature, seed, cycle, seq_ids=None, row_ids=None):
    """Draft tokens from the proposal rows' logits [B, R, V].

    T > 0: the exponential race -- y* = argmax_y q(y) / E_y with E_y = -ln U_y,
    i.e. argmax_y logits[y] / T - ln(-ln U_y), a draw from softmax(logits / T)
    (no normalisation needed).  T == 0: argmax of the logits.  Ties go to the
    lowest index.  Returns (tokens [B, R] int64, near_tie [B, R] bool): a row is
    flagged when its two largest keys are within DRAFT_TIE_EPS.  seq_ids [B] and
    row_ids [R] (default 0 .. B-1, 0 .. R-1) are the sequence and proposal-row
    numbers used in the random-number counter, so that a subset can be checked.
    """
    z = np.asarray(logits, dtype=F64)
    B, R, V = z.shape
    ids = np.arange(B) if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    kid = np.arange(R) if row_ids is None else np.asarray(row_ids, dtype=np.int64)
    T = float(temperature)
    tok = np.zeros((B, R), dtype=np.int64)
    near = np.zeros((B, R), dtype=bool)
    for b in range(B):
        for k in range(R):
            key = z[b, k].copy()
            if T > 0.0:
                u = draft_race_uniforms(seed, cycle, ids[b], kid[k], V)
                with np.errstate(divide="ignore"):  # U = 1: E = 0 and the key is +inf (that index wins)
                    key = key / T - np.log(-np.log(u))
            y = int(np.argmax(key))  # first maximum = lowest index
            tok[b, k] = y
            if V > 1:
                top2 = np.partition(key, V - 2)[V - 2:]
                near[b, k] = (top2[1] - top2[0]) < DRAFT_TIE_EPS
    return tok, near


# --------------------------------------------------------------------------
# size arithmetic printed by the pages ([E4B] "The parameter count exposes the
# real cost", "Cache and latency have separate break-even points"; [DF2] 4.1)
# --------------------------------------------------------------------------


def draft_param_count(vocab, d_model, num_taps, d_target, num_layers, num_q_heads,
                      num_kv_heads, head_dim, mlp_dim):
    """Logical parameters of a DFlash drafter with a Qwen3-style layer.

    LM head V*D, fusion W_c (J*d_t)*D, per layer q/k/v/o projections, a
    gated MLP (3*D*I), two RMSNorm gains of D and the per-head q/k norm gains
    of d, plus the fusion norm and the final norm (2*D).  The embedding is
    shared with the target and not counted ([E4B]).
    """
    attn = d_model * num_q_heads * head_dim + 2 * d_model * num_kv_heads * head_dim \
        + num_q_heads * head_dim * d_model
    layer = attn + 3 * d_model * mlp_dim + 2 * d_model + 2 * head_dim
    return vocab * d_model + num_taps * d_target * d_model + num_layers * layer + 2 * d_model


def kv_cache_payload_bytes(num_layers, num_kv_heads, positions, head_dim, bytes_per_elem):
    """Logical K+V cache payload of one sequence ([E4B] cache section)."""
    return num_layers * num_kv_heads * positions * head_dim * 2 * bytes_per_elem


def fusion_weight_bytes(d_model, num_taps, bytes_per_elem):
    """Bytes of W_c in R^{D x J*D} ([DF2] 4.1 memory-overhead example)."""
    return d_model * num_taps * d_model * bytes_per_elem


def gather_pages(pool, block_table, page_size):
    """Linear cache view [L][B][Hkv][max_pages * page_size][d] of a paged pool.

    [E4B] "Cache and latency have separate break-even points" counts the
    per-sequence cache payload before paging; [DF2] 7.2 has the serving stack
    keep the draft cache in paged memory.  Neither fixes a layout; this one is
    the library's: pool [L][num_pages][Hkv][page_size][d], and position p of
    sequence b is row p % page_size of page block_table[b, p // page_size].
    Entries outside [0, num_pages) give zero rows.
    """
    pool = np.asarray(pool)
    table = np.asarray(block_table)
    L, NP, H, P, d = pool.shape
    assert P == page_size
    B, MP = table.shape
    out = np.zeros((L, B, H, MP * P, d), dtype=pool.dtype)
    for b in range(B):
        for j in range(MP):
            pg = int(table[b, j])
            if 0 <= pg < NP:
                out[:, b, :, j * P:(j + 1) * P, :] = pool[:, pg]
    return out


# DFlash2 variants  ([DF2] 5 "DFlash2 innovations": local depthwise
# convolutions and the candidate path selector)

def block_conv(h, w, bias, block_size, residual=False):
    """[DF2] 5.1: ConvOutput_t = sum_{j=0}^{k-1} W_conv,j (.) H_{t-j} + b_conv,
    a depthwise (per-channel) 1D convolution along the block positions.

    h [B * block_size, D]: the block rows of B sequences, sequence-major; w
    [k, D]; bias [D] or None.  Readings: positions before a block's first row
    contribute zero (the sum stays within one sequence's block and only looks
    back); with residual the output is h + ConvOutput (the convolution as a
    sub-layer on the residual stream between attention and the MLP).
    """
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    R, D = h.shape
    k = w.shape[0]
    out = np.zeros_like(h)
    for r in range(R):
        t = r % block_size
        acc = np.zeros(D) if bias is None else np.asarray(bias, dtype=np.float64).copy()
        for j in range(k):
            if t - j >= 0:
                acc = acc + w[j] * h[r - j]
        out[r] = acc
    return h + out if residual else out


def draft_topm(logits, m, temperature, lam):
    """[DF2] 5.2: the draft head's top-m candidates per block position and the
    path score S(path) = sum_j log P_draft(x_j^(m_j)) + lam * Entropy(P_draft(x_j)).

    logits [B, R, V] (R draft positions per sequence), P_draft = softmax(l / T),
    T > 0.  Per row: the m candidates by logit (descending, ties to the lower
    index; dividing by T > 0 keeps the order), their log-probabilities, and the
    entropy -sum p ln p.  The score is a sum of per-position terms and the
    entropy term does not depend on the choice, so the best path takes every
    position's first candidate; its score is returned per sequence.
    Returns (idx [B, R, m] int64, logp [B, R, m], entropy [B, R], best [B]).
    """
    l = np.asarray(logits, dtype=np.float64)
    B, R, V = l.shape
    s = l / temperature
    mx = s.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(mx[..., 0])     # a row of -inf logits carries no probability mass
    mxs = np.where(np.isfinite(mx), mx, 0.0)
    with np.errstate(divide="ignore"):   # ln 0 of an empty row is replaced just below
        logz = np.where(empty, -np.inf, mxs[..., 0] + np.log(np.exp(s - mxs).sum(axis=-1)))
    logp_all = np.where(empty[..., None], -np.inf, s - np.where(empty, 0.0, logz)[..., None])
    p = np.exp(logp_all)
    plogp = np.where(p > 0, p * np.where(p > 0, logp_all, 0.0), 0.0)   # 0 ln 0 = 0 (tokens of zero probability)
    ent = -plogp.sum(axis=-1)
    idx = np.zeros((B, R, m), dtype=np.int64)
    for b in range(B):
        for r in range(R):
            order = sorted(range(V), key=lambda y: (-l[b, r, y], y))   # descending, lower index first
            idx[b, r] = order[:m]
    logp = np.take_along_axis(logp_all, idx, axis=-1)
    best = logp[..., 0].sum(axis=-1) + lam * ent.sum(axis=-1)
    return idx, logp, ent, best


def path_score(logp, entropy, choice, lam):
    """S of one path ([DF2] 5.2): choice [B, R] picks candidate choice[b, r] of
    each position from logp [B, R, m]; entropy [B, R]."""
    logp = np.asarray(logp, dtype=np.float64)
    ch = np.asarray(choice)
    sel = np.take_along_axis(logp, ch[..., None], axis=-1)[..., 0]
    return sel.sum(axis=-1) + lam * np.asarray(entropy, dtype=np.float64).sum(axis=-1)
