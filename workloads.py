"""Seeded synthetic inputs for the DFlash cycle workloads.

Input generation only: this module holds none of the method's arithmetic.  It
is shared by the tests (which feed the same tensors to the CUDA path and to
the CPU oracle) and by bench.py.  Shapes and value distributions follow the
workloads the hot path is measured on:

  tiny_fp32      B=1, S=64 context rows fused into an empty cache, bs=8, L=1,
                 fp32, V=4096, target logits N(0,2), draft = target + N(0,0.5)
  single_stream  B=1, S=4096, L=5, bs=8, bf16, V=262144,
                 target N(0,3), draft = target + N(0,1)
  batched        B=32, per-sequence S uniform in [1024, 8192], L=5, bs=8, bf16,
                 V=262144, logits as single_stream, 20% of the sequences with
                 draft logits equal to the target logits (all-accept path)
  high_batch     B=128, S=2048, L=5, bs in {4, 8, 16}, draft noise sigma in
                 {0.25, 1, 4}
  long_context   B=4, S=131072, L=5, bs=8; prefill fusion of 2048-row chunks

Common to all: GQA 32/8, head 128, draft width D = 2560, five taps of width
2560, fusion and K/V weights N(0, 0.02), norm gains 1 + N(0, 0.1), block
Q/K/V N(0, 1), cached K/V N(0, 1) (already normalised and rotated), hidden
states N(0, 1).  Draft tokens are drawn from the draft distribution
(Gumbel-max on logits/T, argmax at T = 0) by this module, like the drafter's
own sampler would.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class CycleConfig:
    name: str
    B: int
    S: int                      # cached context (max when ragged)
    S_min: int | None = None    # ragged: per-sequence S uniform in [S_min, S]
    bs: int = 8
    L: int = 5
    Hq: int = 32
    Hkv: int = 8
    d: int = 128
    D: int = 2560
    mlp_dim: int = 5120         # drafter layer MLP width
    J: int = 5
    d_target: int = 2560
    V: int = 262144
    dtype: torch.dtype = torch.bfloat16
    logit_std: float = 3.0
    draft_noise: float = 1.0
    all_accept_frac: float = 0.0
    temperature: float = 1.0
    fuse_rows_per_seq: int | None = None   # None: bs rows per sequence (one cycle)
    seed: int = 0

    @property
    def capacity(self) -> int:
        extra = max(self.bs, self.fuse_rows_per_seq or 0)
        return int(math.ceil((self.S + extra) / 64.0)) * 64


TINY_FP32 = CycleConfig("tiny_fp32", B=1, S=64, bs=8, L=1, V=4096, dtype=torch.float32, logit_std=2.0,
                        draft_noise=0.5, temperature=1.0, fuse_rows_per_seq=64, seed=1)
SINGLE_STREAM = CycleConfig("single_stream", B=1, S=4096, seed=2)
BATCHED = CycleConfig("batched", B=32, S=8192, S_min=1024, all_accept_frac=0.2, seed=3)
HIGH_BATCH = CycleConfig("high_batch", B=128, S=2048, seed=4)
LONG_CONTEXT = CycleConfig("long_context", B=4, S=131072, seed=5)

CONFIGS = {c.name: c for c in (TINY_FP32, SINGLE_STREAM, BATCHED, HIGH_BATCH, LONG_CONTEXT)}


def high_batch(bs: int, sigma: float) -> CycleConfig:
    return replace(HIGH_BATCH, bs=bs, draft_noise=sigma, name="high_batch_bs%d_sigma%g" % (bs, sigma))


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, std, gen, device, dtype):
    return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)


def seq_lens(cfg: CycleConfig, device="cpu") -> torch.Tensor:
    """Per-sequence cached lengths (int32)."""
    if cfg.S_min is None:
        return torch.full((cfg.B,), cfg.S, dtype=torch.int32, device=device)
    g = generator(cfg.seed * 1000 + 1, "cpu")
    s = torch.randint(cfg.S_min, cfg.S + 1, (cfg.B,), generator=g, dtype=torch.int32)
    return s.to(device)


@dataclass
class Weights:
    w_fuse: torch.Tensor    # [D, J*d_target]
    g_fuse: torch.Tensor    # [D]
    w_kv: torch.Tensor      # [L*2*Hkv*d, D]
    k_gain: torch.Tensor    # [L, d]
    q_gain: torch.Tensor    # [L, d]


def weights(cfg: CycleConfig, device="cpu") -> Weights:
    g = generator(cfg.seed * 1000 + 2, device)
    dt = cfg.dtype
    w_fuse = _randn((cfg.D, cfg.J * cfg.d_target), 0.02, g, device, dt)
    g_fuse = (1.0 + _randn((cfg.D,), 0.1, g, device, torch.float32)).to(dt)
    w_kv = _randn((cfg.L * 2 * cfg.Hkv * cfg.d, cfg.D), 0.02, g, device, dt)
    k_gain = (1.0 + _randn((cfg.L, cfg.d), 0.1, g, device, torch.float32)).to(dt)
    q_gain = (1.0 + _randn((cfg.L, cfg.d), 0.1, g, device, torch.float32)).to(dt)
    return Weights(w_fuse, g_fuse, w_kv, k_gain, q_gain)


def cache(cfg: CycleConfig, device="cpu", layers=None, fill=True):
    """(k, v) [L, B, Hkv, cap, d]; N(0, 1) contents when `fill`, zeros otherwise."""
    L = cfg.L if layers is None else layers
    shape = (L, cfg.B, cfg.Hkv, cfg.capacity, cfg.d)
    if not fill:
        return torch.zeros(shape, dtype=cfg.dtype, device=device), torch.zeros(shape, dtype=cfg.dtype, device=device)
    g = generator(cfg.seed * 1000 + 3, device)
    return _randn(shape, 1.0, g, device, cfg.dtype), _randn(shape, 1.0, g, device, cfg.dtype)


def taps(cfg: CycleConfig, rows: int, device="cpu", seed_offset=0):
    g = generator(cfg.seed * 1000 + 4 + seed_offset, device)
    return [_randn((rows, cfg.d_target), 1.0, g, device, cfg.dtype) for _ in range(cfg.J)]


def cu_rows(n_new, device="cpu") -> torch.Tensor:
    n = torch.as_tensor(n_new, dtype=torch.int64)
    return torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(n, 0)]).to(torch.int32).to(device)


def block(cfg: CycleConfig, device="cpu", layer=0):
    """(q [B,Hq,bs,d], kb [B,Hkv,bs,d], vb [B,Hkv,bs,d]) of one layer."""
    g = generator(cfg.seed * 1000 + 10 + layer, device)
    q = _randn((cfg.B, cfg.Hq, cfg.bs, cfg.d), 1.0, g, device, cfg.dtype)
    kb = _randn((cfg.B, cfg.Hkv, cfg.bs, cfg.d), 1.0, g, device, cfg.dtype)
    vb = _randn((cfg.B, cfg.Hkv, cfg.bs, cfg.d), 1.0, g, device, cfg.dtype)
    return q, kb, vb


def all_accept_sequences(cfg: CycleConfig):
    n = int(round(cfg.all_accept_frac * cfg.B))
    g = generator(cfg.seed * 1000 + 5, "cpu")
    return sorted(torch.randperm(cfg.B, generator=g)[:n].tolist())


def logits(cfg: CycleConfig, device="cpu"):
    """(target [B, bs, V], draft [B, bs-1, V]) in cfg.dtype."""
    g = generator(cfg.seed * 1000 + 6, device)
    lt = torch.randn((cfg.B, cfg.bs, cfg.V), generator=g, device=device, dtype=torch.float32) * cfg.logit_std
    ld = lt[:, :cfg.bs - 1] + torch.randn((cfg.B, cfg.bs - 1, cfg.V), generator=g, device=device,
                                          dtype=torch.float32) * cfg.draft_noise
    lt = lt.to(cfg.dtype)
    ld = ld.to(cfg.dtype)
    for b in all_accept_sequences(cfg):
        ld[b] = lt[b, :cfg.bs - 1]
    return lt, ld


def draft_tokens(draft_logits: torch.Tensor, temperature: float, seed: int) -> torch.Tensor:
    """Draft tokens [B, bs-1] int32 drawn from softmax(draft/T) (argmax at T=0)."""
    x = draft_logits.float()
    if temperature > 0:
        g = generator(seed, x.device)
        u = torch.rand(x.shape, generator=g, device=x.device, dtype=torch.float64).clamp_(1e-300, 1.0)
        x = x.double() / temperature - torch.log(-torch.log(u))
    return x.argmax(dim=-1).to(torch.int32)
