"""Benchmark of one DFlash draft-and-verify cycle on GB300.

A step is one cycle over the batched workload (B = 32 sequences, cached
context uniform in [1024, 8192], block 8, five draft layers, V = 262144, bf16,
T = 1): context fusion of the cycle's bs new rows per sequence into every
layer's cache, the five layers' block attention, and verification.  Inputs
are seeded synthetic tensors resident in HBM; each step streams ~3.3 GB
(more than the 129 MB L2).

Prints one JSON line.  Arms:
  (default)         the CUDA path (libdflash.so) on N GPUs, one process each,
                    each rank its own batch (weak scaling, no collective on the
                    data path); value = cycles/s of the whole job.
  --impl reference  the CPU oracle timed on the host cores on a bounded sample
                    of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "draft-verify cycles/sec at B=32 (tokens/sec and HBM GB/s as % of peak reported beside it)"
UNIT = "cycles/s"
ATTN_SRC = os.path.join(ROOT, "block_speculative_decoding_gb300", "csrc", "attn.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_main_batched.md")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max_sum(elapsed_s: float, tokens: float, device):
    """Max of the elapsed time and sum of the tokens over ranks (1 rank: identity)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, tokens
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    s = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(s, op=dist.ReduceOp.SUM)
    return float(t.item()), float(s.item())


def rank_config(rank: int, batch: int | None = None, layers: int | None = None) -> workloads.CycleConfig:
    """Each rank runs its own batch: same shapes, seed offset by the rank.
    `batch` / `layers` shrink the case (profiling runs only)."""
    from dataclasses import replace
    c = workloads.BATCHED
    if batch is not None and batch != c.B:
        c = replace(c, B=batch)
    if layers is not None and layers != c.L:
        c = replace(c, L=layers)
    return replace(c, seed=c.seed + 100 * rank) if rank else c


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                       "-i", str(gpu_index), "-lms", "100"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_traffic():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, or None if absent or taken on a different kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    text = open(TRAFFIC_FILE).read()
    m = re.search(r"traffic_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    h = re.search(r"attn\.cu sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(ATTN_SRC, "rb").read()).hexdigest()
    return float(m.group(1)) if h.group(1) == cur else None


# ----------------------------------------------------------------- inputs ---

class Cycle:
    """Device-resident inputs and preallocated outputs/workspaces of one rank."""

    def __init__(self, cfg, device, temperature):
        import block_speculative_decoding_gb300 as dfl
        self.dfl = dfl
        self.cfg, self.dev, self.T = cfg, device, temperature
        self.seq = workloads.seq_lens(cfg, device)
        self.k, self.v = workloads.cache(cfg, device)
        self.w = workloads.weights(cfg, device)
        self.M = cfg.B * cfg.bs
        self.taps = workloads.taps(cfg, self.M, device)
        self.cu = workloads.cu_rows([cfg.bs] * cfg.B, device)
        self.blocks = [workloads.block(cfg, device, layer=l) for l in range(cfg.L)]
        self.lt, self.ld = workloads.logits(cfg, device)
        self.x = workloads.draft_tokens(self.ld, temperature, seed=cfg.seed + 7)
        self.cache = dfl.KVCache(self.k, self.v, self.seq)
        self.outs = [torch.empty_like(b[0]) for b in self.blocks]
        self.acc = torch.empty(cfg.B, dtype=torch.int32, device=device)
        self.tok = torch.empty(cfg.B, cfg.bs, dtype=torch.int32, device=device)
        dt = dfl.BF16
        self.ws_f = torch.empty(dfl.fuse_context_workspace_size(self.M, cfg.J, cfg.d_target, cfg.D, cfg.L, cfg.Hkv, dt),
                                dtype=torch.uint8, device=device)
        self.ws_a = torch.empty(dfl.block_attn_workspace_size(cfg.B, cfg.bs, cfg.Hq, cfg.Hkv, cfg.capacity, 0, dt),
                                dtype=torch.uint8, device=device)
        self.ws_v = torch.empty(dfl.verify_workspace_size(cfg.B, cfg.bs, cfg.V, dt), dtype=torch.uint8, device=device)
        self.cycle = 0
        s = self.seq.cpu().numpy().astype(np.int64)
        self.attn_bytes_per_call = int(s.sum()) * cfg.Hkv * cfg.d * 2 * 2
        self.verify_bytes = cfg.B * (2 * cfg.bs - 1) * cfg.V * 2
        self.fuse_bytes = (self.w.w_fuse.numel() + self.w.w_kv.numel()) * 2 + self.M * cfg.J * cfg.d_target * 2 \
            + self.M * cfg.L * 2 * cfg.Hkv * cfg.d * 2
        self.fuse_flops = 2 * self.M * (cfg.J * cfg.d_target * cfg.D + cfg.D * cfg.L * 2 * cfg.Hkv * cfg.d)

    def inputs(self):
        """The per-step inputs (what a serving loop would receive each cycle)."""
        return {"taps": self.taps, "blocks": self.blocks, "lt": self.lt, "ld": self.ld, "x": self.x}

    def step(self, stream, ev=None, only="all", inputs=None):
        dfl, c = self.dfl, self.cfg
        inp = inputs if inputs is not None else self.inputs()
        if ev is not None:
            ev[0].record(stream)
        if only in ("all", "fuse"):
            dfl.fuse_context(inp["taps"], self.cu, self.w.w_fuse, self.w.g_fuse, self.w.w_kv, self.w.k_gain,
                             self.cache, workspace=self.ws_f, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if only in ("all", "attn"):
            for l in range(c.L):
                q, kb, vb = inp["blocks"][l]
                dfl.block_attn(l, q, kb, vb, self.w.q_gain[l], self.w.k_gain[l], self.cache, out=self.outs[l],
                               workspace=self.ws_a, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        if only in ("all", "verify"):
            dfl.verify(inp["lt"], inp["ld"], inp["x"], self.T, 1234, self.cycle, accepted_len=self.acc,
                       out_tokens=self.tok, workspace=self.ws_v, stream=stream)
        if ev is not None:
            ev[3].record(stream)
        self.cycle += 1


def launches_per_step(M: int, layers: int) -> int:
    """The library's kernel launches in one step: fusion 4 for up to 256 new rows (fusion GEMM, row
    norm, K/V GEMM, K/V epilogue) else 3 (the K/V epilogue fused into the GEMM), block attention 3 per
    layer (counter clear, main, combine), verification 2 (stats, finish)."""
    return (4 if M <= 256 else 3) + 3 * layers + 2


def run_gpu(args):
    rank, world, local = env_rank()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from __graft_entry__ import build
    if rank == 0:
        build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    build()
    cfg = rank_config(rank, args.batch, args.layers)
    cyc = Cycle(cfg, dev, args.temperature)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            cyc.step(stream, only=args.only)
    torch.cuda.synchronize()
    # tokens per cycle from this rank's verification outputs
    tokens_per_cycle = float((cyc.acc.cpu() + 1).sum())

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def timed_region():
        """Exactly `steps` cycles bracketed by a barrier and a device
        synchronisation on both sides; seconds on the stream's clock."""
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        # the timed steps run back to back, nothing between the calls (an event
        # between two kernels would stop the second from launching early)
        t0.record(stream)
        for i in range(args.steps):
            cyc.step(stream, only=args.only)
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        return t0.elapsed_time(t1) / 1e3

    clocks = ClockSampler(local)
    time.sleep(0.3)
    # the timed region runs `repeats` times back to back (enough for about two
    # seconds of load unless given), so that the clock sampler sees the GPU
    # under load; the median region is reported
    regions = [timed_region()]
    repeats = args.repeats if args.repeats > 0 else int(min(500, max(5, np.ceil(2.0 / max(regions[0], 1e-4)))))
    if world > 1:      # every rank runs the same number of regions (each one ends in a barrier)
        import torch.distributed as dist
        r = torch.tensor([repeats], dtype=torch.int64, device=dev)
        dist.all_reduce(r, op=dist.ReduceOp.MAX)
        repeats = int(r.item())
    for _ in range(repeats - 1):
        regions.append(timed_region())
    clk = clocks.stop()
    elapsed = float(np.median(regions))
    # per-call times (rooflines): a second pass of the same steps with events between the calls
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            cyc.step(stream, evs[i], only=args.only)
    torch.cuda.synchronize()
    fuse_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / cfg.L
    ver_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    # verification calls back to back (one event pair around them, none between
    # calls, so each call's first kernel launches early as in the timed steps)
    ver_b2b_ms = None
    if args.only in ("all", "verify"):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                cyc.step(stream, only="verify")
            e1.record(stream)
        torch.cuda.synchronize()
        ver_b2b_ms = e0.elapsed_time(e1) / args.steps
    elapsed_max, tokens_all = reduce_max_sum(elapsed, tokens_per_cycle * args.steps, dev)

    if args.only != "all" or args.batch is not None or args.layers is not None:
        if rank == 0:
            print(json.dumps({"profiling_run": True, "only": args.only, "B": cfg.B, "steps": args.steps,
                              "ms_per_step": elapsed * 1e3 / args.steps, "fuse_ms": fuse_ms,
                              "attn_ms_per_layer": attn_ms, "verify_ms": ver_ms, "verify_b2b_ms": ver_b2b_ms}),
                  flush=True)
        return
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(cyc, stream, args, dev)
    tensor_lines = None
    if rank == 0 and not args.no_e2e:
        tensor_lines = fusion_tensor_rooflines(dev, peaks()[1])
        tensor_lines.update(window_attention_roofline(cyc, dev, peaks()[0]))
        tensor_lines.update(paged_attention_roofline(cyc, dev, peaks()[0]))
        tensor_lines.update(draft_head_roofline(cyc, dev, peaks()[0]))
        tensor_lines.update(dflash2_roofline(cyc, dev, peaks()[0]))
        tensor_lines.update(layer_tail_roofline(cyc, dev, peaks()[0], peaks()[1]))
        tensor_lines.update(full_drafter_cycle(cyc, dev, peaks()[0]))

    if rank != 0:
        return
    hbm, tfl, src = peaks()
    cycles = world * args.steps
    attn_gbs = cyc.attn_bytes_per_call / (attn_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": cycles / elapsed_max, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max * 1e3 / args.steps, "higher_is_better": True,
        "repeats": {"count": repeats, "reported": "median",
                    "ms_per_step_min": min(regions) * 1e3 / args.steps,
                    "ms_per_step_max": max(regions) * 1e3 / args.steps},
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "batched: B=32, cached context uniform in [1024, 8192] (ragged), 5 draft layers, "
                               "GQA 32/8, head 128, D=2560, block 8, V=262144, T=%g; per step: fusion of 8 new rows "
                               "per sequence, 5 x block attention, verification" % args.temperature,
                   "B": cfg.B, "block_size": cfg.bs, "vocab": cfg.V, "layers": cfg.L,
                   "mean_context": float(cyc.seq.float().mean()), "parallelism": "dp%d (independent batches)" % world,
                   "l2": "inputs larger than L2: %.2f GB streamed per step" % (
                       (cfg.L * cyc.attn_bytes_per_call + cyc.verify_bytes + cyc.fuse_bytes) / 1e9)},
        "tokens_per_sec": tokens_all / elapsed_max,
        "mean_tokens_per_cycle": tokens_per_cycle / cfg.B,
        "roofline": {"kernel": "block attention (counter clear + split-KV main with in-kernel Q/K norm and RoPE + combine), per layer call",
                     "bound": "hbm", "achieved": attn_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": attn_gbs / hbm, "peak_source": src,
                     "algorithmic_bytes_per_launch": cyc.attn_bytes_per_call,
                     "traffic": measured_traffic()},
        "components_ms": {"fuse_context": fuse_ms, "block_attn_per_layer": attn_ms, "verify": ver_ms,
                          "timing": "a second pass of the same steps with CUDA events between the calls (the "
                                    "events stop each call's first kernel from launching early, so these are "
                                    "slightly longer than the calls take in the timed steps)"},
        "rooflines": {
            "attention_plus_verify": {
                "bound": "hbm", "peak": hbm, "unit": "GB/s",
                "achieved": (cfg.L * cyc.attn_bytes_per_call + cyc.verify_bytes) / ((cfg.L * attn_ms + ver_ms) * 1e-3) / 1e9,
                "frac": (cfg.L * cyc.attn_bytes_per_call + cyc.verify_bytes) / ((cfg.L * attn_ms + ver_ms) * 1e-3) / 1e9
                        / hbm,
                "note": "the cycle's five block-attention calls and its verification together: their algorithmic "
                        "bytes over their summed component times"},
            "verify": {"bound": "hbm", "achieved": cyc.verify_bytes / (ver_ms * 1e-3) / 1e9, "peak": hbm,
                       "unit": "GB/s", "frac": cyc.verify_bytes / (ver_ms * 1e-3) / 1e9 / hbm},
            "verify_back_to_back": {
                "bound": "hbm", "achieved": cyc.verify_bytes / (ver_b2b_ms * 1e-3) / 1e9, "peak": hbm,
                "unit": "GB/s", "frac": cyc.verify_bytes / (ver_b2b_ms * 1e-3) / 1e9 / hbm, "ms_per_call": ver_b2b_ms,
                "note": "the same verification call repeated %d times after the timed steps, one event pair around "
                        "them: no event between calls, so each call's stats pass launches early as in the cycle; "
                        "the 251.7 MB of logits exceed L2 and are read from DRAM every call" % args.steps},
            "fuse_context": {"bound": "hbm (M=%d: weight-bound)" % cyc.M,
                             "achieved": cyc.fuse_bytes / (fuse_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": cyc.fuse_bytes / (fuse_ms * 1e-3) / 1e9 / hbm,
                             "tflops": cyc.fuse_flops / (fuse_ms * 1e-3) / 1e12}},
        "peak_note": "HBM and bf16 peaks are the measured copy bandwidth and cuBLAS bf16 GEMM (burst) of this GPU",
        "gpu_launches": launches_per_step(cyc.M, cfg.L) * args.steps,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if tensor_lines is not None:
        line["rooflines"].update(tensor_lines)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds, args.temperature)
    print(json.dumps(line), flush=True)


def window_attention_roofline(cyc, dev, peak_gbs, W=1024, iters=20):
    """Block attention of the batched workload over the drafter's sliding
    window kept as a ring cache of W rows (every sequence is longer than W, so
    each attends to exactly W cached keys): five layer calls back to back,
    CUDA events on the launching stream, 3 warm-up rounds; algorithmic bytes
    B * W * 4096 per layer call."""
    import block_speculative_decoding_gb300 as dfl
    from dataclasses import replace
    cfg = replace(cyc.cfg, S=W, S_min=None)
    k, v = workloads.cache(replace(cfg, bs=0, fuse_rows_per_seq=0), dev)
    ring = dfl.KVCache(k[..., :W, :].contiguous(), v[..., :W, :].contiguous(), cyc.seq.clone(), ring=True)
    del k, v
    ws = torch.empty(dfl.block_attn_workspace_size(cfg.B, cfg.bs, cfg.Hq, cfg.Hkv, W, 0, dfl.BF16),
                     dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)

    def layers():
        for l in range(cfg.L):
            q, kb, vb = cyc.blocks[l]
            dfl.block_attn(l, q, kb, vb, cyc.w.q_gain[l], cyc.w.k_gain[l], ring, out=cyc.outs[l], workspace=ws,
                           stream=st)
    with torch.cuda.stream(st):
        for _ in range(3):
            layers()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(iters):
            layers()
        e1.record(st)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (iters * cfg.L)
    gbs = cfg.B * W * cfg.Hkv * cfg.d * 2 * 2 / (ms * 1e-3) / 1e9
    del ring, ws
    torch.cuda.empty_cache()
    return {"block_attn_ring_window_%d" % W: {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s",
                                             "frac": gbs / peak_gbs, "ms_per_layer_call": ms,
                                             "note": "ring cache of %d rows per (layer, sequence, KV head); every "
                                                     "sequence longer than the window" % W}}


def paged_attention_roofline(cyc, dev, peak_gbs, P=128, iters=20):
    """Block attention of the batched workload over the same cache contents in
    a paged pool: 128-row pages, a random permutation of the pool as the block
    table; five layer calls back to back, CUDA events on the launching stream,
    3 warm-up rounds; algorithmic bytes as for the linear cache (every cached
    key and value read once)."""
    import block_speculative_decoding_gb300 as dfl
    cfg = cyc.cfg
    L, B, H, cap, d = cyc.k.shape
    MP = -(-cap // P)
    g = torch.Generator().manual_seed(cfg.seed * 1000 + 25)
    perm = torch.randperm(B * MP, generator=g).to(dev)

    def pool_of(lin):
        x = torch.nn.functional.pad(lin, (0, 0, 0, MP * P - cap))
        x = x.view(L, B, H, MP, P, d).permute(0, 1, 3, 2, 4, 5).reshape(L, B * MP, H, P, d)
        out = torch.empty_like(x)
        out[:, perm] = x
        return out
    pages = dfl.KVCache(pool_of(cyc.k), pool_of(cyc.v), cyc.seq.clone(),
                        block_table=perm.view(B, MP).to(torch.int32).contiguous())
    ws = torch.empty(dfl.block_attn_workspace_size(B, cfg.bs, cfg.Hq, H, MP * P, 0, dfl.BF16),
                     dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)

    def layers():
        for l in range(cfg.L):
            q, kb, vb = cyc.blocks[l]
            dfl.block_attn(l, q, kb, vb, cyc.w.q_gain[l], cyc.w.k_gain[l], pages, out=cyc.outs[l], workspace=ws,
                           stream=st)
    with torch.cuda.stream(st):
        for _ in range(3):
            layers()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(iters):
            layers()
        e1.record(st)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (iters * cfg.L)
    gbs = cyc.attn_bytes_per_call / (ms * 1e-3) / 1e9
    del pages, ws
    torch.cuda.empty_cache()
    return {"block_attn_paged_%d" % P: {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s",
                                        "frac": gbs / peak_gbs, "ms_per_layer_call": ms,
                                        "note": "the batched cache in %d-row pages of a shared pool, block table = "
                                                "a random permutation of the pool" % P}}


def dflash2_roofline(cyc, dev, peak_gbs, m=8, lam=0.2, iters=20):
    """The DFlash2 candidate pass on the batched workload's draft logits: B x
    (bs - 1) rows of V = 262144 bf16, top-8 candidates, entropies and the
    best-path score per sequence.  Algorithmic bytes: every logit read once,
    B (bs - 1) V 2.  Beside it, the depthwise block convolution (k = 5) of the
    B x bs block rows of width D.  CUDA events on the launching stream, 3
    warm-up calls."""
    import block_speculative_decoding_gb300 as dfl
    cfg = cyc.cfg
    R = cfg.bs - 1
    g = workloads.generator(cfg.seed * 1000 + 27, dev)
    logits = (cfg.logit_std * torch.randn(cfg.B, R, cfg.V, generator=g, device=dev)).to(torch.bfloat16)
    ws = torch.empty(dfl.draft_topm_workspace_size(cfg.B, R, cfg.V, m), dtype=torch.uint8, device=dev)
    h = torch.randn(cfg.B * cfg.bs, cfg.D, generator=g, device=dev).to(torch.bfloat16)
    wc = (0.3 * torch.randn(5, cfg.D, generator=g, device=dev)).to(torch.bfloat16)
    st = torch.cuda.Stream(device=dev)

    def timed(fn):
        with torch.cuda.stream(st):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(iters):
                fn()
            e1.record(st)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters
    ms = timed(lambda: dfl.draft_topm(logits, m, cyc.T if cyc.T > 0 else 1.0, lam, workspace=ws, stream=st))
    conv_ms = timed(lambda: dfl.block_conv(h, wc, None, cfg.bs, residual=True, out=h, stream=st))
    nbytes = cfg.B * R * cfg.V * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    del logits, ws, h
    torch.cuda.empty_cache()
    return {"dflash2_topm": {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
                             "ms_per_call": ms, "rows": cfg.B * R, "vocab": cfg.V, "m": m,
                             "block_conv_k5_ms_per_call": conv_ms}}


def draft_head_roofline(cyc, dev, peak_gbs, iters=10):
    """The drafter's head on the batched workload's proposal rows: B x (bs - 1)
    rows, D = 2560, V = 262144 (final RMSNorm, LM head, draft race at T).
    Algorithmic bytes: the head's weights V * D * 2 read once, the logits
    M * V * 2 written, the rows M * D * 2 read; CUDA events on the launching
    stream, 3 warm-up calls."""
    import block_speculative_decoding_gb300 as dfl
    cfg = cyc.cfg
    R = cfg.bs - 1
    M = cfg.B * R
    g = workloads.generator(cfg.seed * 1000 + 21, dev)
    x = (torch.randn(M, cfg.D, generator=g, device=dev) * 2.0).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(cfg.D, generator=g, device=dev)).to(torch.bfloat16)
    w = (torch.randn(cfg.V, cfg.D, generator=g, device=dev) * 0.05).to(torch.bfloat16)
    logits = torch.empty(M, cfg.V, dtype=torch.bfloat16, device=dev)
    tok = torch.empty(M, dtype=torch.int32, device=dev)
    ws = torch.empty(dfl.draft_head_workspace_size(cfg.B, R, cfg.D, cfg.V), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    call = lambda c: dfl.draft_head(x, gain, w, R, cyc.T, 1234, c, logits=logits, tokens=tok,  # noqa: E731
                                    workspace=ws, stream=st)
    with torch.cuda.stream(st):
        for c in range(3):
            call(c)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for c in range(iters):
            call(c)
        e1.record(st)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    nbytes = cfg.V * cfg.D * 2 + M * cfg.V * 2 + M * cfg.D * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    del x, w, logits, ws
    torch.cuda.empty_cache()
    return {"draft_head": {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
                           "ms_per_call": ms, "rows": M, "vocab": cfg.V, "temperature": cyc.T,
                           "tflops": 2.0 * M * cfg.V * cfg.D / (ms * 1e-3) / 1e12}}


def full_drafter_cycle(cyc, dev, peak_gbs, iters=20):
    """One whole draft-and-verify cycle with the drafter's own forward on the
    batched workload, beside the headline cycle: context fusion of 8 new rows
    per sequence; five layers of input norm + q/k/v projections, block
    attention over the cache and the layer remainder (D = 2560, 32/8 heads,
    MLP 5120); the head (final norm, LM head over V = 262144, draft race) on
    the 7 mask rows of each sequence; verification of the head's own draft
    tokens and logits against the target logits.  Synthetic weights; the
    block's input rows are copied in fresh each cycle.  Algorithmic bytes:
    every weight read once, the cache rows attended, the logits written by
    the head and read by verification, the target logits read.  Steps run back
    to back; CUDA events around them; 3 warm-up cycles."""
    import block_speculative_decoding_gb300 as dfl
    cfg = cyc.cfg
    M, D, I, Hq, Hkv, V, R = cfg.B * cfg.bs, cfg.D, cfg.mlp_dim, cfg.Hq, cfg.Hkv, cfg.V, cfg.bs - 1
    g = workloads.generator(cfg.seed * 1000 + 31, dev)
    r = lambda *s, std=0.02: (torch.randn(*s, generator=g, device=dev) * std).to(torch.bfloat16)  # noqa: E731
    gain = lambda *s: (1 + 0.1 * torch.randn(*s, generator=g, device=dev)).to(torch.bfloat16)  # noqa: E731
    g_in, w_qkv = gain(cfg.L, D), r(cfg.L, (Hq + 2 * Hkv) * 128, D)
    w_o, g_post, w_gu, w_dn = r(cfg.L, D, Hq * 128), gain(cfg.L, D), r(cfg.L, 2 * I, D), r(cfg.L, D, I)
    g_final, w_head = gain(D), r(V, D, std=0.05)
    x0 = r(M, D, std=1.0)
    x = torch.empty_like(x0)
    mask_rows = torch.tensor([b * cfg.bs + j for b in range(cfg.B) for j in range(1, cfg.bs)], device=dev)
    xh = torch.empty(cfg.B * R, D, dtype=torch.bfloat16, device=dev)
    q, kb, vb = (torch.empty(cfg.B, h, cfg.bs, 128, dtype=torch.bfloat16, device=dev) for h in (Hq, Hkv, Hkv))
    o = torch.empty_like(q)
    logits = torch.empty(cfg.B * R, V, dtype=torch.bfloat16, device=dev)
    tok = torch.empty(cfg.B * R, dtype=torch.int32, device=dev)
    ws = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)  # noqa: E731
    ws_q = ws(dfl.draft_layer_qkv_workspace_size(cfg.B, cfg.bs, Hq, Hkv, D))
    ws_t = ws(dfl.draft_layer_tail_workspace_size(cfg.B, cfg.bs, Hq, D, I))
    ws_h = ws(dfl.draft_head_workspace_size(cfg.B, R, D, V))
    st = torch.cuda.Stream(device=dev)

    def step(c):
        dfl.fuse_context(cyc.taps, cyc.cu, cyc.w.w_fuse, cyc.w.g_fuse, cyc.w.w_kv, cyc.w.k_gain, cyc.cache,
                         workspace=cyc.ws_f, stream=st)
        x.copy_(x0)                                   # the block's input rows of this cycle
        for l in range(cfg.L):
            dfl.draft_layer_qkv(x, g_in[l], w_qkv[l], cfg.B, Hq, Hkv, q=q, kb=kb, vb=vb, workspace=ws_q, stream=st)
            dfl.block_attn(l, q, kb, vb, cyc.w.q_gain[l], cyc.w.k_gain[l], cyc.cache, out=o, workspace=cyc.ws_a,
                           stream=st)
            dfl.draft_layer_tail(x, o, w_o[l], g_post[l], w_gu[l], w_dn[l], workspace=ws_t, stream=st)
        torch.index_select(x, 0, mask_rows, out=xh)   # the 7 mask rows of each sequence
        dfl.draft_head(xh, g_final, w_head, R, cyc.T, 1234, c, logits=logits, tokens=tok, workspace=ws_h, stream=st)
        dfl.verify(cyc.lt, logits.view(cfg.B, R, V), tok.view(cfg.B, R), cyc.T, 1234, c, accepted_len=cyc.acc,
                   out_tokens=cyc.tok, workspace=cyc.ws_v, stream=st)

    with torch.cuda.stream(st):
        for c in range(3):
            step(c)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for c in range(iters):
            step(c)
        e1.record(st)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    tokens = float((cyc.acc.cpu() + 1).sum())
    weights = (cyc.w.w_fuse.numel() + cyc.w.w_kv.numel() + w_qkv.numel() + w_o.numel() + w_gu.numel() +
               w_dn.numel() + w_head.numel()) * 2
    nbytes = weights + cfg.L * cyc.attn_bytes_per_call + 2 * cfg.B * R * V * 2 + cfg.B * cfg.bs * V * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    launches = (4 + 3 * cfg.L + 2) + cfg.L * 3 + cfg.L * 6 + 3
    del w_qkv, w_o, w_gu, w_dn, w_head, logits, ws_q, ws_t, ws_h
    torch.cuda.empty_cache()
    return {"full_drafter_cycle": {
        "bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
        "ms_per_cycle": ms, "cycles_per_sec": 1e3 / ms, "tokens_per_sec": tokens * 1e3 / ms,
        "algorithmic_bytes": nbytes, "gpu_launches_per_cycle": launches,
        "note": "fusion + 5 x (q/k/v + block attention + layer remainder) + head (7 mask rows per sequence, "
                "V=262144) + verification of the head's own draft; synthetic weights, so the acceptance (and "
                "tokens_per_sec) is that of a random drafter against synthetic target logits; the mask rows are "
                "gathered with torch.index_select (1.1 MB) and the block's input rows copied in with torch each "
                "cycle"}}


def layer_tail_roofline(cyc, dev, peak_gbs, peak_tflops, iters=20):
    """The rest of one draft layer on the batched workload's block rows: M = B x bs
    rows, 32 heads of 128, D = 2560, MLP width I = 5120 (output projection +
    residual, post-attention RMSNorm, SwiGLU MLP + residual).  Algorithmic bytes:
    the weights (D Hq 128 + 3 I D) x 2 read once, the attention output M Hq 128 x 2
    read, the residual rows M D x 2 read and written; flops 2 M (Hq 128 D + 3 I D).
    CUDA events on the launching stream, 3 warm-up calls."""
    import block_speculative_decoding_gb300 as dfl
    cfg = cyc.cfg
    M, D, I, Kq = cfg.B * cfg.bs, cfg.D, cfg.mlp_dim, cfg.Hq * cfg.d
    g = workloads.generator(cfg.seed * 1000 + 23, dev)
    r = lambda *s, std=1.0: (torch.randn(*s, generator=g, device=dev) * std).to(torch.bfloat16)  # noqa: E731
    x, o = r(M, D, std=2.0), r(cfg.B, cfg.Hq, cfg.bs, cfg.d)
    w_o, w_gu, w_dn = r(D, Kq, std=0.02), r(2 * I, D, std=0.05), r(D, I, std=0.02)
    g_post = (1 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    ws = torch.empty(dfl.draft_layer_tail_workspace_size(cfg.B, cfg.bs, cfg.Hq, D, I), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    call = lambda: dfl.draft_layer_tail(x, o, w_o, g_post, w_gu, w_dn, workspace=ws, stream=st)  # noqa: E731
    with torch.cuda.stream(st):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(iters):
            call()
        e1.record(st)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    nbytes = (D * Kq + 3 * I * D) * 2 + M * Kq * 2 + 2 * M * D * 2
    flops = 2.0 * M * (Kq * D + 3 * I * D)
    gbs = nbytes / (ms * 1e-3) / 1e9
    tf = flops / (ms * 1e-3) / 1e12
    del x, o, w_o, w_gu, w_dn, ws
    torch.cuda.empty_cache()
    return {"draft_layer_tail": {"bound": "hbm", "achieved": gbs, "peak": peak_gbs, "unit": "GB/s",
                                 "frac": gbs / peak_gbs, "ms_per_call": ms, "rows": M, "mlp_dim": I,
                                 "tflops": tf, "tensor_frac": tf / peak_tflops}}


def fusion_tensor_rooflines(dev, peak_tflops, iters=10):
    """The fusion call on its tensor-bound shapes (the GEMMs' roofline): a 4 x 2048-row prefill chunk of the
    long-context workload and the 128 x 16-row cycle of the high-batch bs = 16 workload.  Flops
    2 M (J d_t D + D L 2 Hkv d) per call, CUDA events on the launching stream, 3 warm-up calls."""
    import block_speculative_decoding_gb300 as dfl
    from dataclasses import replace
    out = {}
    for name, B, rows, cap in (("fusion_prefill_4x2048", 4, 2048, 4096), ("fusion_cycle_128x16", 128, 16, 2064)):
        cfg = replace(workloads.LONG_CONTEXT, B=B, S=cap - rows)
        w = workloads.weights(cfg, dev)
        M = B * rows
        taps = workloads.taps(cfg, M, dev)
        cu = workloads.cu_rows([rows] * B, dev)
        k = torch.empty(cfg.L, B, cfg.Hkv, cap, cfg.d, dtype=torch.bfloat16, device=dev)
        cache = dfl.KVCache(k, torch.empty_like(k), torch.zeros(B, dtype=torch.int32, device=dev))
        ws = torch.empty(dfl.fuse_context_workspace_size(M, cfg.J, cfg.d_target, cfg.D, cfg.L, cfg.Hkv, dfl.BF16),
                         dtype=torch.uint8, device=dev)
        st = torch.cuda.Stream(device=dev)
        call = lambda: dfl.fuse_context(taps, cu, w.w_fuse, w.g_fuse, w.w_kv, w.k_gain, cache,  # noqa: E731
                                        workspace=ws, stream=st)
        with torch.cuda.stream(st):
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(iters):
                call()
            e1.record(st)
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        flops = 2 * M * (cfg.J * cfg.d_target * cfg.D + cfg.D * cfg.L * 2 * cfg.Hkv * cfg.d)
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"bound": "tensor", "achieved": tf, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": tf / peak_tflops, "M": M, "ms_per_call": ms}
        del taps, k, cache, ws
    torch.cuda.empty_cache()
    return out


def run_e2e(cyc, stream, args, dev):
    """Same cycle through the public API with the step's inputs in pinned host
    memory: every step copies its new context rows, block projections, logits
    and draft tokens to the device, runs the calls and reads the accepted
    lengths and tokens back.  As a serving loop would, the copies of step i+1
    run on a second stream into a second set of device buffers while step i
    computes (double buffering)."""
    host = {
        "taps": [t.cpu().pin_memory() for t in cyc.taps],
        "blocks": [[t.cpu().pin_memory() for t in b] for b in cyc.blocks],
        "lt": cyc.lt.cpu().pin_memory(), "ld": cyc.ld.cpu().pin_memory(), "x": cyc.x.cpu().pin_memory(),
    }
    res_h = [(torch.empty(cyc.cfg.B, dtype=torch.int32).pin_memory(),
              torch.empty(cyc.cfg.B, cyc.cfg.bs, dtype=torch.int32).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host["taps"]) + \
        sum(t.numel() * t.element_size() for b in host["blocks"] for t in b) + \
        sum(host[k].numel() * host[k].element_size() for k in ("lt", "ld", "x"))
    d2h = res_h[0][0].numel() * 4 + res_h[0][1].numel() * 4
    base = cyc.inputs()
    sets = [base, {"taps": [t.clone() for t in base["taps"]], "blocks": [[t.clone() for t in b] for b in base["blocks"]],
                   "lt": base["lt"].clone(), "ld": base["ld"].clone(), "x": base["x"].clone()}]
    copy_stream = torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    released = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        k = i % 2
        d = sets[k]
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(released[k])   # step i-2 is done with this set
            for dt, ht in zip(d["taps"], host["taps"]):
                dt.copy_(ht, non_blocking=True)
            for db, hb in zip(d["blocks"], host["blocks"]):
                for dt, ht in zip(db, hb):
                    dt.copy_(ht, non_blocking=True)
            for key in ("lt", "ld", "x"):
                d[key].copy_(host[key], non_blocking=True)
            uploaded[k].record(copy_stream)

    def compute(i):
        k = i % 2
        with torch.cuda.stream(stream):
            stream.wait_event(uploaded[k])
            cyc.step(stream, inputs=sets[k])
            released[k].record(stream)
            res_h[k][0].copy_(cyc.acc, non_blocking=True)
            res_h[k][1].copy_(cyc.tok, non_blocking=True)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)

    run(max(1, args.warmup))
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 50))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(copy_stream)
    stream.wait_event(t0)
    run(n)
    t1.record(stream)
    torch.cuda.synchronize()
    el = t0.elapsed_time(t1) / 1e3
    el, _ = reduce_max_sum(el, 0.0, dev)
    _, world, _ = env_rank()
    return {"value": world * n / el, "unit": UNIT, "steps": n, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "pipelining": "double-buffered: the host-to-device copies of step i+1 run on a second stream while "
                          "step i computes; every step's copies and result read are inside the timed region"}


# ------------------------------------------------------------ CPU oracle ----

def oracle_verify_batch(cfg, T):
    """(target logits [B, bs, V], draft logits [B, bs-1, V], both float32
    holding bf16 values; draft tokens [B, bs-1]) from the seeded generators."""
    lt, ld = workloads.logits(cfg, "cpu")
    x = workloads.draft_tokens(ld, T, seed=cfg.seed + 7)
    return lt.float().numpy(), ld.float().numpy(), x.numpy()


def oracle_verify_rows(cfg, T, seqs, batch=None):
    """Per sequence b: (target logits [1, bs, V], draft logits [1, bs-1, V],
    draft tokens [1, bs-1]), sliced from the batch's (drawn if not given)."""
    lt, ld, x = batch if batch is not None else oracle_verify_batch(cfg, T)
    return {b: (lt[b:b + 1], ld[b:b + 1], x[b:b + 1]) for b in seqs}


def oracle_weights(cfg):
    """The seeded weights as float64 arrays."""
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    w = workloads.weights(cfg, "cpu")
    return {"w_fuse": f(w.w_fuse), "g_fuse": f(w.g_fuse), "w_kv": f(w.w_kv), "k_gain": f(w.k_gain),
            "q_gain": f(w.q_gain)}


def oracle_cache(cfg):
    """(k, v) [L, 1, Hkv, max seq_len, d] float32 holding bf16 N(0, 1) values."""
    g = workloads.generator(cfg.seed * 1000 + 3, "cpu")
    n = int(workloads.seq_lens(cfg).max())
    shape = (cfg.L, 1, cfg.Hkv, n, cfg.d)
    return (torch.randn(shape, generator=g).to(torch.bfloat16).float().numpy(),
            torch.randn(shape, generator=g).to(torch.bfloat16).float().numpy())


class OracleSample:
    """Host (float64) copies of the workload for a few sampled sequences.

    Weights, taps and block projections are the same seeded tensors the GPU
    arm uses; logits and draft tokens come from the seeded batch generators
    (`oracle_verify_rows`).  The cached K/V (synthetic N(0, 1) in bf16 values,
    as float32) is one array of the longest sequence's length per layer and
    head (`oracle_cache`); sequence b reads its first seq_len[b] rows."""

    def __init__(self, cfg, T, seqs, verify_rows=None, kv=None, weights=None):
        f = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
        self.cfg, self.T, self.seqs = cfg, T, list(seqs)
        self.w = weights if weights is not None else oracle_weights(cfg)
        self.seq = workloads.seq_lens(cfg).numpy().astype(np.int64)
        taps = workloads.taps(cfg, cfg.B * cfg.bs, "cpu")
        self.taps = {b: [f(t[b * cfg.bs:(b + 1) * cfg.bs]) for t in taps] for b in self.seqs}
        blocks = [workloads.block(cfg, "cpu", layer=l) for l in range(cfg.L)]
        self.blocks = {b: [[f(t[b:b + 1]) for t in blocks[l]] for l in range(cfg.L)] for b in self.seqs}
        rows = verify_rows if verify_rows is not None else oracle_verify_rows(cfg, T, self.seqs)
        self.lt = {b: rows[b][0].astype(np.float64) for b in self.seqs}
        self.ld = {b: rows[b][1].astype(np.float64) for b in self.seqs}
        self.x = {b: rows[b][2] for b in self.seqs}
        self._kv = kv if kv is not None else oracle_cache(cfg)

    def kv(self, b):
        k, v = self._kv
        n = int(self.seq[b])
        return k[:, :, :, :n], v[:, :, :, :n]

    # the three parts of one sequence's cycle, as the oracle computes them
    def fuse(self, b):
        import oracle
        c = self.cfg
        pos = self.seq[b] + np.arange(c.bs)
        oracle.fuse_rows(self.taps[b], self.w["w_fuse"], self.w["g_fuse"], self.w["w_kv"], self.w["k_gain"], pos,
                         c.L, c.Hkv, c.d, bf16=True)

    def attn(self, b, l, g=None):
        """Layer l of sequence b; g = one KV head (with its query group) or all heads."""
        import oracle
        c = self.cfg
        k, v = self.kv(b)
        q, kb, vb = self.blocks[b][l]
        ck, cv = k[l], v[l]
        if g is not None:
            G = c.Hq // c.Hkv
            q, kb, vb = q[:, g * G:(g + 1) * G], kb[:, g:g + 1], vb[:, g:g + 1]
            ck, cv = ck[:, g:g + 1], cv[:, g:g + 1]
        oracle.block_attn(q, kb, vb, self.w["q_gain"][l], self.w["k_gain"][l], ck, cv, self.seq[b:b + 1],
                          bf16=True)

    def verify(self, b):
        import oracle
        oracle.verify(self.lt[b], self.ld[b], self.x[b], self.T, 1234, 0, seq_ids=np.asarray([b]))

    def cycle(self, b):
        self.fuse(b)
        for l in range(self.cfg.L):
            self.attn(b, l)
        self.verify(b)


def _oracle_worker(conn, T, seqs, paths):
    """A host worker for the oracle timings: single-threaded (its BLAS thread
    count is fixed to 1 by the environment it was spawned with), holding the
    inputs of its own sequences.  Commands: ("cycle",) runs one cycle of each
    of its sequences and answers the seconds taken; ("budget", s) runs cycles
    over its sequences until s seconds have passed and answers (count, seconds,
    summed context); ("stop",) ends it."""
    torch.set_num_threads(1)
    rows = oracle_verify_rows(workloads.BATCHED, T, seqs,
                              batch=tuple(np.load(paths[n], mmap_mode="r") for n in ("lt", "ld", "x")))
    kv = tuple(np.load(paths[n], mmap_mode="r") for n in ("k", "v"))
    weights = {n: np.load(paths[n], mmap_mode="r") for n in ("w_fuse", "g_fuse", "w_kv", "k_gain", "q_gain")}
    sample = OracleSample(workloads.BATCHED, T, seqs, verify_rows=rows, kv=kv, weights=weights)
    conn.send("ready")
    while True:
        cmd = conn.recv()
        if cmd[0] == "cycle":
            t0 = time.perf_counter()
            for b in sample.seqs:
                sample.cycle(b)
            conn.send(time.perf_counter() - t0)
        elif cmd[0] == "budget":
            t0 = time.perf_counter()
            done, ctx = 0, 0
            while done == 0 or time.perf_counter() - t0 < cmd[1]:
                b = sample.seqs[done % len(sample.seqs)]
                sample.cycle(b)
                ctx += int(sample.seq[b])
                done += 1
            conn.send((done, time.perf_counter() - t0, ctx))
        else:
            conn.close()
            return


class OraclePool:
    """Spawned host processes that split the batch's sequences between them
    (sequence-parallel: the sequences of a cycle are independent), one thread
    each.  Spawned, not forked, so it is safe after CUDA has been used."""

    def __init__(self, T, n_workers, seqs_of, inputs):
        import multiprocessing as mp
        paths = inputs.paths
        ctx = mp.get_context("spawn")
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in keep:
            os.environ[k] = "1"          # inherited by the spawned workers before they import numpy
        try:
            self.conns, self.procs = [], []
            for i in range(n_workers):
                a, b = ctx.Pipe()
                mine = seqs_of(i)
                pr = ctx.Process(target=_oracle_worker, args=(b, T, mine, paths), daemon=True)
                pr.start()
                self.conns.append(a)
                self.procs.append(pr)
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for c in self.conns:
            assert c.recv() == "ready"

    def ask(self, cmd):
        for c in self.conns:
            c.send(cmd)
        return [c.recv() for c in self.conns]

    def close(self):
        for c in self.conns:
            c.send(("stop",))
        for pr in self.procs:
            pr.join(timeout=30)


class OracleInputs:
    """The oracle workers' shared inputs -- the verification logits and draft
    tokens, the weights and the synthetic cache -- drawn once and saved to
    files that every worker maps (one copy in the page cache instead of one
    per process, and nothing large to send to a starting process)."""

    def __init__(self, cfg, T):
        self.dir = tempfile.mkdtemp(prefix="dflash_oracle_")
        arrays = dict(oracle_weights(cfg))
        arrays["k"], arrays["v"] = oracle_cache(cfg)
        arrays["lt"], arrays["ld"], arrays["x"] = oracle_verify_batch(cfg, T)
        self.paths = {}
        for n, a in arrays.items():
            self.paths[n] = os.path.join(self.dir, n + ".npy")
            np.save(self.paths[n], a)

    def close(self):
        for pth in self.paths.values():
            os.unlink(pth)
        os.rmdir(self.dir)


def host_cores():
    return max(1, os.cpu_count() or 1)


def cpu_baseline(cfg, seconds, T):
    """Oracle cycles/s on the host, two ways, each over about `seconds`:
    one thread running whole single-sequence cycles of sequences 0-7, and
    every host core with the batch's sequences split between single-threaded
    processes (sequence-parallel).  Both are scaled to the B-sequence batch;
    `value` is the all-cores figure."""
    inputs = OracleInputs(cfg, T)
    one = OraclePool(T, 1, lambda i: list(range(8)), inputs)
    done1, el1, ctx1 = one.ask(("budget", seconds / 2))[0]
    one.close()
    n = min(host_cores(), cfg.B)
    pool = OraclePool(T, n, lambda i: list(range(i, cfg.B, n)), inputs)
    res = pool.ask(("budget", seconds / 2))
    pool.close()
    inputs.close()
    done_n = sum(r[0] for r in res)
    el_n = max(r[1] for r in res)
    ctx_n = sum(r[2] for r in res)
    mean_ctx = float(workloads.seq_lens(cfg).float().mean())
    v1 = done1 / el1 / cfg.B
    vn = done_n / el_n / cfg.B
    return {"value": vn, "unit": UNIT, "cores": n, "kind": "oracle",
            "single_thread_value": v1,
            "sample": "whole single-sequence cycles (fusion of its 8 rows, 5 layers of block attention, "
                      "verification) scaled to the %d-sequence batch.  One thread: %d cycles over sequences 0-7 "
                      "(mean context %.0f vs %.0f for the batch) in %.1f s -> %.4f cycles/s.  All %d cores: the "
                      "batch's sequences split over %d single-threaded processes (sequence-parallel), %d cycles "
                      "(mean context %.0f) in %.1f s -> %.4f cycles/s"
                      % (cfg.B, done1, ctx1 / done1, mean_ctx, el1, v1, n, n, done_n, ctx_n / done_n, el_n, vn)}


def run_reference(args):
    """The oracle as the reference arm: each step is one whole cycle of the
    batch (fusion, five layers of block attention and verification for all
    B sequences), computed by single-threaded host processes that split the
    sequences between them, one per core (rank 0 only)."""
    rank, world, _ = env_rank()
    if rank != 0:
        return
    cfg = workloads.BATCHED
    steps = args.steps if args.steps is not None else 5
    n = min(host_cores(), cfg.B)
    inputs = OracleInputs(cfg, args.temperature)
    pool = OraclePool(args.temperature, n, lambda i: list(range(i, cfg.B, n)), inputs)
    for _ in range(args.warmup):
        pool.ask(("cycle",))
    t0 = time.perf_counter()
    per = []
    for _ in range(steps):
        ts = time.perf_counter()
        pool.ask(("cycle",))
        per.append(time.perf_counter() - ts)
    el = time.perf_counter() - t0
    pool.close()
    inputs.close()
    value = steps / el
    sample_txt = ("%d whole batch cycles (B=%d sequences: fusion of 8 rows each, 5 layers of block attention, "
                  "verification), the sequences split over %d single-threaded processes, %.1f s"
                  % (steps, cfg.B, n, el))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "batched: B=32, ragged context [1024, 8192], 5 layers, block 8, V=262144, T=%g"
                       % args.temperature},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample_txt},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """One roofline measurement (3 warm-up calls, then the timed calls) of a call
    outside the cycle, on the batched workload's shapes, for ncu launch lists."""
    from types import SimpleNamespace
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from __graft_entry__ import build
    build()
    cyc = SimpleNamespace(cfg=workloads.BATCHED, T=args.temperature)
    hbm, tfl, _ = peaks()
    if args.profile == "fusion_tensor":
        line = fusion_tensor_rooflines(dev, tfl)
    elif args.profile == "layer_tail":
        line = layer_tail_roofline(cyc, dev, hbm, tfl)
    elif args.profile == "dflash2":
        line = dflash2_roofline(cyc, dev, hbm)
    else:
        line = draft_head_roofline(cyc, dev, hbm)
    print(json.dumps({"profiling_run": True, "profile": args.profile, **line}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 1000 GPU cycles per repeat; 5 batch cycles for the reference arm)")
    ap.add_argument("--repeats", type=int, default=0,
                    help="timed regions of --steps steps each (default: enough for about 2 s of load); the "
                         "median is reported")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dflash", choices=["dflash", "reference"])
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", default="all", choices=["all", "fuse", "attn", "verify"],
                    help="profiling runs: time one component of the cycle only")
    ap.add_argument("--batch", type=int, default=None, help="profiling runs: smaller batch")
    ap.add_argument("--layers", type=int, default=None, help="profiling runs: fewer draft layers")
    ap.add_argument("--profile", default=None, choices=["layer_tail", "draft_head", "dflash2", "fusion_tensor"],
                    help="profiling runs: only this call's roofline measurement on the batched workload")
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3 and args.impl == "dflash":
        args.warmup = 3
    if args.impl == "dflash" and args.steps is None:
        args.steps = 1000
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
