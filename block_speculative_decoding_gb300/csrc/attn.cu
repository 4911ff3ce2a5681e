// Non-causal draft-block attention of one layer over the cached context.
//
// Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash",
// sections "The released serving cycle" (one non-causal forward over the
// eight-position block) and "Five target states become persistent draft
// context" (Q [B,32,8,128], K/V [B,8,8,128], four query heads per KV head,
// per-head Q/K RMSNorm before RoPE, attention over the cached context plus the
// block); "DFlash & DFlash2: Block-Diffusion LLM-Speedup" 4.1 (K_i, V_i are the
// injected context rows followed by the block rows).
//
// Kernels:
//   prologue -- per (sequence, block row): RMSNorm * gain and RoPE of every
//               query head and block key, rounded to the storage dtype; also
//               clears the split counters of the merge below.
//   main     -- split-KV, memory-bound: a persistent grid walks work items
//               (sequence, KV head, key split).  A producer warp streams 64-key
//               K/V tiles of the cache (and, for the last split, the block's
//               own keys) with TMA (128-byte swizzle) through a 4-stage ring;
//               one thread issues tcgen05.mma for S = Q K^T and O += P V into
//               tensor memory; two softmax warps own one query row per thread
//               (all Hq/Hkv heads x bs block rows of the KV head share every
//               tile).  The last CTA to finish a (sequence, KV head) merges the
//               splits' partial outputs (log-sum-exp).
// fp32 storage uses a plain SIMT kernel (parity path for the tiny fp32 case).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dflash_device.cuh"
#include "dflash_internal.h"

namespace dflash {
namespace {

constexpr int HD = 128;
constexpr int kTile = 64;                       // keys per TMA stage
constexpr int kHalfTileBytes = kTile * 64 * 2;  // 64 keys x 64 dims bf16 = 8 KB (one TMA box)
constexpr int kStageBytes = 4 * kHalfTileBytes; // K (2 boxes) + V (2 boxes) = 32 KB
constexpr int kMaxBatch = 2048;
constexpr double kTwoPi = 6.283185307179586476925286766559;

struct InvFreq {
  double v[HD / 2];
};

struct AttnParams {
  int B, bs, G, Hkv, Hq, cap, layer, window, chunk, max_splits, rows;
  const int32_t* seq_len;
  const __nv_bfloat16* qh;   // [B, Hq, bs, 128]   prologue output
  const __nv_bfloat16* kbh;  // [B, Hkv, bs, 128]  prologue output
  const __nv_bfloat16* vb;   // [B, Hkv, bs, 128]  block values (input)
  __nv_bfloat16* out;        // [B, Hq, bs, 128]
  float* opart;              // [B, Hkv, max_splits, rows, 128] normalised partial outputs
  float2* mlpart;            // [B, Hkv, max_splits, rows]      (max, sum) in log2 units
  float scale_log2;          // log2(e) / sqrt(128)
  int* counters;             // [B, Hkv] finished splits (cleared by the prologue)
  unsigned* status;
};

__device__ __forceinline__ int clamp_seq(int n, int cap, unsigned* status) {
  if (n < 0 || n > cap) {
    raise_status(status, DFLASH_DEV_BAD_SEQLEN);
    return n < 0 ? 0 : cap;
  }
  return n;
}

__host__ __device__ __forceinline__ int n_splits(int ncache, int chunk) {
  return ncache <= 0 ? 1 : (ncache + chunk - 1) / chunk;
}

// --------------------------------------------------------------------------
// prologue: q^ = RoPE(RMSNorm(q) * q_gain), k^_b = RoPE(RMSNorm(kb) * k_gain)
// --------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) attn_prologue_kernel(
    const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ qg,
    const T* __restrict__ kg, const int32_t* __restrict__ seq_len, int B, int bs, int Hq, int Hkv,
    int cap, float eps, InvFreq inv_freq, T* __restrict__ qh, T* __restrict__ kbh,
    int* __restrict__ counters, int n_counters, unsigned* status) {
  pdl_launch_dependents();
  if (blockIdx.x == 0 && counters)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  const int b = blockIdx.x / bs, j = blockIdx.x % bs;
  const int n = clamp_seq(seq_len[b], cap, status);
  const int pos = n + j;
  __shared__ float s_cos[HD / 2], s_sin[HD / 2];
  if (threadIdx.x < HD / 2) {
    double ang = static_cast<double>(pos) * inv_freq.v[threadIdx.x];
    ang -= kTwoPi * rint(ang / kTwoPi);
    float sv, cv;
    sincosf(static_cast<float>(ang), &sv, &cv);
    s_cos[threadIdx.x] = cv;
    s_sin[threadIdx.x] = sv;
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = 2 * lane;  // this lane owns elements e0, e0+1 and e0+64, e0+65
  for (int v = warp; v < Hq + Hkv; v += 8) {
    const bool isq = v < Hq;
    const T* src = isq ? q + ((static_cast<size_t>(b) * Hq + v) * bs + j) * HD
                       : kb + ((static_cast<size_t>(b) * Hkv + (v - Hq)) * bs + j) * HD;
    T* dst = isq ? qh + ((static_cast<size_t>(b) * Hq + v) * bs + j) * HD
                 : kbh + ((static_cast<size_t>(b) * Hkv + (v - Hq)) * bs + j) * HD;
    const T* gain = isq ? qg : kg;
    float x0 = to_f32<T>(src[e0]), x1 = to_f32<T>(src[e0 + 1]);
    float y0 = to_f32<T>(src[e0 + 64]), y1 = to_f32<T>(src[e0 + 65]);
    const float ss = warp_sum(x0 * x0 + x1 * x1 + y0 * y0 + y1 * y1);
    const float r = rsqrtf(ss * (1.0f / HD) + eps);
    const float g0 = gain ? to_f32<T>(gain[e0]) : 1.f, g1 = gain ? to_f32<T>(gain[e0 + 1]) : 1.f;
    const float g2 = gain ? to_f32<T>(gain[e0 + 64]) : 1.f, g3 = gain ? to_f32<T>(gain[e0 + 65]) : 1.f;
    x0 *= r * g0;
    x1 *= r * g1;
    y0 *= r * g2;
    y1 *= r * g3;
    const float c0 = s_cos[e0], s0 = s_sin[e0], c1 = s_cos[e0 + 1], s1 = s_sin[e0 + 1];
    dst[e0] = from_f32<T>(x0 * c0 - y0 * s0);
    dst[e0 + 1] = from_f32<T>(x1 * c1 - y1 * s1);
    dst[e0 + 64] = from_f32<T>(y0 * c0 + x0 * s0);
    dst[e0 + 65] = from_f32<T>(y1 * c1 + x1 * s1);
  }
}

// --------------------------------------------------------------------------
// --------------------------------------------------------------------------
// main split-KV kernel (bf16): tcgen05 tensor cores, TMA, TMEM accumulators
// --------------------------------------------------------------------------
//
// Work item = (sequence b, KV head g, key split s).  Per 64-key tile:
//   S   = Q K^T   tcgen05.mma M=128 (query rows; the Hq/Hkv*bs real rows sit in
//                 TMEM lanes 0..rows-1), N=64 keys, K=128 -> TMEM (2 buffers)
//   P   = 2^(S*scale - m)   one thread per query row (softmax warps 0, 1),
//                 written to shared memory as bf16 hi + lo (K-major, swizzled)
//   O  += P V     tcgen05.mma M=128, N=128 dims, K=64 keys, V read MN-major
//                 straight from the TMA tile -> TMEM accumulator
// The running max is only refreshed (and O rescaled) when it grows by more
// than 2^8, so P stays within [0, 256].
// Roles: warps 0-1 softmax/epilogue, warp 2 TMA producer, warp 3 MMA issuer.

struct Item {
  int b, g, s, nsplit, kstart, kend, ntiles, nt;  // nt = ntiles + (last split ? 1 block tile : 0)
  bool last;
};

// Work items in the order the queue hands them out: first every non-last
// split (all `chunk` keys long), then the last split of every (b, g) (the
// ragged remainder plus the block keys) -- largest first, so the dynamic queue
// balances like longest-processing-time scheduling.
__device__ __forceinline__ Item decode_item(int w, const int* s_full_prefix, const int* s_n, const AttnParams& p) {
  Item it;
  const int F = s_full_prefix[p.B];
  int b, g, s;
  if (w < F) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {  // largest b with prefix[b] <= w
      const int mid = (lo + hi + 1) >> 1;
      if (s_full_prefix[mid] <= w) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int nfull = (s_full_prefix[b + 1] - s_full_prefix[b]) / p.Hkv;
    const int r = w - s_full_prefix[b];
    g = r / nfull;
    s = r % nfull;
  } else {
    b = (w - F) / p.Hkv;
    g = (w - F) % p.Hkv;
    s = -1;
  }
  const int n = s_n[b];
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int ncache = n - first;
  it.b = b;
  it.g = g;
  it.nsplit = n_splits(ncache, p.chunk);
  it.s = s < 0 ? it.nsplit - 1 : s;
  it.kstart = first + it.s * p.chunk;
  it.kend = first + min(ncache, (it.s + 1) * p.chunk);
  it.ntiles = it.kend > it.kstart ? (it.kend - it.kstart + kTile - 1) / kTile : 0;
  it.last = it.s == it.nsplit - 1;
  it.nt = it.ntiles + (it.last ? 1 : 0);
  return it;
}

constexpr int kMaxStages = 6;
constexpr int kTcThreads = 224;   // 7 warps, roles below
constexpr int kRowBytes = 128;    // 64 bf16
constexpr int kItemRing = 4;
constexpr int kItemConsumers = 6; // QK issuer, PV issuer, 2 softmax warps, 2 epilogue warps
constexpr int kNumBars = 2 * kMaxStages + 2 * 2 * 6 + 2 * kItemRing;
constexpr int kTmemCols = 512;
// tensor-memory columns: S[2] 64 each, O[2] 128 each, P[2] = {hi 32, lo 32}
// (bf16 pairs packed per 32-bit column)
constexpr uint32_t kColS = 0, kColO0 = 128, kColP = 256, kColO1 = 384;
constexpr uint32_t kIdescQK = umma_idesc_bf16(128, 64, false);
constexpr uint32_t kIdescPV = umma_idesc_bf16(128, 128, true);
constexpr float kRescaleLog2 = 8.0f;

__device__ __forceinline__ uint32_t col_o(int ob) { return ob ? kColO1 : kColO0; }

// Shared-memory plan (byte offsets from the 1024-aligned base): Q double
// buffer (the A operand of S = Q K^T; the M=128 MMA reads 128 rows, the rows
// past rows_pad fall on the following buffers and only feed accumulator lanes
// that are never read), then the K/V stage ring, barriers and small arrays.
struct TcLayout {
  int rows_pad, half;   // half = rows_pad * 128 bytes: one 64-dim half of Q
  int off_q, off_kv, stages, off_bar, off_misc, bytes;
};

__host__ __device__ inline TcLayout tc_layout(int rows, int B, int smem_limit) {
  TcLayout L;
  L.rows_pad = rows > 32 ? 64 : 32;
  L.half = L.rows_pad * kRowBytes;
  L.off_q = 0;                      // Q[buf][box] at (2*buf + box) * half
  L.off_kv = 4 * L.half;            // stage s at off_kv + s * kStageBytes
  const int misc = 64 + 2 * 64 * 8 + (2 * B + 1) * 4;  // tmem slot, flags, items, (m, l)[2][64], prefix, n
  const int fixed = 1024 + L.off_kv + 8 * kNumBars + misc;
  int st = (smem_limit - fixed) / kStageBytes;
  L.stages = st > kMaxStages ? kMaxStages : st;
  L.off_bar = L.off_kv + L.stages * kStageBytes;
  L.off_misc = L.off_bar + 8 * kNumBars;
  L.bytes = 1024 + L.off_misc + misc;
  return L;
}

// Thread `row` owns one query row: write its final output, or its normalised
// partial and (m, l); the last CTA to finish a (b, g) merges the splits.
// `bar_id` / `leader` name the named barrier and thread of the 64 epilogue threads.
__device__ __forceinline__ void finish_item(const Item& it, const AttnParams& p, int row, const float (&o)[HD],
                                            float m, float l, int* s_flag, int bar_id, int leader) {
  const bool real = row < p.rows;
  const size_t out_row0 = (static_cast<size_t>(it.b) * p.Hq + it.g * p.G) * p.bs;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (it.nsplit == 1) {
    if (real) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (out_row0 + row) * HD);
#pragma unroll
      for (int i = 0; i < HD / 8; ++i)
        dst[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                            pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                            pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                            pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
    }
    return;
  }
  const size_t bg = static_cast<size_t>(it.b) * p.Hkv + it.g;
  const size_t part0 = bg * p.max_splits * p.rows;
  if (real) {
    float4* dst = reinterpret_cast<float4*>(p.opart + (part0 + static_cast<size_t>(it.s) * p.rows + row) * HD);
#pragma unroll
    for (int i = 0; i < HD / 4; ++i)
      dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
    p.mlpart[part0 + static_cast<size_t>(it.s) * p.rows + row] = make_float2(m, l);
  }
  __threadfence();
  named_barrier_sync(bar_id, 64);
  if (threadIdx.x == leader) *s_flag = (atomicAdd(p.counters + bg, 1) == it.nsplit - 1);
  named_barrier_sync(bar_id, 64);
  const int last = *s_flag;
  named_barrier_sync(bar_id, 64);  // s_flag is reused by the next item
  if (!last) return;
  __threadfence();
  if (!real) return;
  // this CTA finished (b, g) last: log-sum-exp merge of all its splits
  const float2* ml = p.mlpart + part0 + row;
  float M = -INFINITY;
  for (int s = 0; s < it.nsplit; ++s) M = fmaxf(M, __ldcg(ml + static_cast<size_t>(s) * p.rows).x);
  const float Mu = M == -INFINITY ? 0.f : M;
  float acc[HD];
#pragma unroll
  for (int i = 0; i < HD; ++i) acc[i] = 0.f;
  float den = 0.f;
  for (int s = 0; s < it.nsplit; ++s) {
    const float2 v = __ldcg(ml + static_cast<size_t>(s) * p.rows);
    const float f = v.y * exp2f(v.x - Mu);
    den += f;
    const float4* src = reinterpret_cast<const float4*>(p.opart + (part0 + static_cast<size_t>(s) * p.rows + row) * HD);
#pragma unroll
    for (int i = 0; i < HD / 4; ++i) {
      const float4 x = __ldcg(src + i);
      acc[4 * i] += f * x.x;
      acc[4 * i + 1] += f * x.y;
      acc[4 * i + 2] += f * x.z;
      acc[4 * i + 3] += f * x.w;
    }
  }
  const float dinv = den > 0.f ? 1.f / den : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(p.out + (out_row0 + row) * HD);
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
    dst[i] = make_uint4(pack_bf16x2(acc[8 * i] * dinv, acc[8 * i + 1] * dinv),
                        pack_bf16x2(acc[8 * i + 2] * dinv, acc[8 * i + 3] * dinv),
                        pack_bf16x2(acc[8 * i + 4] * dinv, acc[8 * i + 5] * dinv),
                        pack_bf16x2(acc[8 * i + 6] * dinv, acc[8 * i + 7] * dinv));
}

struct AttnMaps {
  CUtensorMap k, v, q, kb, vb;
};

// Ring of two-phase mbarriers shared by one producer role and one consumer role.
struct Ring {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Reads the next work item from the shared item ring (-1 = no more work).
__device__ __forceinline__ int next_item(uint32_t it_full, uint32_t it_empty, const int* s_item, Ring& r,
                                         unsigned* status, bool warp_wide) {
  if (!mbar_wait(it_full + 8 * r.idx, r.phase, status)) return -1;
  const int w = s_item[r.idx];
  if (warp_wide) __syncwarp();
  if (!warp_wide || (threadIdx.x & 31) == 0) mbar_arrive(it_empty + 8 * r.idx);
  r.next(kItemRing);
  return w;
}

// Roles: warp 0/1 softmax of query rows 0-31 / 32-63 (tensor-memory lane
// quarters 0/1), warp 2 TMA producer, warp 3 S = Q K^T issuer, warp 4/5
// epilogue of rows 0-31 / 32-63, warp 6 O += P V issuer.
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ AttnMaps maps,
                                                                const AttnParams p, const TcLayout lay) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int S = lay.stages;
  const int half = lay.half;
  const uint32_t bar0 = base + lay.off_bar;
  const uint32_t kv_full = bar0, kv_empty = bar0 + 8 * kMaxStages;
  const uint32_t q_full = bar0 + 16 * kMaxStages, q_empty = q_full + 16;
  const uint32_t s_full = q_empty + 16, s_empty = s_full + 16;
  const uint32_t p_full = s_empty + 16, p_empty = p_full + 16;
  const uint32_t o_full = p_empty + 16, o_free = o_full + 16;
  const uint32_t ml_full = o_free + 16, ml_empty = ml_full + 16;
  const uint32_t it_full = ml_empty + 16, it_empty = it_full + 8 * kItemRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + lay.off_misc);
  int* s_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_item = reinterpret_cast<int*>(tmem_slot + 8);            // kItemRing entries
  float2* s_ml = reinterpret_cast<float2*>(gbase + lay.off_misc + 64);  // [2][64] (m, l) per row
  int* s_prefix = reinterpret_cast<int*>(gbase + lay.off_misc + 64 + 2 * 64 * 8);
  int* s_n = s_prefix + (p.B + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(kv_full + 8 * s, 1);
      mbar_init(kv_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + 8 * i, 1);
      mbar_init(q_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, 2);
      mbar_init(p_full + 8 * i, 2);
      mbar_init(p_empty + 8 * i, 1);
      mbar_init(o_full + 8 * i, 1);
      mbar_init(o_free + 8 * i, 2);
      mbar_init(ml_full + 8 * i, 2);
      mbar_init(ml_empty + 8 * i, 2);
    }
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(it_full + 8 * i, 1);
      mbar_init(it_empty + 8 * i, kItemConsumers);
    }
    mbar_fence_init();
  }
  if (warp == 3) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {  // per-sequence lengths and the prefix of full (non-last) splits
    for (int b = lane; b < p.B; b += 32) s_n[b] = clamp_seq(p.seq_len[b], p.cap, p.status);
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int b = 0; b < p.B; ++b) {
        s_prefix[b] = acc;
        const int first = p.window > 0 ? max(0, s_n[b] - p.window) : 0;
        acc += (n_splits(s_n[b] - first, p.chunk) - 1) * p.Hkv;
      }
      s_prefix[p.B] = acc;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int n_items = s_prefix[p.B] + p.B * p.Hkv;

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.q);
      pdl_wait_primary();  // the prologue's Q, block keys and cleared counters
      const uint64_t pol = l2_policy_evict_first();
      Ring kv, q, itr;
      bool ok = true;
      while (ok) {
        const int w = atomicAdd(p.counters + p.B * p.Hkv, 1);
        if (!(ok = mbar_wait(it_empty + 8 * itr.idx, itr.phase ^ 1u, p.status))) break;
        s_item[itr.idx] = w < n_items ? w : -1;
        mbar_arrive(it_full + 8 * itr.idx);
        itr.next(kItemRing);
        if (w >= n_items) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        if (!(ok = mbar_wait(q_empty + 8 * q.idx, q.phase ^ 1u, p.status))) break;
        mbar_arrive_expect_tx(q_full + 8 * q.idx, 2 * half);
        const int qrow = (it.b * p.Hq + it.g * p.G) * p.bs;
        const uint32_t qdst = base + lay.off_q + 2 * q.idx * half;
        tma_load_2d(qdst, &maps.q, q_full + 8 * q.idx, 0, qrow);
        tma_load_2d(qdst + half, &maps.q, q_full + 8 * q.idx, 64, qrow);
        q.next(2);
        const int rowbase = ((p.layer * p.B + it.b) * p.Hkv + it.g) * p.cap;
        const int brow = (it.b * p.Hkv + it.g) * p.bs;
        for (int t = 0; t < it.nt; ++t) {
          if (!(ok = mbar_wait(kv_empty + 8 * kv.idx, kv.phase ^ 1u, p.status))) break;
          const uint32_t fb = kv_full + 8 * kv.idx;
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint32_t dst = base + lay.off_kv + kv.idx * kStageBytes;
          if (t < it.ntiles) {
            const int y = rowbase + it.kstart + t * kTile;
            tma_load_2d_hint(dst, &maps.k, fb, 0, y, pol);
            tma_load_2d_hint(dst + kHalfTileBytes, &maps.k, fb, 64, y, pol);
            tma_load_2d_hint(dst + 2 * kHalfTileBytes, &maps.v, fb, 0, y, pol);
            tma_load_2d_hint(dst + 3 * kHalfTileBytes, &maps.v, fb, 64, y, pol);
          } else {  // the block's own keys and values
            tma_load_2d(dst, &maps.kb, fb, 0, brow);
            tma_load_2d(dst + kHalfTileBytes, &maps.kb, fb, 64, brow);
            tma_load_2d(dst + 2 * kHalfTileBytes, &maps.vb, fb, 0, brow);
            tma_load_2d(dst + 3 * kHalfTileBytes, &maps.vb, fb, 64, brow);
          }
          kv.next(S);
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      Ring kv, q, sr, itr;
      bool ok = true;
      while (ok) {
        const int w = next_item(it_full, it_empty, s_item, itr, p.status, false);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        if (!(ok = mbar_wait(q_full + 8 * q.idx, q.phase, p.status))) break;
        const uint32_t qa = base + lay.off_q + 2 * q.idx * half;
        for (int t = 0; t < it.nt && ok; ++t) {
          if (!(ok = mbar_wait(kv_full + 8 * kv.idx, kv.phase, p.status))) break;
          if (!(ok = mbar_wait(s_empty + 8 * sr.idx, sr.phase ^ 1u, p.status))) break;
          tc_fence_after_sync();
          const uint32_t kb = base + lay.off_kv + kv.idx * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_desc_kmajor_sw128(qa + (kk >> 2) * half) + 2 * (kk & 3);
            const uint64_t bd = umma_desc_kmajor_sw128(kb + (kk >> 2) * kHalfTileBytes) + 2 * (kk & 3);
            umma_bf16(tmem + kColS + 64 * sr.idx, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full + 8 * sr.idx);
          sr.next(2);
          kv.next(S);
        }
        if (!ok) break;
        umma_commit(q_empty + 8 * q.idx);
        q.next(2);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------ O += P V issuer
    if (lane == 0) {
      Ring kv, pr, orr, itr;
      bool ok = true;
      while (ok) {
        const int w = next_item(it_full, it_empty, s_item, itr, p.status, false);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        const uint32_t od = tmem + col_o(orr.idx);
        for (int t = 0; t < it.nt && ok; ++t) {
          if (!(ok = mbar_wait(p_full + 8 * pr.idx, pr.phase, p.status))) break;
          if (t == 0 && !(ok = mbar_wait(o_free + 8 * orr.idx, orr.phase ^ 1u, p.status))) break;
          tc_fence_after_sync();
          const uint32_t vbase = base + lay.off_kv + kv.idx * kStageBytes + 2 * kHalfTileBytes;
          const uint64_t vdesc = umma_desc_mnmajor_sw128(vbase, kHalfTileBytes, 1024);
          const uint32_t pa = tmem + kColP + 64 * pr.idx;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ts(od, pa + 32 * h + 8 * kk, vdesc + 128 * kk, kIdescPV, (t == 0 && h == 0 && kk == 0) ? 0u : 1u);
          umma_commit(kv_empty + 8 * kv.idx);
          umma_commit(p_empty + 8 * pr.idx);
          pr.next(2);
          kv.next(S);
        }
        if (!ok) break;
        umma_commit(o_full + 8 * orr.idx);
        orr.next(2);
      }
    }
  } else if (warp <= 1) {
    // ------------------------------------------------ softmax (one thread per query row)
    const int row = 32 * warp + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    // A warp whose 32 rows are all padding keeps every wait and arrive (so
    // the barrier phases stay in step) but does no math.
    const bool act = 32 * warp < lay.rows_pad;
    const float scale = p.scale_log2;
    Ring sr, pr, mlr, itr;
    int ob = 0;
    int pcnt[2] = {0, 0};
    bool ok = true;
    while (ok) {
      const int w = next_item(it_full, it_empty, s_item, itr, p.status, true);
      if (w < 0) break;
      const Item it = decode_item(w, s_prefix, s_n, p);
      float m_used = -INFINITY, l = 0.f;
      for (int t = 0; t < it.nt; ++t) {
        if (!(ok = mbar_wait(s_full + 8 * sr.idx, sr.phase, p.status))) break;
        tc_fence_after_sync();
        uint32_t sv[64];
        if (act) {
          tmem_ld_32cols(tl + kColS + 64 * sr.idx, *reinterpret_cast<uint32_t(*)[32]>(sv));
          tmem_ld_32cols(tl + kColS + 64 * sr.idx + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
          tmem_ld_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty + 8 * sr.idx);
        sr.next(2);
        uint32_t hv[32], lv[32];
        if (act) {
          float x[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(sv[i]);
          const int nvalid = t < it.ntiles ? min(kTile, it.kend - (it.kstart + t * kTile)) : p.bs;
          if (nvalid < kTile) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i >= nvalid) x[i] = -INFINITY;
          }
          // tile max of the raw scores (scale > 0), tree-reduced
          float mx[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[i] = fmaxf(fmaxf(x[4 * i], x[4 * i + 1]), fmaxf(x[4 * i + 2], x[4 * i + 3]));
#pragma unroll
          for (int w2 = 8; w2 >= 1; w2 >>= 1)
#pragma unroll
            for (int i = 0; i < w2; ++i) mx[i] = fmaxf(mx[i], mx[i + w2]);
          const float mt = mx[0] * scale;
          if (t == 0) {
            m_used = mt;
          } else {
            const bool need = mt > m_used + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
              // O must hold every P V product up to tile t-1 before it is rescaled
              const int xb = pr.idx ^ 1;
              if (!(ok = mbar_wait(p_empty + 8 * xb, (pcnt[xb] - 1) & 1, p.status))) break;
              tc_fence_after_sync();
              const float f = need ? exp2f(m_used - mt) : 1.f;
              if (need) {
                l *= f;
                m_used = mt;
              }
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld_32cols(tl + col_o(ob) + 32 * c, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                tmem_st_32cols(tl + col_o(ob) + 32 * c, r);
              }
              tmem_st_wait();
              tc_fence_before_sync();
            }
          }
          const float nm = -(m_used == -INFINITY ? 0.f : m_used);
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float a = exp2f(fmaf(x[2 * i], scale, nm));
            const float b = exp2f(fmaf(x[2 * i + 1], scale, nm));
            ls[i & 3] += a + b;
            hv[i] = pack_bf16x2(a, b);
            lv[i] = pack_bf16x2(a - bf16_lo(hv[i]), b - bf16_hi(hv[i]));
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        // P[pb] is free once the P V product that last read it has completed
        if (pcnt[pr.idx] > 0 && !(ok = mbar_wait(p_empty + 8 * pr.idx, (pcnt[pr.idx] - 1) & 1, p.status))) break;
        tc_fence_after_sync();
        if (act) {
          tmem_st_32cols(tl + kColP + 64 * pr.idx, hv);
          tmem_st_32cols(tl + kColP + 64 * pr.idx + 32, lv);
          tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 8 * pr.idx);
        ++pcnt[pr.idx];
        pr.next(2);
      }
      if (!ok) break;
      // hand (m, l) of this item to the epilogue warps
      if (!(ok = mbar_wait(ml_empty + 8 * mlr.idx, mlr.phase ^ 1u, p.status))) break;
      s_ml[mlr.idx * 64 + row] = make_float2(m_used, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(ml_full + 8 * mlr.idx);
      mlr.next(2);
      ob ^= 1;
    }
  } else {
    // ------------------------------------------------ epilogue (warps 4, 5)
    const int row = 32 * (warp - 4) + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp - 4)) << 16);
    const bool act = 32 * (warp - 4) < lay.rows_pad;
    Ring orr, mlr, itr;
    bool ok = true;
    while (ok) {
      const int w = next_item(it_full, it_empty, s_item, itr, p.status, true);
      if (w < 0) break;
      const Item it = decode_item(w, s_prefix, s_n, p);
      if (!(ok = mbar_wait(o_full + 8 * orr.idx, orr.phase, p.status))) break;
      tc_fence_after_sync();
      float o[HD];
      if (act) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tl + col_o(orr.idx) + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = __uint_as_float(r[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < HD; ++i) o[i] = 0.f;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free + 8 * orr.idx);
      orr.next(2);
      if (!(ok = mbar_wait(ml_full + 8 * mlr.idx, mlr.phase, p.status))) break;
      const float2 ml = s_ml[mlr.idx * 64 + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(ml_empty + 8 * mlr.idx);
      mlr.next(2);
      finish_item(it, p, row, o, ml.x, ml.y, s_flag, 2, 128);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 3) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------------------
// fp32 SIMT path: one CTA per (sequence, query head)
// --------------------------------------------------------------------------
constexpr int kF32Keys = 128;

__global__ void __launch_bounds__(128) attn_f32_kernel(const float* __restrict__ qh,
                                                       const float* __restrict__ kbh,
                                                       const float* __restrict__ vb,
                                                       const float* __restrict__ ck,
                                                       const float* __restrict__ cv,
                                                       const int32_t* __restrict__ seq_len, int B,
                                                       int bs, int Hq, int Hkv, int cap, int layer,
                                                       int window, float scale,
                                                       float* __restrict__ out) {
  const int b = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const int g = h / (Hq / Hkv);
  const int n = min(max(seq_len[b], 0), cap);
  const int first = window > 0 ? max(0, n - window) : 0;
  const int ncache = n - first;
  const int total = ncache + bs;
  __shared__ float s_q[16][HD];
  __shared__ float s_p[16][kF32Keys];
  __shared__ float s_corr[16];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid; i < bs * HD; i += blockDim.x)
    s_q[i / HD][i % HD] = qh[((static_cast<size_t>(b) * Hq + h) * bs + i / HD) * HD + i % HD];
  float m_run[16], l_run[16], o[16];
  for (int j = 0; j < 16; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
    o[j] = 0.f;
  }
  const size_t crow = ((static_cast<size_t>(layer) * B + b) * Hkv + g) * cap;
  const size_t brow = (static_cast<size_t>(b) * Hkv + g) * bs;
  auto key_ptr = [&](int v, const float* c, const float* blk) -> const float* {
    return v < ncache ? c + (crow + first + v) * HD : blk + (brow + (v - ncache)) * HD;
  };
  __syncthreads();
  for (int t0 = 0; t0 < total; t0 += kF32Keys) {
    const int v = t0 + tid;
    if (v < total) {
      const float* kp = key_ptr(v, ck, kbh);
      for (int j = 0; j < bs; ++j) {
        float acc = 0.f;
        for (int e = 0; e < HD; ++e) acc += s_q[j][e] * kp[e];
        s_p[j][tid] = acc * scale;
      }
    } else {
      for (int j = 0; j < bs; ++j) s_p[j][tid] = -INFINITY;
    }
    __syncthreads();
    for (int j = warp; j < bs; j += 4) {  // each warp owns rows j = warp (mod 4)
      float mx = -INFINITY;
      for (int i = lane; i < kF32Keys; i += 32) mx = fmaxf(mx, s_p[j][i]);
      mx = warp_max(mx);
      const float mnew = fmaxf(m_run[j], mx);
      const float corr = expf(m_run[j] - mnew);
      float sum = 0.f;
      for (int i = lane; i < kF32Keys; i += 32) {
        const float pv = expf(s_p[j][i] - mnew);
        s_p[j][i] = pv;
        sum += pv;
      }
      sum = warp_sum(sum);
      l_run[j] = l_run[j] * corr + sum;
      m_run[j] = mnew;
      if (lane == 0) s_corr[j] = corr;
    }
    __syncthreads();
    for (int j = 0; j < bs; ++j) {
      float acc = o[j] * s_corr[j];
      for (int i = 0; i < kF32Keys && t0 + i < total; ++i)
        acc += s_p[j][i] * key_ptr(t0 + i, cv, vb)[tid];
      o[j] = acc;
    }
    __syncthreads();
  }
  __shared__ float s_l[16];
  for (int j = warp; j < bs; j += 4)
    if (lane == 0) s_l[j] = l_run[j];
  __syncthreads();
  for (int j = 0; j < bs; ++j)
    out[((static_cast<size_t>(b) * Hq + h) * bs + j) * HD + tid] = o[j] / s_l[j];
}


int pick_chunk(int B, int Hkv, int cap, int window) {
  const long keys = window > 0 ? std::min(window, cap) : cap;
  long c = (static_cast<long>(B) * Hkv * keys) / 2400;
  c = (c + 63) / 64 * 64;
  return static_cast<int>(std::min<long>(4096, std::max<long>(256, c)));
}

}  // namespace

size_t attn_ws_bytes(int B, int bs, int Hq, int Hkv, int cap, int window, dflash_dtype dt) {
  const size_t esz = dt == DFLASH_BF16 ? 2 : 4;
  const int rows = (Hq / Hkv) * bs;
  const int chunk = pick_chunk(B, Hkv, cap, window);
  const int keys = window > 0 ? std::min(window, cap) : cap;
  const int max_splits = n_splits(keys, chunk);
  size_t s = align256(static_cast<size_t>(B) * Hq * bs * HD * esz) +
             align256(static_cast<size_t>(B) * Hkv * bs * HD * esz);
  if (dt == DFLASH_BF16)
    s += align256(static_cast<size_t>(B) * Hkv * max_splits * rows * HD * sizeof(float)) +
         align256(static_cast<size_t>(B) * Hkv * max_splits * rows * sizeof(float2)) +
         align256((static_cast<size_t>(B) * Hkv + 1) * sizeof(int));
  return s + 256;
}

dflash_status launch_block_attn(int layer, int B, int bs, int Hq, const void* q, const void* kb,
                                const void* vb, const void* qg, const void* kg, float theta,
                                float eps, const dflash_kv_cache& c, int window, void* out, void* ws,
                                cudaStream_t st, const DeviceInfo& dev) {
  const int Hkv = c.num_kv_heads;
  const int G = Hq / Hkv;
  InvFreq inv;
  for (int e = 0; e < HD / 2; ++e) inv.v[e] = std::pow(static_cast<double>(theta), -2.0 * e / HD);
  WsCarver w(ws);
  const float scale = 1.0f / std::sqrt(static_cast<float>(HD));
  if (c.dtype == DFLASH_F32) {
    float* qh = w.take<float>(static_cast<size_t>(B) * Hq * bs * HD);
    float* kbh = w.take<float>(static_cast<size_t>(B) * Hkv * bs * HD);
    attn_prologue_kernel<float><<<B * bs, 256, 0, st>>>(
        static_cast<const float*>(q), static_cast<const float*>(kb), static_cast<const float*>(qg),
        static_cast<const float*>(kg), c.seq_len, B, bs, Hq, Hkv, c.capacity, eps, inv, qh, kbh, nullptr, 0,
        dev.status);
    attn_f32_kernel<<<B * Hq, 128, 0, st>>>(qh, kbh, static_cast<const float*>(vb),
                                            static_cast<const float*>(c.k), static_cast<const float*>(c.v),
                                            c.seq_len, B, bs, Hq, Hkv, c.capacity, layer, window, scale,
                                            static_cast<float*>(out));
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "fp32 block attention launch");
  }
  if (B > kMaxBatch) return fail(DFLASH_ERR_UNSUPPORTED, "block_attn: bf16 batch must be <= 2048");
  AttnParams p;
  p.B = B;
  p.bs = bs;
  p.G = G;
  p.Hkv = Hkv;
  p.Hq = Hq;
  p.cap = c.capacity;
  p.layer = layer;
  p.window = window;
  p.chunk = pick_chunk(B, Hkv, c.capacity, window);
  const int keys = window > 0 ? std::min(window, c.capacity) : c.capacity;
  p.max_splits = n_splits(keys, p.chunk);
  p.rows = G * bs;
  p.seq_len = c.seq_len;
  auto* qh = w.take<__nv_bfloat16>(static_cast<size_t>(B) * Hq * bs * HD);
  auto* kbh = w.take<__nv_bfloat16>(static_cast<size_t>(B) * Hkv * bs * HD);
  p.qh = qh;
  p.kbh = kbh;
  p.vb = static_cast<const __nv_bfloat16*>(vb);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.opart = w.take<float>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows * HD);
  p.mlpart = w.take<float2>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows);
  p.counters = w.take<int>(static_cast<size_t>(B) * Hkv + 1);  // + the work-queue counter
  p.scale_log2 = 1.4426950408889634f * scale;
  p.status = dev.status;

  AttnMaps maps;
  const uint64_t rows = static_cast<uint64_t>(c.num_layers) * c.batch * Hkv * c.capacity;
  dflash_status s = make_tmap_bf16_2d(&maps.k, c.k, rows, HD, kTile, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.v, c.v, rows, HD, kTile, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.q, qh, static_cast<uint64_t>(B) * Hq * bs, HD, p.rows > 32 ? 64 : 32, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.kb, kbh, static_cast<uint64_t>(B) * Hkv * bs, HD, kTile, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.vb, vb, static_cast<uint64_t>(B) * Hkv * bs, HD, kTile, 64);
  if (s) return s;

  attn_prologue_kernel<__nv_bfloat16><<<B * bs, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kb),
      static_cast<const __nv_bfloat16*>(qg), static_cast<const __nv_bfloat16*>(kg), c.seq_len, B, bs, Hq, Hkv,
      c.capacity, eps, inv, qh, kbh, p.counters, B * Hkv + 1, dev.status);

  const TcLayout lay = tc_layout(p.rows, B, static_cast<int>(dev.max_smem_optin));
  if (lay.stages < 2) return fail(DFLASH_ERR_UNSUPPORTED, "block_attn: shared memory");
  static int configured_device = -1;
  if (configured_device != dev.device) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(dev.max_smem_optin));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_tc_kernel)");
    configured_device = dev.device;
  }
  const long upper = static_cast<long>(B) * Hkv * p.max_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<long>(upper, dev.num_sms)));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(lay.bytes);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, attn_tc_kernel, maps, p, lay);
  if (le != cudaSuccess) return cuda_fail(le, "attn_tc_kernel launch");
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "block attention launch");
}

}  // namespace dflash
