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
//               clears the work-queue counter of the main kernel.
//   main     -- split-KV, memory-bound: a persistent grid (one CTA per SM)
//               takes work items (sequence, KV head, key split) from an atomic
//               queue; splits of one (sequence, KV head) are near-equal.  A
//               producer warp streams 64-key K/V tiles of the cache (and, for
//               the last split, the block's own keys) with TMA (128-byte
//               swizzle) through a ring of up to six stages.  Q is loaded twice,
//               as MMA rows 0.. and 64.. (two lane quarters); one thread issues
//               S = Q K^T and another O += P V with tcgen05.mma; softmax warps
//               own one query row per thread and per copy, each copy taking
//               one half of every tile's keys, and write P (bf16 hi + lo) to
//               tensor memory.  Epilogue warps merge the two copies (log-sum-
//               exp) and write the output row, or a normalised fp32 partial
//               and its (max, sum) when the item is one of several splits.
//   combine  -- one warp per output row merges the splits' partials
//               (log-sum-exp); launched as a programmatic dependent of main.
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
  int* counters;             // [1] work-queue counter (cleared by the prologue)
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
// split, then the last split of every (b, g), which also carries the block
// keys.  The splits of a sequence are near-equal, so the dynamic queue keeps
// the tail short.
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
  // the sequence's cached keys are cut into nsplit near-equal ranges
  it.kstart = first + static_cast<int>((static_cast<long>(it.s) * ncache) / it.nsplit);
  it.kend = first + static_cast<int>((static_cast<long>(it.s + 1) * ncache) / it.nsplit);
  it.ntiles = it.kend > it.kstart ? (it.kend - it.kstart + kTile - 1) / kTile : 0;
  it.last = it.s == it.nsplit - 1;
  it.nt = it.ntiles + (it.last ? 1 : 0);
  return it;
}

constexpr int kMaxStages = 6;
constexpr int kTcThreads = 352;   // 11 warps, roles below
constexpr int kRowBytes = 128;    // 64 bf16
constexpr int kItemRing = 4;
constexpr int kNumBars = 2 * kMaxStages + 6 * 2 * 2 + 2 * kItemRing;
constexpr int kTmemCols = 512;
// tensor-memory columns: S[2] (fp32, 64 keys), P[2] (bf16 pairs: hi 32, lo 32),
// O[2] (fp32, 128 dims)
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
constexpr uint32_t kIdescQK = umma_idesc_bf16(128, 64, false);
constexpr uint32_t kIdescPV = umma_idesc_bf16(128, 128, true);
constexpr float kRescaleLog2 = 8.0f;

// The Q tile is copied to MMA rows 0.. and 64.. (rows_pad = 32 or 64 query
// rows each), so every query row owns two tensor-memory lanes: copy 0 keeps
// keys 0-31 of each 64-key tile, copy 1 keys 32-63.  Each copy runs its own
// online softmax and accumulates its own partial O; the epilogue merges the
// two (log-sum-exp).  The softmax work of a tile is thus spread over two
// (rows_pad 32) or four (rows_pad 64) SM sub-partitions.
struct TcLayout {
  int rows_pad;
  int off_q, off_x, off_kv, stages, off_bar, off_misc, bytes;
};

__host__ __device__ inline TcLayout tc_layout(int rows, int B, int smem_limit) {
  TcLayout L;
  L.rows_pad = rows > 32 ? 64 : 32;
  // Q: two 64-dim boxes of 128 MMA rows; buffer q sits rows_pad rows in, so for
  // rows_pad = 32 both buffers fit in one 32 KB region, for 64 in two.
  const int qbytes = L.rows_pad == 32 ? 32768 : 65536;
  L.off_q = 0;
  L.off_x = qbytes;                                   // O exchange of copy 1 -> copy 0
  L.off_kv = L.off_x + L.rows_pad * 128 * 4;
  const int misc = 64 + 2 * 2 * 64 * 8 + (2 * B + 1) * 4;
  const int fixed = 1024 + L.off_kv + 8 * kNumBars + misc;
  int st = (smem_limit - fixed) / kStageBytes;
  L.stages = st > kMaxStages ? kMaxStages : st;
  L.off_bar = L.off_kv + L.stages * kStageBytes;
  L.off_misc = L.off_bar + 8 * kNumBars;
  L.bytes = 1024 + L.off_misc + misc;
  return L;
}

// Byte offset of Q buffer `qb` copy `c` box `h` (64-dim half) in the Q region.
__device__ __forceinline__ uint32_t q_off(const TcLayout& L, int qb, int c, int h) {
  if (L.rows_pad == 32) return static_cast<uint32_t>(h * 16384 + c * 8192 + qb * 4096);
  return static_cast<uint32_t>(qb * 32768 + h * 16384 + c * 8192);
}

// Thread `row` owns one query row: write its final output (single split) or
// its normalised partial output and (m, l) for the combine kernel.
__device__ __forceinline__ void finish_item(const Item& it, const AttnParams& p, int row, const float (&o)[HD],
                                            float m, float l) {
  if (row >= p.rows) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (it.nsplit == 1) {
    const size_t out_row0 = (static_cast<size_t>(it.b) * p.Hq + it.g * p.G) * p.bs;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (out_row0 + row) * HD);
#pragma unroll
    for (int i = 0; i < HD / 8; ++i)
      dst[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                          pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                          pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                          pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
    return;
  }
  const size_t r = ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.max_splits + it.s) * p.rows + row;
  float4* dst = reinterpret_cast<float4*>(p.opart + r * HD);
#pragma unroll
  for (int i = 0; i < HD / 4; ++i)
    dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
  p.mlpart[r] = make_float2(m, l);
}

// Log-sum-exp merge of the split partials of every (sequence, KV head) that
// has more than one split: one warp per output row, 4 dims per lane.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
  pdl_wait_primary();
  const int gw = blockIdx.x * 8 + threadIdx.x / 32;   // global warp = (b, g, row)
  const int lane = threadIdx.x % 32;
  const int row = gw % p.rows;
  const int bg = gw / p.rows;
  if (bg >= p.B * p.Hkv) return;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int n = min(max(p.seq_len[b], 0), p.cap);
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int ns = n_splits(n - first, p.chunk);
  if (ns <= 1) return;
  const size_t r0 = static_cast<size_t>(bg) * p.max_splits * p.rows + row;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.mlpart[r0 + static_cast<size_t>(s) * p.rows].x);
  M = warp_max(M);
  const float Mu = M == -INFINITY ? 0.f : M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const size_t r = r0 + static_cast<size_t>(s) * p.rows;
    const float2 ml = p.mlpart[r];
    const float4 o = reinterpret_cast<const float4*>(p.opart + r * HD)[lane];
    const float f = ml.y * exp2f(ml.x - Mu);
    den += f;
    acc.x += f * o.x;
    acc.y += f * o.y;
    acc.z += f * o.z;
    acc.w += f * o.w;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const size_t out_row = (static_cast<size_t>(b) * p.Hq + g * p.G) * p.bs + row;
  reinterpret_cast<uint2*>(p.out + out_row * HD)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

struct AttnMaps {
  CUtensorMap k, v, q, kb, vb;
};

// Index and phase of a ring of two-phase mbarriers.
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
                                         unsigned* status) {
  if (!mbar_wait(it_full + 8 * r.idx, r.phase, status)) return -1;
  const int w = s_item[r.idx];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(it_empty + 8 * r.idx);
  r.next(kItemRing);
  return w;
}

// Roles: warps 0-3 softmax of tensor-memory lane quarter = warp, warps 4-7
// epilogue of lane quarter = warp - 4 (only the quarters holding query rows
// are active), warp 8 TMA producer, warp 9 S = Q K^T issuer, warp 10
// O += P V issuer.
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ AttnMaps maps,
                                                                const AttnParams p, const TcLayout lay) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int S = lay.stages;
  const uint32_t bar0 = base + lay.off_bar;
  const uint32_t kv_full = bar0, kv_empty = bar0 + 8 * kMaxStages;
  const uint32_t q_full = bar0 + 16 * kMaxStages, q_empty = q_full + 16;
  const uint32_t s_full = q_empty + 16, s_empty = s_full + 16;
  const uint32_t p_full = s_empty + 16, p_empty = p_full + 16;
  const uint32_t o_full = p_empty + 16, o_free = o_full + 16;
  const uint32_t ml_full = o_free + 16, ml_empty = ml_full + 16;
  const uint32_t it_full = ml_empty + 16, it_empty = it_full + 8 * kItemRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + lay.off_misc);
  int* s_item = reinterpret_cast<int*>(tmem_slot + 8);                    // kItemRing entries
  float2* s_ml = reinterpret_cast<float2*>(gbase + lay.off_misc + 64);    // [2 buf][2 copy][64 row]
  int* s_prefix = reinterpret_cast<int*>(gbase + lay.off_misc + 64 + 2 * 2 * 64 * 8);
  int* s_n = s_prefix + (p.B + 1);
  float* s_x = reinterpret_cast<float*>(gbase + lay.off_x);             // [rows_pad][128]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = lay.rows_pad / 32;   // lane quarters per copy: 1 or 2
  const int n_sm = 2 * nq;            // active softmax warps (and epilogue warps)
  // quarter q is active when its lanes hold a query row: q % 2 < nq
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(kv_full + 8 * s, 1);
      mbar_init(kv_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + 8 * i, 1);
      mbar_init(q_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, n_sm);
      mbar_init(p_full + 8 * i, n_sm);
      mbar_init(p_empty + 8 * i, 1);
      mbar_init(o_full + 8 * i, 1);
      mbar_init(o_free + 8 * i, n_sm);
      mbar_init(ml_full + 8 * i, n_sm);
      mbar_init(ml_empty + 8 * i, n_sm);
    }
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(it_full + 8 * i, 1);
      mbar_init(it_empty + 8 * i, 2 + 2 * n_sm);
    }
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8) {  // per-sequence lengths and the prefix of full (non-last) splits
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
  pdl_launch_dependents();  // the combine kernel may launch; it waits for this grid
  const uint32_t tmem = *tmem_slot;
  const int n_items = s_prefix[p.B] + p.B * p.Hkv;

  if (warp == 8) {
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
        const int w = atomicAdd(p.counters, 1);
        if (!(ok = mbar_wait(it_empty + 8 * itr.idx, itr.phase ^ 1u, p.status))) break;
        s_item[itr.idx] = w < n_items ? w : -1;
        mbar_arrive(it_full + 8 * itr.idx);
        itr.next(kItemRing);
        if (w >= n_items) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        if (!(ok = mbar_wait(q_empty + 8 * q.idx, q.phase ^ 1u, p.status))) break;
        mbar_arrive_expect_tx(q_full + 8 * q.idx, 4 * lay.rows_pad * kRowBytes);
        const int qrow = (it.b * p.Hq + it.g * p.G) * p.bs;
        for (int c = 0; c < 2; ++c)
          for (int h = 0; h < 2; ++h)
            tma_load_2d(base + lay.off_q + q_off(lay, q.idx, c, h), &maps.q, q_full + 8 * q.idx, 64 * h, qrow);
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
  } else if (warp == 9) {
    // ------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      Ring kv, q, sq, itr;
      bool ok = true;
      while (ok) {
        if (!(ok = mbar_wait(it_full + 8 * itr.idx, itr.phase, p.status))) break;
        const int w = s_item[itr.idx];
        mbar_arrive(it_empty + 8 * itr.idx);
        itr.next(kItemRing);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        if (!(ok = mbar_wait(q_full + 8 * q.idx, q.phase, p.status))) break;
        for (int t = 0; t < it.nt && ok; ++t) {
          if (!(ok = mbar_wait(kv_full + 8 * kv.idx, kv.phase, p.status))) break;
          if (!(ok = mbar_wait(s_empty + 8 * sq.idx, sq.phase ^ 1u, p.status))) break;
          tc_fence_after_sync();
          const uint32_t kb = base + lay.off_kv + kv.idx * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_desc_kmajor_sw128(base + lay.off_q + q_off(lay, q.idx, 0, kk >> 2)) + 2 * (kk & 3);
            const uint64_t bd = umma_desc_kmajor_sw128(kb + (kk >> 2) * kHalfTileBytes) + 2 * (kk & 3);
            umma_bf16(tmem + kColS + 64 * sq.idx, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full + 8 * sq.idx);
          sq.next(2);
          kv.next(S);
        }
        if (!ok) break;
        umma_commit(q_empty + 8 * q.idx);
        q.next(2);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------ O += P V issuer
    if (lane == 0) {
      Ring kv, pr, o, itr;
      bool ok = true;
      while (ok) {
        if (!(ok = mbar_wait(it_full + 8 * itr.idx, itr.phase, p.status))) break;
        const int w = s_item[itr.idx];
        mbar_arrive(it_empty + 8 * itr.idx);
        itr.next(kItemRing);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        const uint32_t od = tmem + kColO + 128 * o.idx;
        for (int t = 0; t < it.nt && ok; ++t) {
          if (!(ok = mbar_wait(p_full + 8 * pr.idx, pr.phase, p.status))) break;
          if (t == 0 && !(ok = mbar_wait(o_free + 8 * o.idx, o.phase ^ 1u, p.status))) break;
          tc_fence_after_sync();
          const uint32_t vbase = base + lay.off_kv + kv.idx * kStageBytes + 2 * kHalfTileBytes;
          const uint64_t vdesc = umma_desc_mnmajor_sw128(vbase, kHalfTileBytes, 1024);
          const uint32_t pa = tmem + kColP + 64 * pr.idx;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ts(od, pa + 32 * h + 8 * kk, vdesc + 128 * kk, kIdescPV, (t == 0 && h == 0 && kk == 0) ? 0u : 1u);
          umma_commit(p_empty + 8 * pr.idx);
          umma_commit(kv_empty + 8 * kv.idx);
          pr.next(2);
          kv.next(S);
        }
        if (!ok) break;
        umma_commit(o_full + 8 * o.idx);
        o.next(2);
      }
    }
  } else if (warp <= 3) {
    // ------------------------------------------------ softmax
    if ((warp & 1) < nq) {
      const int lg = 32 * warp + lane;         // tensor-memory lane
      const int row = lg % 64;                 // query row (rows_pad = 32: quarters 0, 2)
      const int copy = lg / 64;                // copy 0: keys 0-31, copy 1: keys 32-63
      const int key0 = 32 * copy;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
      const float scale = p.scale_log2;
      {  // the other copy's key columns of both P buffers stay zero for the whole kernel
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
        for (int pb = 0; pb < 2; ++pb) {
          tmem_st_32cols(tl + kColP + 64 * pb, z);
          tmem_st_32cols(tl + kColP + 64 * pb + 32, z);
        }
        tmem_st_wait();
        tc_fence_before_sync();
      }
      Ring sr, mlr, itr;
      int ob = 0, pb = 0;
      int pcnt[2] = {0, 0};
      bool ok = true;
      while (ok) {
        const int w = next_item(it_full, it_empty, s_item, itr, p.status);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        float m_used = -INFINITY, l = 0.f;
        for (int t = 0; t < it.nt; ++t) {
          if (!(ok = mbar_wait(s_full + 8 * sr.idx, sr.phase, p.status))) break;
          tc_fence_after_sync();
          float x[32];
          {
            uint32_t r[32];
            tmem_ld_32cols(tl + kColS + 64 * sr.idx + key0, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_empty + 8 * sr.idx);
          sr.next(2);
          const int nvalid = (t < it.ntiles ? min(kTile, it.kend - (it.kstart + t * kTile)) : p.bs) - key0;
          if (nvalid < 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i >= nvalid) x[i] = -INFINITY;
          }
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(x[4 * i], x[4 * i + 1]), fmaxf(x[4 * i + 2], x[4 * i + 3]));
#pragma unroll
          for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
            for (int i = 0; i < w2; ++i) mx[i] = fmaxf(mx[i], mx[i + w2]);
          const float mt = mx[0] * scale;
          const bool need = m_used == -INFINITY ? (mt != -INFINITY) : (mt > m_used + kRescaleLog2);
          if (__any_sync(0xffffffffu, need) && t > 0) {
            // this copy's O must hold every P V product up to tile t-1 before it is rescaled
            const int xb = pb ^ 1;
            if (!(ok = mbar_wait(p_empty + 8 * xb, (pcnt[xb] - 1) & 1, p.status))) break;
            tc_fence_after_sync();
            const float f = need ? (m_used == -INFINITY ? 0.f : exp2f(m_used - mt)) : 1.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t r[32];
              tmem_ld_32cols(tl + kColO + 128 * ob + 32 * c, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
              tmem_st_32cols(tl + kColO + 128 * ob + 32 * c, r);
            }
            tmem_st_wait();
          }
          if (need) {
            l = (m_used == -INFINITY) ? 0.f : l * exp2f(m_used - mt);
            m_used = mt;
          }
          const float nm = -(m_used == -INFINITY ? 0.f : m_used);
          // P over this copy's 32 keys as bf16 hi + lo pairs
          uint32_t hv[16], lv[16];
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = exp2f(fmaf(x[2 * i], scale, nm));
            const float c2 = exp2f(fmaf(x[2 * i + 1], scale, nm));
            ls[i & 3] += a + c2;
            hv[i] = pack_bf16x2(a, c2);
            lv[i] = pack_bf16x2(a - bf16_lo(hv[i]), c2 - bf16_hi(hv[i]));
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          // P[pb] is free once the P V product that last read it has completed
          if (pcnt[pb] > 0 && !(ok = mbar_wait(p_empty + 8 * pb, (pcnt[pb] - 1) & 1, p.status))) break;
          tc_fence_after_sync();
          tmem_st_16cols(tl + kColP + 64 * pb + 16 * copy, hv);
          tmem_st_16cols(tl + kColP + 64 * pb + 32 + 16 * copy, lv);
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full + 8 * pb);
          ++pcnt[pb];
          pb ^= 1;
        }
        if (!ok) break;
        // hand (m, l) of this copy to the epilogue warps
        if (!(ok = mbar_wait(ml_empty + 8 * mlr.idx, mlr.phase ^ 1u, p.status))) break;
        s_ml[(mlr.idx * 2 + copy) * 64 + row] = make_float2(m_used, l);
        __syncwarp();
        if (lane == 0) mbar_arrive(ml_full + 8 * mlr.idx);
        mlr.next(2);
        ob ^= 1;
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 4-7)
    const int e = warp - 4;
    if ((e & 1) < nq) {
      const int lg = 32 * e + lane;
      const int row = lg % 64;
      const int copy = lg / 64;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * e) << 16);
      Ring orr, mlr, itr;
      bool ok = true;
      while (ok) {
        const int w = next_item(it_full, it_empty, s_item, itr, p.status);
        if (w < 0) break;
        const Item it = decode_item(w, s_prefix, s_n, p);
        if (!(ok = mbar_wait(o_full + 8 * orr.idx, orr.phase, p.status))) break;
        tc_fence_after_sync();
        float o[HD];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tl + kColO + 128 * orr.idx + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = __uint_as_float(r[i]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free + 8 * orr.idx);
        orr.next(2);
        if (!(ok = mbar_wait(ml_full + 8 * mlr.idx, mlr.phase, p.status))) break;
        const float2 mine = s_ml[(mlr.idx * 2 + copy) * 64 + row];
        const float2 other = s_ml[(mlr.idx * 2 + (copy ^ 1)) * 64 + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(ml_empty + 8 * mlr.idx);
        mlr.next(2);
        // merge the two copies' partial softmax states (log-sum-exp)
        const float M = fmaxf(mine.x, other.x);
        const float Mu = M == -INFINITY ? 0.f : M;
        const float fm = mine.x == -INFINITY ? 0.f : exp2f(mine.x - Mu);
        const float fo = other.x == -INFINITY ? 0.f : exp2f(other.x - Mu);
        if (copy == 1) {
          float4* xr = reinterpret_cast<float4*>(s_x + row * HD);
#pragma unroll
          for (int i = 0; i < HD / 4; ++i)
            xr[i] = make_float4(o[4 * i] * fm, o[4 * i + 1] * fm, o[4 * i + 2] * fm, o[4 * i + 3] * fm);
        }
        named_barrier_sync(1, 32 * n_sm);
        if (copy == 0) {
          const float4* xr = reinterpret_cast<const float4*>(s_x + row * HD);
#pragma unroll
          for (int i = 0; i < HD / 4; ++i) {
            const float4 v = xr[i];
            o[4 * i] = o[4 * i] * fm + v.x;
            o[4 * i + 1] = o[4 * i + 1] * fm + v.y;
            o[4 * i + 2] = o[4 * i + 2] * fm + v.z;
            o[4 * i + 3] = o[4 * i + 3] * fm + v.w;
          }
        }
        named_barrier_sync(1, 32 * n_sm);  // s_x is free for the next item
        if (copy == 0) finish_item(it, p, row, o, M, mine.y * fm + other.y * fo);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
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
  long c = (static_cast<long>(B) * Hkv * keys) / 3600;
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
         align256(sizeof(int));
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
  p.counters = w.take<int>(1);
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
      c.capacity, eps, inv, qh, kbh, p.counters, 1, dev.status);

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
  if (p.max_splits > 1) {
    cudaLaunchConfig_t cc = cfg;
    const long warps = static_cast<long>(B) * Hkv * p.rows;
    cc.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
    cc.blockDim = dim3(256);
    cc.dynamicSmemBytes = 0;
    le = cudaLaunchKernelEx(&cc, attn_combine_kernel, p);
    if (le != cudaSuccess) return cuda_fail(le, "attn_combine_kernel launch");
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "block attention launch");
}

}  // namespace dflash
