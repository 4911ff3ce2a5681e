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
// Kernels (three launches per call, each a programmatic dependent of the one
// before it):
//   clear    -- one CTA: waits for the preceding grid, releases the main
//               kernel, and clears the work-queue counter and the per-pair
//               counters.
//   main     -- split-KV, memory-bound: a persistent grid (one CTA per SM)
//               takes work items (sequence, KV head, key split), the first one
//               per CTA by its index (so it starts while the counters are
//               being cleared) and the rest from an atomic queue; the producer
//               warp decodes each item once and hands it to the other roles
//               through shared memory.  The producer loads the pair's raw query
//               rows (and the block's raw keys) into shared memory, where the
//               epilogue warps apply RMSNorm * gain and RoPE in place, one item
//               ahead of their epilogue work.  The products are
//               taken transposed: the 128 keys of a tile fill the tensor
//               core's M and the G * bs query rows of the pair (padded to
//               NC = 32 or 64) its N.  The producer streams 128-key K and V
//               tiles of the cache (and, for the last split, the block's own
//               values; its keys sit in their own buffer) with TMA (128-byte
//               swizzle) through K and V rings sized to the shared memory (two
//               K and three V stages at 227 KB); one thread issues
//               S^T = K Q^T into tensor memory, eight softmax warps (one key per thread) write
//               P^T = 2^(S^T scale - m) to shared memory as bf16 hi + lo parts,
//               another thread issues O^T += V^T [P_hi^T P_lo^T], and four
//               epilogue warps add the hi and lo columns and write the output
//               row, or a normalised fp32 partial and its (max, sum) when the
//               item is one of several splits.  The running max of each row is
//               fixed per item from its first tile.
//   combine  -- one warp per output row merges the splits' partials
//               (log-sum-exp) as soon as its pair's splits are written, and
//               recomputes exactly any pair whose scores outgrew the max.
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
constexpr int kKeys = 128;                      // keys per tile (the tensor core's M)
constexpr int kBoxBytes = kKeys * 64 * 2;       // 128 keys x 64 dims bf16 = 16 KB (one TMA box)
constexpr int kHalfBytes = 2 * kBoxBytes;       // K (or V) of one tile: 32 KB
constexpr int kMaxBatch = 2048;

struct InvFreq {
  unsigned long long v[HD / 2];  // round(2^64 inv_freq[e] / 2 pi): turns per position, 64-bit fraction
};

struct AttnParams {
  int B, bs, G, Hkv, Hq, cap, ring, layer, window, chunk, max_splits, rows;
  const int32_t* seq_len;
  const __nv_bfloat16* q;    // [B, Hq, bs, 128]   block queries (input, before norm and RoPE)
  const __nv_bfloat16* kb;   // [B, Hkv, bs, 128]  block keys (input, before norm and RoPE)
  const __nv_bfloat16* qg;   // [128] query-norm gain (nullptr = ones)
  const __nv_bfloat16* kg;   // [128] key-norm gain (nullptr = ones)
  const __nv_bfloat16* vb;   // [B, Hkv, bs, 128]  block values (input)
  __nv_bfloat16* out;        // [B, Hq, bs, 128]
  float* opart;              // [B, Hkv, max_splits, rows, 128] normalised partial outputs
  float2* mlpart;            // [B, Hkv, max_splits, rows]      (max, sum) in log2 units
  const __nv_bfloat16* ck;   // this cache's K and V, [L, B, Hkv, cap, 128] (paged: [L, num_pages, Hkv, page_size, 128])
  const __nv_bfloat16* cv;
  const int32_t* table;      // paged layout: [B, max_pages] block table; nullptr: linear or ring
  int max_pages, page_size, num_pages;
  float scale_log2;          // log2(e) / sqrt(128)
  int* counters;             // [1 + 2 B Hkv], cleared before the main kernel: the work-queue counter, per (b, g)
                             // a flag (scores outgrew the running max), then per (b, g) the count of
                             // epilogue warps (4 per split) that finished writing
  unsigned* status;
  unsigned long long wait_limit_ns;  // the combine kernel's bounded wait for a pair's splits
  float eps;                         // RMSNorm epsilon of the query and key norms
  InvFreq inv;                       // RoPE frequencies as fixed-point turns per position
};

// Cached rows a sequence attends to: its length, clamped to the capacity; a
// ring cache (sliding window) holds the latest min(n, cap) positions.
__device__ __forceinline__ int cached_rows(int n, int cap, int ring, unsigned* status) {
  if (n < 0 || (!ring && n > cap)) raise_status(status, DFLASH_DEV_BAD_SEQLEN);
  return min(max(n, 0), cap);
}

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

// sin and cos of the RoPE angle at position pos of the frequency whose turns
// per position are f (a 64-bit fraction): pos * f mod 2^64 is the angle in
// turns, exact to 2^-34 turn for any position below 2^31; its top 32 bits, as
// a signed turn in [-1/2, 1/2), give sin / cos of pi * [-1, 1).
__device__ __forceinline__ void rope_sincos(int pos, unsigned long long f, float* sv, float* cv) {
  const unsigned long long t = static_cast<unsigned long long>(pos) * f;
  sincospif(static_cast<float>(static_cast<int>(t >> 32)) * 0x1p-31f, sv, cv);
}

// --------------------------------------------------------------------------
// fp32 prologue: q^ = RoPE(RMSNorm(q) * q_gain), k^_b = RoPE(RMSNorm(kb) * k_gain)
// into the workspace (the bf16 path does this inside the main kernel)
// --------------------------------------------------------------------------
constexpr int kPrologueThreads = 256;

// Elements (e, e + 1) of an fp32 head vector, e even: one 8-byte access,
// aligned because the rows are 16-byte aligned.
template <typename T>
__device__ __forceinline__ float2 load_pair(const T* p);
template <>
__device__ __forceinline__ float2 load_pair<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <typename T>
__device__ __forceinline__ void store_pair(T* p, float a, float b);
template <>
__device__ __forceinline__ void store_pair<float>(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}

template <typename T>
__global__ void __launch_bounds__(kPrologueThreads) attn_prologue_kernel(
    const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ qg,
    const T* __restrict__ kg, const int32_t* __restrict__ seq_len, int B, int bs, int Hq, int Hkv,
    int cap, int ring, float eps, InvFreq inv_freq, T* __restrict__ qh, T* __restrict__ kbh,
    int* __restrict__ counters, int n_counters, unsigned* status) {
  // Launched as a programmatic dependent of whatever precedes it in the stream
  // (its CTAs become resident early): nothing is read or written before the
  // preceding grid has completed, and the main kernel (which reads sequence
  // lengths before its own wait) is released only after that.
  pdl_wait_primary();
  pdl_launch_dependents();
  q = pdl_fresh(q);
  kb = pdl_fresh(kb);
  qg = pdl_fresh(qg);
  kg = pdl_fresh(kg);
  seq_len = pdl_fresh(seq_len);
  const int b = blockIdx.x / bs, j = blockIdx.x % bs;
  // the sequence length first: the angles that depend on it are this
  // kernel's longest chain, so its load is not queued behind the others
  const int n_in = seq_len[b];
  if (blockIdx.x == 0 && counters)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = 2 * lane;  // this lane owns elements e0, e0+1 and e0+64, e0+65
  constexpr int kWarps = kPrologueThreads / 32;
  constexpr int kBatch = 5;  // head vectors a warp loads before working on them
  // this lane's elements of the two gains, shared by all head vectors
  const float gq0 = qg ? to_f32<T>(qg[e0]) : 1.f, gq1 = qg ? to_f32<T>(qg[e0 + 1]) : 1.f;
  const float gq2 = qg ? to_f32<T>(qg[e0 + 64]) : 1.f, gq3 = qg ? to_f32<T>(qg[e0 + 65]) : 1.f;
  const float gk0 = kg ? to_f32<T>(kg[e0]) : 1.f, gk1 = kg ? to_f32<T>(kg[e0 + 1]) : 1.f;
  const float gk2 = kg ? to_f32<T>(kg[e0 + 64]) : 1.f, gk3 = kg ? to_f32<T>(kg[e0 + 65]) : 1.f;
  // a batch of a warp's head vectors, two pair loads per vector
  float2 xa[kBatch], xb[kBatch];
  auto load_batch = [&](int v0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + u * kWarps;
      if (v < Hq + Hkv) {
        const T* src = v < Hq ? q + ((static_cast<size_t>(b) * Hq + v) * bs + j) * HD
                              : kb + ((static_cast<size_t>(b) * Hkv + (v - Hq)) * bs + j) * HD;
        xa[u] = load_pair<T>(src + e0);
        xb[u] = load_pair<T>(src + e0 + 64);
      }
    }
  };
  // the first batch does not depend on the position: load it before the angles
  load_batch(warp);
  // the block's positions follow the sequence: seq_len (a ring cache's
  // length may exceed its capacity) plus j
  const int n = ring ? max(n_in, 0) : clamp_seq(n_in, cap, status);
  const int pos = n + j;
  __shared__ float s_cos[HD / 2], s_sin[HD / 2];
  if (threadIdx.x < HD / 2) {
    float sv, cv;
    rope_sincos(pos, inv_freq.v[threadIdx.x], &sv, &cv);
    s_cos[threadIdx.x] = cv;
    s_sin[threadIdx.x] = sv;
  }
  __syncthreads();
  const float c0 = s_cos[e0], s0 = s_sin[e0], c1 = s_cos[e0 + 1], s1 = s_sin[e0 + 1];
  for (int v0 = warp; v0 < Hq + Hkv; v0 += kWarps * kBatch) {
    if (v0 != warp) load_batch(v0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + u * kWarps;
      if (v >= Hq + Hkv) break;
      const bool isq = v < Hq;
      T* dst = isq ? qh + ((static_cast<size_t>(b) * Hq + v) * bs + j) * HD
                   : kbh + ((static_cast<size_t>(b) * Hkv + (v - Hq)) * bs + j) * HD;
      float x0 = xa[u].x, x1 = xa[u].y, y0 = xb[u].x, y1 = xb[u].y;
      const float ss = warp_sum(x0 * x0 + x1 * x1 + y0 * y0 + y1 * y1);
      const float r = rsqrtf(ss * (1.0f / HD) + eps);
      x0 *= r * (isq ? gq0 : gk0);
      x1 *= r * (isq ? gq1 : gk1);
      y0 *= r * (isq ? gq2 : gk2);
      y1 *= r * (isq ? gq3 : gk3);
      store_pair<T>(dst + e0, x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
      store_pair<T>(dst + e0 + 64, y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
    }
  }
}

// --------------------------------------------------------------------------
// main split-KV kernel (bf16): tcgen05 tensor cores, TMA, TMEM accumulators
// --------------------------------------------------------------------------
//
// The products are taken transposed, so that the 128 keys of a tile fill the
// tensor core's M dimension and the few query rows of a (sequence, KV head)
// (G * bs <= 64, padded to NC = 32 or 64) its N dimension:
//   S^T = K Q^T    M = 128 keys, N = NC query rows, K = 128 dims; A = the K
//                  tile (K-major), B = Q (K-major) -> tensor memory, key k in
//                  lane k
//   P^T = 2^(S^T * scale - m)   one softmax thread per key (lane), NC/32
//                  warps per lane quarter; written to shared memory as bf16
//                  hi and lo parts side by side (MN-major: the 2 NC values of
//                  one key contiguous)
//   O^T += V^T [P_hi^T P_lo^T]   M = 128 dims, N = 2 NC, K = 128 keys; A = the
//                  V tile read MN-major, B = P^T -> tensor memory, dim d in
//                  lane d; the epilogue adds the hi and lo columns
// The running max m of each query row is set once per work item, from its
// first tile, and shared by all keys (threads).  A later score may exceed it
// by up to 2^64 without loss: P, its sums and O stay finite in fp32 / bf16 and
// bf16 hi + lo keeps ~16 bits relative to each value.  If any score exceeds it
// by more than that, the (sequence, KV head) is flagged and the combine kernel
// recomputes its rows exactly.  The row sums are kept per thread and reduced
// over the keys once per work item.

struct Item {
  int b, g, s, nsplit, kstart, kend, ntiles, nt;  // nt = ntiles + (last split ? 1 block tile : 0)
  bool last;
};

__host__ __device__ __forceinline__ int split_start(int s, int nsplit, int ncache) {
  if (s <= 0) return 0;
  if (s >= nsplit) return ncache;
  // near-equal ranges, interior boundaries on whole tiles
  return static_cast<int>((static_cast<long>(s) * ncache) / nsplit) & ~(kKeys - 1);
}

// Work items in the order the queue hands them out: first every non-last
// split, then the last split of every (b, g), which also carries the block
// keys.  The splits of a sequence are near-equal, so the dynamic queue keeps
// the tail short.
__device__ __forceinline__ Item decode_item(int w, const int* s_full_prefix, const int* s_n, const int* s_multi,
                                            const AttnParams& p) {
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
    // last splits: those of sequences with several splits first (their merges
    // can then finish before the queue's end), then the one-split sequences
    const int M = s_multi[p.B];
    const int wl = w - F;
    const bool multi = wl < M * p.Hkv;
    const int idx = multi ? wl / p.Hkv : (wl - M * p.Hkv) / p.Hkv;
    g = wl % p.Hkv;
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {  // largest b whose count of earlier multi (or one-split) sequences is <= idx
      const int mid = (lo + hi + 1) >> 1;
      const int before = multi ? s_multi[mid] : mid - s_multi[mid];
      if (before <= idx) lo = mid; else hi = mid - 1;
    }
    b = lo;
    s = -1;
  }
  const int n = s_n[b];
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int ncache = n - first;
  it.b = b;
  it.g = g;
  it.nsplit = n_splits(ncache, p.chunk);
  it.s = s < 0 ? it.nsplit - 1 : s;
  it.kstart = first + split_start(it.s, it.nsplit, ncache);
  it.kend = first + split_start(it.s + 1, it.nsplit, ncache);
  it.ntiles = it.kend > it.kstart ? (it.kend - it.kstart + kKeys - 1) / kKeys : 0;
  it.last = it.s == it.nsplit - 1;
  it.nt = it.ntiles + (it.last ? 1 : 0);
  return it;
}

// Keys of tile t of an item that hold data (the block tile holds bs keys).
__device__ __forceinline__ int tile_keys(const Item& it, int t, int bs) {
  return t < it.ntiles ? min(kKeys, it.kend - (it.kstart + t * kKeys)) : bs;
}

constexpr int kMaxRing = 4;       // K and V ring stages (each)
constexpr int kSBufs = 4;         // S^T buffers in tensor memory
constexpr int kItemRing = 4;
constexpr int kBlockBoxRows = 16; // block keys per TMA box (bs <= 16)
constexpr int kBlkBoxBytes = kBlockBoxRows * 128;  // one 64-dim box of the block keys
constexpr int kNumBars = 4 * kMaxRing + 2 * 2 + 2 * kSBufs + 4 * 2 + 2 * 2 + 2 * kItemRing + 2 + 2;
constexpr float kOverflowLog2 = 64.0f;  // largest score above the running max, in log2 units

template <int NC>
struct TcCfg {
  static constexpr int kCPW = NC == 32 ? 16 : 32;    // query rows (columns) per softmax warp
  static constexpr int kSoftWarps = 4 * (NC / kCPW);  // two softmax warps per lane quarter
  static constexpr int kEpiWarp0 = kSoftWarps;      // 4 epilogue warps, one per lane quarter
  static constexpr int kProdWarp = kSoftWarps + 4;
  static constexpr int kSWarp = kSoftWarps + 5;     // S^T = K Q^T issuer (also allocates TMEM)
  static constexpr int kOWarp = kSoftWarps + 6;     // O^T += V^T P^T issuer
  static constexpr int kThreads = 32 * (kSoftWarps + 7);
  // tensor memory: S^T [kSBufs] x NC columns, then O^T [2] x 2 NC columns (hi, lo)
  static constexpr uint32_t kTmemCols = NC == 32 ? 256 : 512;
  static constexpr uint32_t kColS = 0, kColO = kSBufs * NC;
  static constexpr int kQBoxBytes = NC * 128;       // NC rows x 64 dims bf16
  // P^T of one tile: 128 keys x (NC hi + NC lo) bf16, 128-byte swizzled rows of
  // 64 values; NC = 32: one row per key (hi | lo); NC = 64: a hi block of 128
  // rows, then a lo block
  static constexpr int kPBytes = kKeys * 2 * NC * 2;
  static constexpr uint32_t kPLoOffset = NC == 32 ? 64u : 16384u;   // lo part of a key's values
  static constexpr uint32_t kIdescS = umma_idesc_bf16(128, NC, false, false);
  static constexpr uint32_t kIdescO = umma_idesc_bf16(128, 2 * NC, true, true);
};

struct TcLayout {
  int nk, nv;
  int off_q, off_kb, off_p, off_k, off_v, off_bar, off_misc, bytes;
};

__host__ __device__ inline int tc_misc_bytes(int B, int nc) {
  // tmem slot (64) | RoPE turns per position [64] (u64) | gains [2][128] (bf16) |
  // s_m [2][NC] | s_l [2][4][NC] | s_red [2 halves][2][4][32] |
  // prefix [B+1], n [B] | decoded item ring [kItemRing]
  return 64 + 512 + 512 + 2 * nc * 4 + 2 * 4 * nc * 4 + 2 * 2 * 4 * 32 * 4 + (3 * B + 2) * 4 +
         kItemRing * static_cast<int>(sizeof(Item));
}

__host__ __device__ inline TcLayout tc_layout(int nc, int B, int smem_limit) {
  TcLayout L;
  L.off_q = 0;                           // 2 buffers x 2 boxes of NC rows
  // 2 buffers x 2 boxes of the block keys.  The block tile's S product reads
  // 128 rows from a box; the 112 past its 16 lie in the next buffers and the
  // P region (masked keys: their scores are never used).
  L.off_kb = 4 * nc * 128;
  L.off_p = L.off_kb + 4 * kBlkBoxBytes;  // 2 buffers of P^T (hi and lo)
  L.off_k = L.off_p + 2 * kKeys * 2 * nc * 2;
  const int fixed = 1024 + L.off_k + 8 * kNumBars + tc_misc_bytes(B, nc);
  int total = (smem_limit - fixed) / kHalfBytes;
  if (total > 2 * kMaxRing) total = 2 * kMaxRing;
  L.nv = (total + 1) / 2;
  L.nk = total - L.nv;
  L.off_v = L.off_k + L.nk * kHalfBytes;
  L.off_bar = L.off_v + L.nv * kHalfBytes;
  L.off_misc = L.off_bar + 8 * kNumBars;
  L.bytes = 1024 + L.off_misc + tc_misc_bytes(B, nc);
  return L;
}

// Row of the cache's [rows][128] view that holds position pos of (sequence b,
// KV head g) in this layer; page: the block-table entry of pos (paged only).
__device__ __forceinline__ long cache_row(const AttnParams& p, int b, int g, int pos, int page) {
  if (p.table) return ((static_cast<long>(p.layer) * p.num_pages + page) * p.Hkv + g) * p.page_size + pos % p.page_size;
  return ((static_cast<long>(p.layer) * p.B + b) * p.Hkv + g) * p.cap + pos;
}

// This lane's four elements (4 lane .. 4 lane + 3) of RoPE(RMSNorm(x) * gain)
// at position pos, rounded to bf16 as the tensor-core path stores them; the
// rotation partner of element e < 64 is e + 64, held by lane ^ 16.
__device__ float4 norm_rope_lanes(const __nv_bfloat16* x, const __nv_bfloat16* gain, float eps, int pos,
                                  const InvFreq& inv) {
  const int lane = threadIdx.x % 32;
  float v[4];
  {
    const float4 t = bf16x4_to_f32(x + 4 * lane);
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  }
  const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
  const float rn = rsqrtf(ss * (1.0f / HD) + eps);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= rn * (gain ? __bfloat162float(gain[4 * lane + i]) : 1.f);
  float out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float w = __shfl_xor_sync(0xffffffffu, v[i], 16);
    float sv, cv;
    rope_sincos(pos, inv.v[(4 * lane + i) & 63], &sv, &cv);
    // first half: x cos - y sin; second half: y cos + x sin (x = element e, y = e + 64)
    out[i] = lane < 16 ? v[i] * cv - w * sv : v[i] * cv + w * sv;
    out[i] = __bfloat162float(__float2bfloat16_rn(out[i]));
  }
  return make_float4(out[0], out[1], out[2], out[3]);
}

// One output row computed key by key (4 dims per lane, exact running max):
// the fallback for a (sequence, KV head) whose scores outgrew the running max
// of the tensor-core kernel.  The query and the block keys are normalised and
// rotated here from the inputs, as the main kernel does in shared memory.
__device__ void attn_row_exact(const AttnParams& p, int b, int g, int row, int first, int n) {
  const int lane = threadIdx.x % 32;
  const int h = g * p.G + row / p.bs, j = row % p.bs;
  // the block's positions follow the sequence: its length (a ring cache's
  // may exceed the capacity), else the cached rows
  const int pos0 = p.ring ? max(p.seq_len[b], 0) : n;
  const float4 q = norm_rope_lanes(p.q + ((static_cast<size_t>(b) * p.Hq + h) * p.bs + j) * HD, p.qg, p.eps,
                                   pos0 + j, p.inv);
  const size_t bbase = (static_cast<size_t>(b) * p.Hkv + g) * p.bs;
  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = first; t < n + p.bs; ++t) {
    const bool blk = t >= n;
    long crow = 0;
    bool zero = false;  // a paged position whose block-table entry is outside the pool reads zeros
    if (!blk) {
      int page = 0;
      if (p.table) {
        page = p.table[static_cast<size_t>(b) * p.max_pages + t / p.page_size];
        zero = page < 0 || page >= p.num_pages;
        if (zero) raise_status(p.status, DFLASH_DEV_BAD_SEQLEN);
      }
      crow = zero ? 0 : cache_row(p, b, g, t, page);
    }
    const __nv_bfloat16* vr = blk ? p.vb + (bbase + (t - n)) * HD : p.cv + crow * HD;
    const float4 k = blk    ? norm_rope_lanes(p.kb + (bbase + (t - n)) * HD, p.kg, p.eps, pos0 + (t - n), p.inv)
                     : zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                            : bf16x4_to_f32(p.ck + crow * HD + 4 * lane);
    const float s = warp_sum(q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w) * p.scale_log2;
    const float4 v = zero ? make_float4(0.f, 0.f, 0.f, 0.f) : bf16x4_to_f32(vr + 4 * lane);
    if (s > m) {
      const float f = exp2f(m - s);
      l *= f;
      acc.x *= f;
      acc.y *= f;
      acc.z *= f;
      acc.w *= f;
      m = s;
    }
    const float e = exp2f(s - m);
    l += e;
    acc.x += e * v.x;
    acc.y += e * v.y;
    acc.z += e * v.z;
    acc.w += e * v.w;
  }
  const float inv = 1.f / l;
  const size_t out_row = (static_cast<size_t>(b) * p.Hq + g * p.G) * p.bs + row;
  reinterpret_cast<uint2*>(p.out + out_row * HD)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// Clears the main kernel's counters.  Launched as a programmatic dependent of
// whatever precedes it in the stream, it waits for that grid (which may have
// written the block's queries, keys or the sequence lengths) and only then
// releases the main kernel, whose first work items need none of the counters;
// the main kernel's threads wait for this grid before they touch them.  It
// also asks L2 for the block's raw query and key rows (a few MB), which every
// work item loads just before it needs them.
constexpr uint32_t kPrefetchChunk = 4096;
__global__ void __launch_bounds__(1024) attn_clear_kernel(int* __restrict__ counters, int n,
                                                          const uint8_t* __restrict__ q, size_t q_bytes,
                                                          const uint8_t* __restrict__ kb, size_t kb_bytes) {
  pdl_wait_primary();
  pdl_launch_dependents();
  for (size_t off = static_cast<size_t>(threadIdx.x) * kPrefetchChunk; off < q_bytes;
       off += static_cast<size_t>(blockDim.x) * kPrefetchChunk)
    prefetch_l2_bulk(q + off, static_cast<uint32_t>(q_bytes - off < kPrefetchChunk ? q_bytes - off : kPrefetchChunk));
  for (size_t off = static_cast<size_t>(threadIdx.x) * kPrefetchChunk; off < kb_bytes;
       off += static_cast<size_t>(blockDim.x) * kPrefetchChunk)
    prefetch_l2_bulk(kb + off, static_cast<uint32_t>(kb_bytes - off < kPrefetchChunk ? kb_bytes - off : kPrefetchChunk));
  for (int i = threadIdx.x; i < n; i += blockDim.x) counters[i] = 0;
}

// Per output row (one warp, 4 dims per lane): the log-sum-exp merge of the
// split partials of a (sequence, KV head) with more than one split, or the
// exact recomputation of a (sequence, KV head) the main kernel flagged.
// Launched as a programmatic dependent of the main kernel but without waiting
// for its whole grid: a warp starts on (b, g) as soon as the main kernel's
// epilogue warps have written all of its splits (a counter per pair, four
// arrivals per split), so the merges overlap the main kernel's last items.
// Five CTAs per SM: the exact path's registers (rare) do not cost the merges' occupancy.
__global__ void __launch_bounds__(256, 5) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_launch_dependents();  // a following call's first kernel may become resident; it waits for this grid
  const int gw = blockIdx.x * 8 + threadIdx.x / 32;   // global warp = (b, g, row)
  const int lane = threadIdx.x % 32;
  const int row = gw % p.rows;
  const int bg = gw / p.rows;
  if (bg >= p.B * p.Hkv) return;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int n = min(max(p.seq_len[b], 0), p.cap);
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int nsplit = n_splits(n - first, p.chunk);
  bool ready = true;
  if (lane == 0)
    ready = wait_counter_at_least(p.counters + 1 + p.B * p.Hkv + bg, 4 * nsplit, p.status, p.wait_limit_ns);
  if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) return;
  if (__ldcg(p.counters + 1 + bg) != 0) {
    attn_row_exact(p, b, g, row, first, n);
    return;
  }
  const int ns = nsplit;
  if (ns <= 1) return;
  const size_t r0 = static_cast<size_t>(bg) * p.max_splits * p.rows + row;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, __ldcg(p.mlpart + r0 + static_cast<size_t>(s) * p.rows).x);
  M = warp_max(M);
  const float Mu = M == -INFINITY ? 0.f : M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const size_t r = r0 + static_cast<size_t>(s) * p.rows;
    const float2 ml = __ldcg(p.mlpart + r);  // written by other SMs during this kernel
    const float4 o = __ldcg(reinterpret_cast<const float4*>(p.opart + r * HD) + lane);
    const float f = ml.y * exp2f(ml.x - Mu);
    den += f;
    acc.x += f * o.x;
    acc.y += f * o.y;
    acc.z += f * o.z;
    acc.w += f * o.w;
  }
  // this row's split outputs (512 bytes each) are read by this warp only: drop
  // them from L2 rather than let the next layer's stream write them back
  __syncwarp();
  for (int i = lane; i < 4 * ns; i += 32)
    discard_l2_line(p.opart + (r0 + static_cast<size_t>(i / 4) * p.rows) * HD + (i % 4) * 32);
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
// The next work item, decoded once by the producer (b < 0: the queue is empty).
__device__ __forceinline__ bool next_item(uint32_t it_full, uint32_t it_empty, const Item* s_items, Ring& r,
                                          unsigned* status, Item& it) {
  if (!mbar_wait(it_full + 8 * r.idx, r.phase, status)) return false;
  it = s_items[r.idx];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(it_empty + 8 * r.idx);
  r.next(kItemRing);
  return it.b >= 0;
}

// Sum over the warp's 32 lanes of each v[j] (N = 16 or 32 values); lane i
// returns the sum of v[i % N].  Exchange rounds halve the values a lane keeps
// (for N = 16 the two half-warps are added first).
template <int N>
__device__ __forceinline__ float warp_reduce_scatter_sum(float (&v)[N], int lane) {
  if (N == 16) {
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 16);
  }
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = upper ? v[j] : v[j + w];
      const float keep = upper ? v[j + w] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// Maximum of N values by a tree of pairwise maxima.
template <int N>
__device__ __forceinline__ float array_max(const float (&v)[N]) {
  float t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) t[i] = fmaxf(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  return t[0];
}

// N (16 or 32) columns of this warp's lane quarter as floats.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&d)[N]) {
  uint32_t r[N];
  if constexpr (N == 16) tmem_ld_16cols(taddr, r);
  else tmem_ld_32cols(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < N; ++j) d[j] = __uint_as_float(r[j]);
}

// RMSNorm * gain and RoPE of one row of head vectors held in shared memory as
// two K-major boxes with the 128-byte swizzle (elements 0..63 and 64..127,
// box_stride bytes apart; row r at r * 128, its 16-byte chunk c at chunk
// c ^ (r & 7)), rewritten in place as bf16.  Sixteen consecutive lanes share
// the row: lane part k owns elements 4k .. 4k+3 and their rotation partners
// 64+4k .. 64+4k+3.  cv, sv: the part's four cos and sin at the row's
// position; g: its gains (elements, then partners) as bf16 pairs.  Every lane
// of the warp calls it; only active lanes store.
__device__ __forceinline__ void norm_rope_row_smem(uint32_t box0, uint32_t box_stride, int r, int k,
                                                   const float (&cv)[4], const float (&sv)[4], const uint2 gx,
                                                   const uint2 gy, float eps, bool active) {
  const uint32_t a = box0 + static_cast<uint32_t>(r) * 128u + 16u * static_cast<uint32_t>((k >> 1) ^ (r & 7)) +
                     8u * static_cast<uint32_t>(k & 1);
  const uint2 xr = ld_shared_v2(a), yr = ld_shared_v2(a + box_stride);
  const float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};
  const float y[4] = {bf16_lo(yr.x), bf16_hi(yr.x), bf16_lo(yr.y), bf16_hi(yr.y)};
  const float g0[4] = {bf16_lo(gx.x), bf16_hi(gx.x), bf16_lo(gx.y), bf16_hi(gx.y)};
  const float g1[4] = {bf16_lo(gy.x), bf16_hi(gy.x), bf16_lo(gy.y), bf16_hi(gy.y)};
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss = fmaf(y[i], y[i], fmaf(x[i], x[i], ss));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rn = rsqrtf(ss * (1.0f / HD) + eps);
  float ox[4], oy[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float xs = x[i] * (rn * g0[i]);
    const float ys = y[i] * (rn * g1[i]);
    ox[i] = xs * cv[i] - ys * sv[i];
    oy[i] = ys * cv[i] + xs * sv[i];
  }
  if (active) {
    st_shared_v2(a, make_uint2(pack_bf16x2(ox[0], ox[1]), pack_bf16x2(ox[2], ox[3])));
    st_shared_v2(a + box_stride, make_uint2(pack_bf16x2(oy[0], oy[1]), pack_bf16x2(oy[2], oy[3])));
  }
}

// One work item's query rows (row h * bs + j of the pair: query head h of the
// KV head at block position j) and, when with_keys, the block's keys (row j),
// normalised and rotated in place by 128 threads: thread t takes positions
// j = t / 16 (+ 8, ...) and part k = t % 16, so the sin and cos of a
// (position, frequency) serve all G heads and the key at that position.
__device__ __forceinline__ void prep_item_rows(uint32_t qbox0, uint32_t qbox_stride, bool with_keys, uint32_t kbox0,
                                               int G, int bs,
                                               int pos0, const unsigned long long* inv, const uint2 (&gq)[2],
                                               const uint2 (&gk)[2], float eps, int t) {
  const int k = t & 15;
  for (int jb = 0; jb < bs; jb += 8) {  // uniform over the 128 threads
    const int j = jb + (t >> 4);
    const bool active = j < bs;
    float cv[4], sv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rope_sincos(pos0 + j, inv[4 * k + i], &sv[i], &cv[i]);
    for (int h = 0; h < G; ++h)
      norm_rope_row_smem(qbox0, qbox_stride, active ? h * bs + j : 0, k, cv, sv, gq[0], gq[1], eps, active);
    if (with_keys) norm_rope_row_smem(kbox0, kBlkBoxBytes, active ? j : 0, k, cv, sv, gk[0], gk[1], eps, active);
  }
}

// Roles (c = NC/2 query rows per softmax warp):
//   warps 0 .. 7       softmax: warp w owns key (lane) 32*(w%4) + lane of every
//                      tile and query rows c*(w/4) .. +c-1
//   warps 8 .. 11      epilogue: O^T lanes (dims) of lane quarter w%4; before
//                      that, one item ahead, RMSNorm * gain and RoPE of the
//                      item's query rows (and block keys) in shared memory
//   warp 12            TMA producer (work queue, raw Q and block keys, K ring, V ring)
//   warp 13            S^T = K Q^T issuer; allocates tensor memory
//   warp 14            O^T += V^T P^T issuer
template <int NC>
__global__ void __launch_bounds__(TcCfg<NC>::kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnMaps maps,
                                                                         const __grid_constant__ AttnParams p,
                                                                         const TcLayout lay) {
  using C = TcCfg<NC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int NK = lay.nk, NV = lay.nv;
  const uint32_t bar0 = base + lay.off_bar;
  const uint32_t k_full = bar0, k_empty = k_full + 8 * kMaxRing;
  const uint32_t v_full = k_empty + 8 * kMaxRing, v_empty = v_full + 8 * kMaxRing;
  const uint32_t q_full = v_empty + 8 * kMaxRing, q_empty = q_full + 16;
  const uint32_t s_full = q_empty + 16, s_empty = s_full + 8 * kSBufs;
  const uint32_t p_full = s_empty + 8 * kSBufs, p_empty = p_full + 16;
  const uint32_t o_full = p_empty + 16, o_free = o_full + 16;
  const uint32_t ml_full = o_free + 16, ml_empty = ml_full + 16;
  const uint32_t it_full = ml_empty + 16, it_empty = it_full + 8 * kItemRing;
  const uint32_t red_bar = it_empty + 8 * kItemRing;  // one per column half
  const uint32_t qraw_full = red_bar + 16;             // per Q buffer: the raw rows landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + lay.off_misc);
  unsigned long long* s_inv = reinterpret_cast<unsigned long long*>(gbase + lay.off_misc + 64);  // [64]
  __nv_bfloat16* s_gain = reinterpret_cast<__nv_bfloat16*>(gbase + lay.off_misc + 576);          // [2][128]
  float* s_m = reinterpret_cast<float*>(gbase + lay.off_misc + 1088);             // [2][NC]
  float* s_l = s_m + 2 * NC;                                                       // [2][4][NC]
  float* s_red = s_l + 2 * 4 * NC;                                                 // [2 halves][2][4][32]
  int* s_prefix = reinterpret_cast<int*>(s_red + 2 * 2 * 4 * 32);
  int* s_n = s_prefix + (p.B + 1);
  int* s_multi = s_n + p.B;                                                        // [B+1]
  Item* s_items = reinterpret_cast<Item*>(s_multi + p.B + 1);                              // kItemRing entries

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_empty + 8 * s, 1);
      mbar_init(v_full + 8 * s, 1);
      mbar_init(v_empty + 8 * s, 1);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(s_full + 8 * s, 1);
      mbar_init(s_empty + 8 * s, C::kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + 8 * i, 4);   // the four epilogue warps, after normalising and rotating in place
      mbar_init(q_empty + 8 * i, 1);
      mbar_init(qraw_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, C::kSoftWarps);
      mbar_init(p_empty + 8 * i, 1);
      mbar_init(o_full + 8 * i, 1);
      mbar_init(o_free + 8 * i, 4);
      mbar_init(ml_full + 8 * i, C::kSoftWarps);
      mbar_init(ml_empty + 8 * i, 4);
    }
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(it_full + 8 * i, 1);
      mbar_init(it_empty + 8 * i, 2 + C::kSoftWarps + 4);
    }
    for (int i = 0; i < 2; ++i) mbar_init(red_bar + 8 * i, 4);
    mbar_fence_init();
  }
  if (warp == C::kSWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp >= C::kEpiWarp0 && warp < C::kEpiWarp0 + 4) {  // the norm gains and RoPE frequencies
    const int et = threadIdx.x - 32 * C::kEpiWarp0;
    s_gain[et] = p.qg ? p.qg[et] : __float2bfloat16_rn(1.f);
    s_gain[HD + et] = p.kg ? p.kg[et] : __float2bfloat16_rn(1.f);
    if (et < HD / 2) s_inv[et] = p.inv.v[et];
  }
  if (warp == C::kProdWarp) {  // per-sequence lengths and the prefix of full (non-last) splits
    int carry = 0, mcarry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {  // a warp scan per 32 sequences
      const int b = b0 + lane;
      int cnt = 0;
      if (b < p.B) {
        const int n = cached_rows(p.seq_len[b], p.cap, p.ring, p.status);
        s_n[b] = n;
        const int first = p.window > 0 ? max(0, n - p.window) : 0;
        cnt = (n_splits(n - first, p.chunk) - 1) * p.Hkv;
      }
      const unsigned mb = __ballot_sync(0xffffffffu, cnt > 0);  // sequences of several splits
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      if (b < p.B) {
        s_prefix[b] = carry + inc - cnt;
        s_multi[b] = mcarry + __popc(mb & ((1u << lane) - 1u));
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
      mcarry += __popc(mb);
    }
    if (lane == 0) {
      s_prefix[p.B] = carry;
      s_multi[p.B] = mcarry;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int n_items = s_prefix[p.B] + p.B * p.Hkv;

  if (warp == C::kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.q);
      const uint64_t pol = l2_policy_evict_first();
      Ring kr, vr, q, itr;
      bool ok = true;
      // The first work item of each CTA is its own index: it needs no queue,
      // so it starts before the counters are known to be cleared.
      int w = static_cast<int>(blockIdx.x);
      bool waited = false;
      while (ok) {
        if (w < 0) {
          if (!waited) {
            pdl_wait_primary();  // the cleared counters
            // Release the combine kernel only now: it trusts the per-pair
            // counters, cleared by the preceding grid.
            pdl_launch_dependents();
            waited = true;
          }
          w = static_cast<int>(gridDim.x) + atomicAdd(p.counters, 1);
        }
        Item it;
        it.b = -1;
        if (w < n_items) it = decode_item(w, s_prefix, s_n, s_multi, p);
        if (!(ok = mbar_wait(it_empty + 8 * itr.idx, itr.phase ^ 1u, p.status))) break;
        s_items[itr.idx] = it;  // decoded once here, read by every role
        mbar_arrive(it_full + 8 * itr.idx);
        itr.next(kItemRing);
        if (w >= n_items) break;
        w = -1;
        // the pair's raw query rows (and, for the last split, the block's raw
        // keys): the epilogue warps normalise and rotate them in place
        if (!(ok = mbar_wait(q_empty + 8 * q.idx, q.phase ^ 1u, p.status))) break;
        const int qrow = (it.b * p.Hq + it.g * p.G) * p.bs;
        const int brow = (it.b * p.Hkv + it.g) * p.bs;
        const uint32_t qdst = base + lay.off_q + q.idx * 2 * C::kQBoxBytes;
        const uint32_t kbdst = base + lay.off_kb + q.idx * 2 * kBlkBoxBytes;
        mbar_arrive_expect_tx(qraw_full + 8 * q.idx, 2 * C::kQBoxBytes + (it.last ? 2 * kBlkBoxBytes : 0));
        tma_load_2d(qdst, &maps.q, qraw_full + 8 * q.idx, 0, qrow);
        tma_load_2d(qdst + C::kQBoxBytes, &maps.q, qraw_full + 8 * q.idx, 64, qrow);
        if (it.last) {
          tma_load_2d(kbdst, &maps.kb, qraw_full + 8 * q.idx, 0, brow);
          tma_load_2d(kbdst + kBlkBoxBytes, &maps.kb, qraw_full + 8 * q.idx, 64, brow);
        }
        q.next(2);
        // paged: the block-table entry of the next tile is requested one tile
        // ahead, so its latency hides behind this tile's ring waits (a key
        // tile never crosses a page: pages are multiples of 128 rows and tiles
        // start at multiples of 128).  An entry outside the pool gives a row
        // outside the tensor map, which TMA fills with zeros.
        const int32_t* trow = p.table ? p.table + static_cast<size_t>(it.b) * p.max_pages : nullptr;
        int page = (trow && it.ntiles > 0) ? __ldg(trow + it.kstart / p.page_size) : 0;
        for (int t = 0; t < it.nt && ok; ++t) {
          const bool blk = t >= it.ntiles;
          const uint32_t bytes = blk ? 2 * kBlockBoxRows * 128 : kHalfBytes;
          const int pos = it.kstart + t * kKeys;
          int next_page = page;
          if (trow && t + 1 < it.ntiles && (pos + kKeys) / p.page_size != pos / p.page_size)
            next_page = __ldg(trow + (pos + kKeys) / p.page_size);
          int y = 0;
          if (!blk) {
            if (trow && (page < 0 || page >= p.num_pages)) {
              raise_status(p.status, DFLASH_DEV_BAD_SEQLEN);
              y = -kKeys;  // wholly outside the map: the tile reads zeros
            } else {
              y = static_cast<int>(cache_row(p, it.b, it.g, pos, page));
            }
          }
          page = next_page;
          if (!blk) {  // the block's keys are not in the ring: the S product reads them from their own buffer
            if (!(ok = mbar_wait(k_empty + 8 * kr.idx, kr.phase ^ 1u, p.status))) break;
            const uint32_t kdst = base + lay.off_k + kr.idx * kHalfBytes;
            mbar_arrive_expect_tx(k_full + 8 * kr.idx, bytes);
            tma_load_2d_hint(kdst, &maps.k, k_full + 8 * kr.idx, 0, y, pol);
            tma_load_2d_hint(kdst + kBoxBytes, &maps.k, k_full + 8 * kr.idx, 64, y, pol);
            kr.next(NK);
          }
          if (!(ok = mbar_wait(v_empty + 8 * vr.idx, vr.phase ^ 1u, p.status))) break;
          const uint32_t vdst = base + lay.off_v + vr.idx * kHalfBytes;
          mbar_arrive_expect_tx(v_full + 8 * vr.idx, bytes);
          if (!blk) {
            tma_load_2d_hint(vdst, &maps.v, v_full + 8 * vr.idx, 0, y, pol);
            tma_load_2d_hint(vdst + kBoxBytes, &maps.v, v_full + 8 * vr.idx, 64, y, pol);
          } else {
            tma_load_2d(vdst, &maps.vb, v_full + 8 * vr.idx, 0, brow);
            tma_load_2d(vdst + kBoxBytes, &maps.vb, v_full + 8 * vr.idx, 64, brow);
          }
          vr.next(NV);
        }
      }
    }
  } else if (warp == C::kSWarp) {
    // ------------------------------------------------ S^T = K Q^T issuer
    if (lane == 0) {
      Ring kr, q, sq, itr;
      bool ok = true;
      while (ok) {
        if (!(ok = mbar_wait(it_full + 8 * itr.idx, itr.phase, p.status))) break;
        const Item it = s_items[itr.idx];
        mbar_arrive(it_empty + 8 * itr.idx);
        itr.next(kItemRing);
        if (it.b < 0) break;
        if (!(ok = mbar_wait(q_full + 8 * q.idx, q.phase, p.status))) break;
        const uint32_t qb = base + lay.off_q + q.idx * 2 * C::kQBoxBytes;
        for (int t = 0; t < it.nt && ok; ++t) {
          const bool blk = t >= it.ntiles;  // the block's keys: their own buffer, ready with Q
          if (!blk && !(ok = mbar_wait(k_full + 8 * kr.idx, kr.phase, p.status))) break;
          if (!(ok = mbar_wait(s_empty + 8 * sq.idx, sq.phase ^ 1u, p.status))) break;
          tc_fence_after_sync();
          const uint32_t kb = blk ? base + lay.off_kb + q.idx * 2 * kBlkBoxBytes : base + lay.off_k + kr.idx * kHalfBytes;
          const uint32_t kbox = blk ? kBlkBoxBytes : kBoxBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_desc_kmajor_sw128(kb + (kk >> 2) * kbox) + 2 * (kk & 3);
            const uint64_t bd = umma_desc_kmajor_sw128(qb + (kk >> 2) * C::kQBoxBytes) + 2 * (kk & 3);
            umma_bf16(tmem + C::kColS + NC * sq.idx, ad, bd, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full + 8 * sq.idx);
          if (!blk) {
            umma_commit(k_empty + 8 * kr.idx);
            kr.next(NK);
          }
          sq.next(kSBufs);
        }
        if (!ok) break;
        umma_commit(q_empty + 8 * q.idx);
        q.next(2);
      }
    }
  } else if (warp == C::kOWarp) {
    // ------------------------------------------------ O^T += V^T P^T issuer
    if (lane == 0) {
      Ring vr, pr, o, itr;
      bool ok = true;
      while (ok) {
        if (!(ok = mbar_wait(it_full + 8 * itr.idx, itr.phase, p.status))) break;
        const Item it = s_items[itr.idx];
        mbar_arrive(it_empty + 8 * itr.idx);
        itr.next(kItemRing);
        if (it.b < 0) break;
        const uint32_t od = tmem + C::kColO + 2 * NC * o.idx;
        for (int t = 0; t < it.nt && ok; ++t) {
          if (!(ok = mbar_wait(p_full + 8 * pr.idx, pr.phase, p.status))) break;
          if (t == 0 && !(ok = mbar_wait(o_free + 8 * o.idx, o.phase ^ 1u, p.status))) break;
          if (!(ok = mbar_wait(v_full + 8 * vr.idx, vr.phase, p.status))) break;
          tc_fence_after_sync();
          const int nsteps = (tile_keys(it, t, p.bs) + 15) / 16;
          // A = V^T: two 64-dim blocks 16 KB apart, 8-key groups 1 KB apart;
          // B = P^T: NC = 32 one 64-value block, NC = 64 two (hi, lo) 16 KB apart
          const uint64_t vd = umma_desc_mnmajor(base + lay.off_v + vr.idx * kHalfBytes, kBoxBytes, 1024, 2u);
          const uint64_t pd = umma_desc_mnmajor(base + lay.off_p + pr.idx * C::kPBytes, 16384, 1024, 2u);
#pragma unroll
          for (int j = 0; j < 8; ++j)  // one step = 16 keys = 2 KB of V^T and of P^T
            if (j < nsteps) umma_bf16(od, vd + 128 * j, pd + 128 * j, C::kIdescO, (t > 0 || j > 0) ? 1u : 0u);
          umma_commit(p_empty + 8 * pr.idx);
          umma_commit(v_empty + 8 * vr.idx);
          pr.next(2);
          vr.next(NV);
        }
        if (!ok) break;
        umma_commit(o_full + 8 * o.idx);
        o.next(2);
      }
    }
  } else if (warp < C::kSoftWarps) {
    // ------------------------------------------------ softmax
    constexpr int CW = C::kCPW;
    const int qd = warp & 3;                 // lane quarter
    const int hc = warp >> 2;                // column group: query rows CW*hc .. +CW-1
    const int key = 32 * qd + lane;          // this thread's key of every tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const float scale = p.scale_log2;
    // this key's P^T values in a P buffer: 128-byte rows, the 16-byte chunk c of
    // a row stored at chunk c ^ (key & 7)
    const uint32_t prow = key * 128;
    // The four warps of a column group agree on the running max of a work item
    // through one mbarrier (bounded waits) on its first tile; the exchange
    // slots alternate by phase.
    const uint32_t rbar = red_bar + 8 * hc;
    uint32_t rph = 0;
    Ring sr, vr, mlr, itr;
    int pb = 0;
    int pcnt[2] = {0, 0};
    bool ok = true;
    while (ok) {
      Item it;
      if (!next_item(it_full, it_empty, s_items, itr, p.status, it)) break;
      float m[CW], l[CW];
      float dmax = -INFINITY;  // largest score above m over the item's later tiles
      for (int t = 0; t < it.nt; ++t) {
        if (!(ok = mbar_wait(s_full + 8 * sr.idx, sr.phase, p.status))) break;
        tc_fence_after_sync();
        float d[CW];
        tmem_ld_cols<CW>(tl + C::kColS + NC * sr.idx + CW * hc, d);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty + 8 * sr.idx);
        sr.next(kSBufs);
        const int nvalid = tile_keys(it, t, p.bs);
        const bool valid = key < nvalid;
        const int live_cols = valid ? min(CW, p.rows - CW * hc) : 0;  // query rows this key scores
        if (t == 0) {
          // the running max of each row: the maximum over the item's first tile
#pragma unroll
          for (int j = 0; j < CW; ++j) d[j] = j < live_cols ? d[j] * scale : -INFINITY;
          float* red = s_red + (hc * 2 + static_cast<int>(rph)) * 128;
#pragma unroll
          for (int j = 0; j < CW; ++j) m[j] = warp_max_redux(d[j]);
          if (lane == 0) {
#pragma unroll
            for (int j4 = 0; j4 < CW / 4; ++j4)
              reinterpret_cast<float4*>(red + 32 * qd)[j4] =
                  make_float4(m[4 * j4], m[4 * j4 + 1], m[4 * j4 + 2], m[4 * j4 + 3]);
            mbar_arrive(rbar);
          }
          if (!(ok = mbar_wait(rbar, rph, p.status))) break;
          rph ^= 1u;
#pragma unroll
          for (int j4 = 0; j4 < CW / 4; ++j4) {
            const float4 a0 = reinterpret_cast<const float4*>(red)[j4];
            const float4 a1 = reinterpret_cast<const float4*>(red + 32)[j4];
            const float4 a2 = reinterpret_cast<const float4*>(red + 64)[j4];
            const float4 a3 = reinterpret_cast<const float4*>(red + 96)[j4];
            m[4 * j4] = fmax3(fmax3(a0.x, a1.x, a2.x), a3.x, -INFINITY);
            m[4 * j4 + 1] = fmax3(fmax3(a0.y, a1.y, a2.y), a3.y, -INFINITY);
            m[4 * j4 + 2] = fmax3(fmax3(a0.z, a1.z, a2.z), a3.z, -INFINITY);
            m[4 * j4 + 3] = fmax3(fmax3(a0.w, a1.w, a2.w), a3.w, -INFINITY);
          }
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            d[j] = j < live_cols ? d[j] - m[j] : -INFINITY;
            l[j] = 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < CW; ++j) d[j] = j < live_cols ? fmaf(d[j], scale, -m[j]) : -INFINITY;
          dmax = fmaxf(dmax, array_max<CW>(d));
        }
        // P^T of this key: bf16 hi (truncated) and lo (the truncated rest);
        // hi + lo is within 2^-14 of P, below it
        uint32_t hv[CW / 2], lv[CW / 2];
#pragma unroll
        for (int i = 0; i < CW / 2; ++i) {
          const float a = ex2_approx(d[2 * i]);
          const float c2 = ex2_approx(d[2 * i + 1]);
          l[2 * i] += a;
          l[2 * i + 1] += c2;
          const uint32_t ua = __float_as_uint(a), uc = __float_as_uint(c2);
          hv[i] = __byte_perm(ua, uc, 0x7632);
          lv[i] = __byte_perm(__float_as_uint(a - __uint_as_float(ua & 0xFFFF0000u)),
                              __float_as_uint(c2 - __uint_as_float(uc & 0xFFFF0000u)), 0x7632);
        }
        // the O^T product reads V rows up to the next multiple of 16 keys: zero
        // the rows past the end of the data, whatever the tile holds there
        const bool zero_row = !valid && key < ((nvalid + 15) & ~15);
        if (__any_sync(0xffffffffu, zero_row)) {
          if (!(ok = mbar_wait(v_full + 8 * vr.idx, vr.phase, p.status))) break;
          if (zero_row && hc == 0) {
            const uint32_t vst = base + lay.off_v + vr.idx * kHalfBytes;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              st_shared_v4(vst + key * 128 + 16 * c, z);
              st_shared_v4(vst + kBoxBytes + key * 128 + 16 * c, z);
            }
          }
        }
        vr.next(NV);
        if (pcnt[pb] > 0 && !(ok = mbar_wait(p_empty + 8 * pb, (pcnt[pb] - 1) & 1, p.status))) break;
        const uint32_t ph = base + lay.off_p + pb * C::kPBytes + prow;
#pragma unroll
        for (int c = 0; c < CW / 8; ++c) {
          const int chi = (CW / 8) * hc + c;            // chunk of the hi values in the row
          const int clo = NC == 32 ? 4 + chi : chi;     // NC = 32: lo in the same row
          const uint32_t lo_base = NC == 32 ? 0u : C::kPLoOffset;
          st_shared_v4(ph + 16 * (chi ^ (key & 7)), make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]));
          st_shared_v4(ph + lo_base + 16 * (clo ^ (key & 7)),
                       make_uint4(lv[4 * c], lv[4 * c + 1], lv[4 * c + 2], lv[4 * c + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 8 * pb);
        ++pcnt[pb];
        pb ^= 1;
      }
      if (!ok) break;
      // a score beyond 2^64 above the running max: the combine kernel redoes
      // this (sequence, KV head) exactly
      if (__any_sync(0xffffffffu, dmax > kOverflowLog2) && lane == 0) {
        pdl_wait_primary();  // the cleared flags (the first work item may run ahead of the clearing)
        atomicOr(p.counters + 1 + it.b * p.Hkv + it.g, 1);
      }
      // row sums over this warp's keys -> the epilogue; the quarter-0 warps also
      // hand over the running max
      if (!(ok = mbar_wait(ml_empty + 8 * mlr.idx, mlr.phase ^ 1u, p.status))) break;
      if (qd == 0 && lane == 0) {
#pragma unroll
        for (int j4 = 0; j4 < CW / 4; ++j4)
          reinterpret_cast<float4*>(s_m + mlr.idx * NC + CW * hc)[j4] =
              make_float4(m[4 * j4], m[4 * j4 + 1], m[4 * j4 + 2], m[4 * j4 + 3]);
      }
      const float lsum = warp_reduce_scatter_sum<CW>(l, lane);   // lane i: column i % CW
      if (lane < CW) s_l[(mlr.idx * 4 + qd) * NC + CW * hc + lane] = lsum;
      __syncwarp();
      if (lane == 0) mbar_arrive(ml_full + 8 * mlr.idx);
      mlr.next(2);
    }
  } else {
    // ------------------------------------------------ epilogue
    // One item ahead of its epilogue, each work item's query rows (and, for a
    // last split, the block's keys), loaded raw by the producer, get their
    // RMSNorm * gain and RoPE in place in shared memory: Q of item i is made
    // before the epilogue of item i - 1.
    const int qd = warp & 3;
    const int dim = 32 * qd + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const int et = threadIdx.x - 32 * C::kEpiWarp0;  // 0 .. 127
    // this thread's gains for its part of every head vector (elements 4k .. 4k+3, partners 64+4k ..)
    const int gpart = 4 * (et & 15);
    const uint2 gq[2] = {*reinterpret_cast<const uint2*>(s_gain + gpart),
                         *reinterpret_cast<const uint2*>(s_gain + 64 + gpart)};
    const uint2 gk[2] = {*reinterpret_cast<const uint2*>(s_gain + HD + gpart),
                         *reinterpret_cast<const uint2*>(s_gain + HD + 64 + gpart)};
    Ring orr, mlr, itr, qq;
    bool ok = true, waited = false, have_prev = false;
    Item prev;
    while (ok) {
      Item it;
      const bool got = next_item(it_full, it_empty, s_items, itr, p.status, it);
      if (got) {
        if (!(ok = mbar_wait(qraw_full + 8 * qq.idx, qq.phase, p.status))) break;
        const int n_in = p.seq_len[it.b];
        // the block's positions follow the sequence: its length (a ring
        // cache's may exceed the capacity), else the cached rows
        const int pos0 = p.ring ? max(n_in, 0) : min(max(n_in, 0), p.cap);
        prep_item_rows(base + lay.off_q + qq.idx * 2 * C::kQBoxBytes, C::kQBoxBytes, it.last,
                       base + lay.off_kb + qq.idx * 2 * kBlkBoxBytes, p.G, p.bs, pos0, s_inv, gq, gk, p.eps, et);
        fence_proxy_async_smem();  // the rows, for the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full + 8 * qq.idx);
        qq.next(2);
      }
      if (have_prev) {
        if (!(ok = mbar_wait(o_full + 8 * orr.idx, orr.phase, p.status))) break;
        tc_fence_after_sync();
        float o[NC];  // O^T lane `dim`: the hi and lo column blocks added
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) {
          uint32_t rh[32], rl[32];
          tmem_ld_32cols(tl + C::kColO + 2 * NC * orr.idx + 32 * c, rh);
          tmem_ld_32cols(tl + C::kColO + 2 * NC * orr.idx + NC + 32 * c, rl);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[32 * c + j] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free + 8 * orr.idx);
        orr.next(2);
        if (!(ok = mbar_wait(ml_full + 8 * mlr.idx, mlr.phase, p.status))) break;
        // lane i: the sum and its reciprocal for rows i and 32 + i
        const float* lrow = s_l + mlr.idx * 4 * NC;
        float den[NC / 32], inv[NC / 32];
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) {
          const int r = 32 * c + lane;
          den[c] = lrow[r] + lrow[NC + r] + lrow[2 * NC + r] + lrow[3 * NC + r];
          inv[c] = r < p.rows ? 1.f / den[c] : 0.f;
        }
        if (prev.nsplit == 1) {
          const size_t row0 = (static_cast<size_t>(prev.b) * p.Hq + prev.g * p.G) * p.bs;
#pragma unroll
          for (int r = 0; r < NC; ++r) {
            const float iv = __shfl_sync(0xffffffffu, inv[r / 32], r % 32);
            if (r < p.rows) p.out[(row0 + r) * HD + dim] = __float2bfloat16_rn(o[r] * iv);
          }
        } else {
          const size_t r0 = ((static_cast<size_t>(prev.b) * p.Hkv + prev.g) * p.max_splits + prev.s) * p.rows;
#pragma unroll
          for (int r = 0; r < NC; ++r) {
            const float iv = __shfl_sync(0xffffffffu, inv[r / 32], r % 32);
            if (r < p.rows) p.opart[(r0 + r) * HD + dim] = o[r] * iv;
          }
          if (qd == 0) {
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) {
              const int r = 32 * c + lane;
              if (r < p.rows) p.mlpart[r0 + r] = make_float2(s_m[mlr.idx * NC + r], den[c]);
            }
          }
        }
        __threadfence();  // this warp's output / partial before the pair's completion count
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(ml_empty + 8 * mlr.idx);
          if (!waited) {
            pdl_wait_primary();  // the cleared pair counts (the first item may run ahead of the clearing)
            waited = true;
          }
          atomicAdd(p.counters + 1 + p.B * p.Hkv + prev.b * p.Hkv + prev.g, 1);
        }
        mlr.next(2);
      }
      if (!got) break;
      prev = it;
      have_prev = true;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::kSWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
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


// Keys per split: aims at ~800 work items for a full cache (about five per
// SM; a cache filled to about half its capacity then gives about three).
// Longer splits amortise each split's partial output (written, then merged by
// the combine kernel) and its pipeline ramp; enough items remain for the
// dynamic queue to balance the SMs.  A split is at least ~1024 keys (a
// work item costs about as much as a few tiles on top of its keys) unless
// that would leave fewer items than the 152 SMs of a GB300.
int pick_chunk(int B, int Hkv, int cap, int window) {
  const long keys = window > 0 ? std::min(window, cap) : cap;
  const long total = static_cast<long>(B) * Hkv * keys;
  long c = total / 800;
  const long lo = std::min<long>(1024, std::max<long>(256, total / 152));
  c = std::max(c, lo);
  c = (c + kKeys - 1) / kKeys * kKeys;
  return static_cast<int>(std::min<long>(4096, std::max<long>(256, c)));
}

}  // namespace

size_t attn_ws_bytes(int B, int bs, int Hq, int Hkv, int cap, int window, dflash_dtype dt) {
  const size_t esz = dt == DFLASH_BF16 ? 2 : 4;
  const int rows = (Hq / Hkv) * bs;
  const int chunk = pick_chunk(B, Hkv, cap, window);
  const int keys = window > 0 ? std::min(window, cap) : cap;
  const int max_splits = n_splits(keys, chunk);
  size_t s = 0;
  if (dt != DFLASH_BF16)  // the fp32 prologue's q^ and k^_b (the bf16 path makes them in shared memory)
    s += align256(static_cast<size_t>(B) * Hq * bs * HD * esz) + align256(static_cast<size_t>(B) * Hkv * bs * HD * esz);
  else
    s += align256(static_cast<size_t>(B) * Hkv * max_splits * rows * HD * sizeof(float)) +
         align256(static_cast<size_t>(B) * Hkv * max_splits * rows * sizeof(float2)) +
         align256((1 + 2 * static_cast<size_t>(B) * Hkv) * sizeof(int));
  return s + 256;
}

dflash_status launch_block_attn(int layer, int B, int bs, int Hq, const void* q, const void* kb,
                                const void* vb, const void* qg, const void* kg, float theta,
                                float eps, const dflash_kv_cache& c, int window, void* out, void* ws,
                                cudaStream_t st, const DeviceInfo& dev) {
  const int Hkv = c.num_kv_heads;
  const int G = Hq / Hkv;
  InvFreq inv;
  for (int e = 0; e < HD / 2; ++e) {
    const long double f = std::pow(static_cast<double>(theta), -2.0 * e / HD);  // inverse frequency, as the fp64 one
    inv.v[e] = static_cast<unsigned long long>(std::llroundl(f * 0x1p64L / (2.0L * 3.14159265358979323846264338327950288L)) );
  }
  WsCarver w(ws);
  const float scale = 1.0f / std::sqrt(static_cast<float>(HD));
  if (c.dtype == DFLASH_F32) {
    float* qh = w.take<float>(static_cast<size_t>(B) * Hq * bs * HD);
    float* kbh = w.take<float>(static_cast<size_t>(B) * Hkv * bs * HD);
    attn_prologue_kernel<float><<<B * bs, kPrologueThreads, 0, st>>>(
        static_cast<const float*>(q), static_cast<const float*>(kb), static_cast<const float*>(qg),
        static_cast<const float*>(kg), c.seq_len, B, bs, Hq, Hkv, c.capacity, c.ring, eps, inv, qh, kbh, nullptr, 0,
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
  p.ring = c.ring;
  p.layer = layer;
  p.window = window;
  p.chunk = pick_chunk(B, Hkv, c.capacity, window);
  const int keys = window > 0 ? std::min(window, c.capacity) : c.capacity;
  p.max_splits = n_splits(keys, p.chunk);
  p.rows = G * bs;
  p.seq_len = c.seq_len;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kb = static_cast<const __nv_bfloat16*>(kb);
  p.qg = static_cast<const __nv_bfloat16*>(qg);
  p.kg = static_cast<const __nv_bfloat16*>(kg);
  p.eps = eps;
  p.inv = inv;
  p.vb = static_cast<const __nv_bfloat16*>(vb);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.opart = w.take<float>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows * HD);
  p.mlpart = w.take<float2>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows);
  p.counters = w.take<int>(1 + 2 * static_cast<size_t>(B) * Hkv);
  p.ck = static_cast<const __nv_bfloat16*>(c.k);
  p.cv = static_cast<const __nv_bfloat16*>(c.v);
  p.table = c.block_table;
  p.max_pages = c.max_pages;
  p.page_size = c.page_size;
  p.num_pages = c.num_pages;
  p.scale_log2 = 1.4426950408889634f * scale;
  p.status = dev.status;
  p.wait_limit_ns = kWaitLimitNs;

  const int nc = p.rows > 32 ? 64 : 32;   // query rows padded to the MMA's N
  AttnMaps maps;
  const uint64_t rows = c.block_table ? static_cast<uint64_t>(c.num_layers) * c.num_pages * Hkv * c.page_size
                                      : static_cast<uint64_t>(c.num_layers) * c.batch * Hkv * c.capacity;
  dflash_status s = make_tmap_bf16_2d(&maps.k, c.k, rows, HD, kKeys, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.v, c.v, rows, HD, kKeys, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.q, q, static_cast<uint64_t>(B) * Hq * bs, HD, nc, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.kb, kb, static_cast<uint64_t>(B) * Hkv * bs, HD, kBlockBoxRows, 64);
  if (!s) s = make_tmap_bf16_2d(&maps.vb, vb, static_cast<uint64_t>(B) * Hkv * bs, HD, kBlockBoxRows, 64);
  if (s) return s;

  {  // one CTA clears the counters; the main kernel's first items run meanwhile
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(1);
    pc.blockDim = dim3(1024);
    pc.stream = st;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    cudaError_t le = cudaLaunchKernelEx(&pc, attn_clear_kernel, p.counters, 1 + 2 * B * Hkv,
                                        static_cast<const uint8_t*>(q), static_cast<size_t>(B) * Hq * bs * HD * 2,
                                        static_cast<const uint8_t*>(kb), static_cast<size_t>(B) * Hkv * bs * HD * 2);
    if (le != cudaSuccess) return cuda_fail(le, "attn_clear_kernel launch");
  }

  const TcLayout lay = tc_layout(nc, B, static_cast<int>(dev.max_smem_optin));
  if (lay.nk < 1 || lay.nv < 1 || lay.bytes > static_cast<int>(dev.max_smem_optin))
    return fail(DFLASH_ERR_UNSUPPORTED, "block_attn: shared memory");
  const long upper = static_cast<long>(B) * Hkv * p.max_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<long>(upper, dev.num_sms)));
  cfg.dynamicSmemBytes = static_cast<size_t>(lay.bytes);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t le;
  if (nc == 32) {
    dflash_status ss = smem_limit_once<attn_tc_kernel<32>>(dev.device, static_cast<int>(dev.max_smem_optin),
                                                           "cudaFuncSetAttribute(attn_tc_kernel)");
    if (ss) return ss;
    cfg.blockDim = dim3(TcCfg<32>::kThreads);
    le = cudaLaunchKernelEx(&cfg, attn_tc_kernel<32>, maps, p, lay);
  } else {
    dflash_status ss = smem_limit_once<attn_tc_kernel<64>>(dev.device, static_cast<int>(dev.max_smem_optin),
                                                           "cudaFuncSetAttribute(attn_tc_kernel)");
    if (ss) return ss;
    cfg.blockDim = dim3(TcCfg<64>::kThreads);
    le = cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, maps, p, lay);
  }
  if (le != cudaSuccess) return cuda_fail(le, "attn_tc_kernel launch");
  {  // always: it also redoes flagged (sequence, KV head) pairs
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

// Test hook for the bounded waits: the combine kernel alone, over per-pair
// counters cleared here and incremented by nothing (no main kernel runs), with
// its wait cut to limit_ns.  Each warp gives up after limit_ns, raises
// DFLASH_DEV_TIMEOUT and returns without touching the output; only the
// sequence lengths and the counters are read.
dflash_status launch_attn_wait_timeout_probe(int B, int bs, int Hq, const dflash_kv_cache& c, void* out, void* ws,
                                             unsigned long long limit_ns, cudaStream_t st, const DeviceInfo& dev) {
  const int Hkv = c.num_kv_heads;
  AttnParams p{};
  p.B = B;
  p.bs = bs;
  p.G = Hq / Hkv;
  p.Hkv = Hkv;
  p.Hq = Hq;
  p.cap = c.capacity;
  p.ring = c.ring;
  p.window = 0;
  p.chunk = pick_chunk(B, Hkv, c.capacity, 0);
  p.max_splits = n_splits(c.capacity, p.chunk);
  p.rows = p.G * bs;
  p.seq_len = c.seq_len;
  WsCarver w(ws);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.opart = w.take<float>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows * HD);
  p.mlpart = w.take<float2>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows);
  p.counters = w.take<int>(1 + 2 * static_cast<size_t>(B) * Hkv);
  p.status = dev.status;
  p.wait_limit_ns = limit_ns;
  cudaError_t e = cudaMemsetAsync(p.counters, 0, (1 + 2 * static_cast<size_t>(B) * Hkv) * sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "clear counters");
  const long warps = static_cast<long>(B) * Hkv * p.rows;
  attn_combine_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, st>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "attn_combine_kernel launch");
}

}  // namespace dflash
