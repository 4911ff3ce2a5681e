// Context fusion and K/V injection into the draft cache.
//
// Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash",
// section "Five target states become persistent draft context" (concatenate
// the five captured target states on the feature axis, project them back to
// the draft width, project that into K/V entries inserted into every draft
// layer's cache; the K/V projections of all layers may run as one matrix
// multiplication); "DFlash & DFlash2: Block-Diffusion LLM-Speedup" 4.1
// (H_t = RMSNorm(W_c [H^(l1); ...; H^(l5)]), K_i = W_i^K H_t, V_i = W_i^V H_t).
//
// bf16 path, launches chained as programmatic dependents:
//   1. gemm_tc (fusion)  Y = [taps] W_c^T on tcgen05 tensor cores: a unit is
//      MT x 128 rows by BN columns of Y over a range of K blocks; TMA loads
//      128x64 A tiles (taken from the tap that owns the K block -- the concat is
//      never materialised) and the BNx64 W_c tile into a ring, one thread
//      issues tcgen05.mma (M=128, N=BN, K=16) into MT accumulators in tensor
//      memory, four epilogue warps drain them.  A few new rows (M <= 256):
//      256 x 128 units, so each W_c tile is read once, split K over ~one unit
//      per SM.  Up to ~3840 rows: 256 x 256 units, stream-K over the SMs;
//      more rows: 128 x 256 units.  The fp32 partial sums stay in the
//      workspace.
//   2. rownorm           row -> (sequence, cache position) and its RoPE table
//      (before waiting for the GEMM), then H_t = bf16(sum_splits(Y) *
//      rsqrt(mean(Y^2) + eps) * g)
//   3. gemm_tc (K/V)     [K|V] = H_t W_kv^T; its producer loads the first W_kv
//      tiles before waiting for H_t.  Few rows (M <= 256): 256 x 128 units (one
//      head), stream-K over all SMs into fp32 slots, and
//   4. kv_epilogue       one warp per (row, head): the slot sum; a K head is
//      RMS-normalised (gain k_gain[l]) and rotated at its cache position, a V
//      head copied, both stored as bf16 cache rows.
//      More rows: 128 x 256 units (two heads) with that epilogue fused into the
//      GEMM (stream-K with the in-kernel fixup for tiles past whole waves).
// fp32 path: the same steps as plain SIMT kernels (parity path).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dflash_device.cuh"
#include "dflash_internal.h"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;

struct InvFreq {
  double v[HD / 2];
};

// One CTA per new row m:
//   * row -> (sequence, cache position) and the RoPE (cos, sin) table of the row
//     (used by the K/V epilogue);
//   * H_t[m] = the sum of the split-K partials of Y[m], RMS-normalised with
//     gain g, stored as TH (workspace copy for the K/V GEMM) and optionally as
//     the caller's copy.  Each thread keeps its float4 slots of the row in
//     registers (rows up to 4096 wide), so the partials are read once.
constexpr int kNormThreads = 256;     // fp32 path
constexpr int kNormMaxThreads = 512;
constexpr int kNormSlots = 2;        // float4 slots per thread (in registers up to 2 x the block)
constexpr int kNormBatch = 4;        // split-K slots requested together (more costs occupancy at large M)

template <typename TG, typename TH>
__global__ void __launch_bounds__(kNormMaxThreads) fuse_rownorm_kernel(
    const float* __restrict__ part, int k_splits, const int* __restrict__ pieces, int tile_rows, int tile_cols,
    int n_tiles, int M, int D, const TG* __restrict__ g, float eps,
    TH* __restrict__ ht, TH* __restrict__ ht_out, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ seq_len, int B, int cap, int ring, InvFreq inv, int2* __restrict__ rowinfo,
    void* __restrict__ rope_cs, int rope_row_major, int* __restrict__ zero_flags, int n_zero,
    const int32_t* __restrict__ table,
    int max_pages, int page_size, int num_pages, unsigned* status) {
  const int m = blockIdx.x;
  // the row's sequence: the largest b with cu_new[b] <= m (cu_new is
  // non-decreasing), found by warp 0 with 32 probes per step, so 128
  // sequences take two dependent loads, not seven; the invariant
  // cu_new[lo] <= m keeps lane 0's probe true
  __shared__ int s_b;
  if (threadIdx.x < 32) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) / 32;
      const int idx = lo + static_cast<int>(threadIdx.x) * step;
      const unsigned bal = __ballot_sync(0xffffffffu, idx < hi && cu_new[idx] <= m);
      lo += (31 - __clz(bal)) * step;
      hi = min(hi, lo + step);
    }
    if (threadIdx.x == 0) s_b = lo;
  }
  __syncthreads();
  if (threadIdx.x <= HD / 2) {
    const int b = s_b;
    const int t = m - cu_new[b];
    const int nnew = cu_new[b + 1] - cu_new[b];
    const int n = seq_len[b];
    // linear cache: position p is row p (n + nnew <= cap); ring cache: row
    // p % cap, at most cap new rows per sequence and call
    const bool seq_ok = n >= 0 && (ring || n <= cap);
    const bool valid = seq_ok && (ring ? nnew <= cap : n + nnew <= cap) && t >= 0 && t < nnew;
    const int pos = valid ? n + t : 0;  // the RoPE position is always the absolute one
    if (threadIdx.x < HD / 2) {
      double ang = static_cast<double>(pos) * inv.v[threadIdx.x];
      ang -= kTwoPi * rint(ang * kInvTwoPi);
      float sv, cv;
      sincosf(static_cast<float>(ang), &sv, &cv);
      // fp32 rows keep fp32 angles; for bf16 rows the (cos, sin) pairs are held
      // as fp16 (relative error 2^-11, a quarter of the bf16 rounding of the
      // stored key), so that a K head's 64 pairs fit one register load each
      // element-major [64][M] for the GEMM's fused epilogue (a warp's lanes are
      // rows); row-major [M][64] for kv_epilogue_kernel (a warp is one row)
      const size_t ci = rope_row_major ? static_cast<size_t>(m) * (HD / 2) + threadIdx.x
                                       : static_cast<size_t>(threadIdx.x) * M + m;
      if (sizeof(TH) == 4)
        static_cast<float2*>(rope_cs)[ci] = make_float2(cv, sv);
      else
        static_cast<__half2*>(rope_cs)[ci] = __floats2half2_rn(cv, sv);
    } else {
      // (cache slab, row): linear (sequence, position), ring (sequence, position
      // mod capacity), paged (page of the position, position mod page size)
      int2 ri = make_int2(-1, -1);
      if (!valid) {
        raise_status(status, seq_ok ? DFLASH_DEV_CAPACITY : DFLASH_DEV_BAD_SEQLEN);
      } else if (table) {
        const int pg = table[static_cast<size_t>(b) * max_pages + pos / page_size];
        if (pg >= 0 && pg < num_pages)
          ri = make_int2(pg, pos % page_size);
        else
          raise_status(status, DFLASH_DEV_BAD_SEQLEN);
      } else {
        ri = make_int2(b, ring ? pos % cap : pos);
      }
      rowinfo[m] = ri;
    }
  }
  pdl_launch_dependents();
  pdl_wait_primary();  // the partials of the fusion GEMM
  pieces = pdl_fresh(pieces);
  // the fixup flags of the K/V GEMM that follows (every earlier grid has completed)
  if (m == 0)
    for (int i = threadIdx.x; i < n_zero; i += static_cast<int>(blockDim.x)) zero_flags[i] = 0;
  const int nv = D / 4;  // float4 slots of the row
  const float4* prow = reinterpret_cast<const float4*>(part + static_cast<size_t>(m) * D);
  const size_t split_stride = static_cast<size_t>(M) * D / 4;
  // stream-K partials: a tile has as many slots as shares that met it
  const int* prow_pieces = pieces ? pieces + (m / tile_rows) * n_tiles : nullptr;
  auto row_sum = [&](int v) {
    float4 t4 = prow[v];
    const int ns = prow_pieces ? prow_pieces[(4 * v) / tile_cols] : k_splits;
    for (int s = 1; s < ns; ++s) {
      const float4 t = prow[s * split_stride + v];
      t4.x += t.x;
      t4.y += t.y;
      t4.z += t.z;
      t4.w += t.w;
    }
    return t4;
  };
  const int nthr = blockDim.x;
  const bool in_regs = nv <= nthr * kNormSlots;
  float4 y[kNormSlots];
  float ss = 0.f;
  int ns[kNormSlots] = {};
  if (in_regs) {
    // slots outermost, so the loads of a thread's float4 slots are independent
    int ns_max = 0;
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i) {
      const int v = threadIdx.x + i * nthr;
      y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      ns[i] = v < nv ? (prow_pieces ? prow_pieces[(4 * v) / tile_cols] : k_splits) : 0;
      ns_max = max(ns_max, ns[i]);
      if (v < nv) y[i] = prow[v];
    }
    for (int s0 = 1; s0 < ns_max; s0 += kNormBatch) {
      float4 t[kNormBatch][kNormSlots];
#pragma unroll
      for (int u = 0; u < kNormBatch; ++u)
#pragma unroll
        for (int i = 0; i < kNormSlots; ++i)
          if (s0 + u < ns[i]) t[u][i] = __ldcg(prow + (s0 + u) * split_stride + threadIdx.x + i * nthr);
#pragma unroll
      for (int u = 0; u < kNormBatch; ++u)
#pragma unroll
        for (int i = 0; i < kNormSlots; ++i)
          if (s0 + u < ns[i]) {
            y[i].x += t[u][i].x;
            y[i].y += t[u][i].y;
            y[i].z += t[u][i].z;
            y[i].w += t[u][i].w;
          }
    }
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i)
      ss += y[i].x * y[i].x + y[i].y * y[i].y + y[i].z * y[i].z + y[i].w * y[i].w;
  }
  if (!in_regs) {
    for (int v = threadIdx.x; v < nv; v += nthr) {
      const float4 t4 = row_sum(v);
      ss += t4.x * t4.x + t4.y * t4.y + t4.z * t4.z + t4.w * t4.w;
    }
  }
  ss = warp_sum(ss);
  __shared__ float red[kNormMaxThreads / 32];
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nthr / 32; ++w) tot += red[w];
  const float r = rsqrtf(tot / static_cast<float>(D) + eps);
  if (in_regs && sizeof(TH) == 2 && D % 32 == 0) {  // whole, aligned 128-byte lines per row
    // every thread's slot loads have returned (the barrier above): the row's
    // slot lines are read by this CTA only, drop them from L2 rather than let
    // them be written back.  A 128-byte line is eight float4 of eight
    // consecutive threads of one warp; the first of them drops it, for the
    // slots its tile has (stream-K tiles past the whole waves have many, the
    // others one).
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i) {
      const int v = threadIdx.x + i * nthr;
      if (v < nv && (v & 7) == 0)
        for (int sl = 0; sl < ns[i]; ++sl) discard_l2_line(prow + sl * split_stride + v);
    }
  }
  auto store = [&](int v, float4 t4) {
    const int e = 4 * v;
    const float g0 = g ? to_f32<TG>(g[e]) : 1.f, g1 = g ? to_f32<TG>(g[e + 1]) : 1.f;
    const float g2 = g ? to_f32<TG>(g[e + 2]) : 1.f, g3 = g ? to_f32<TG>(g[e + 3]) : 1.f;
    const TH h0 = from_f32<TH>(t4.x * r * g0), h1 = from_f32<TH>(t4.y * r * g1);
    const TH h2 = from_f32<TH>(t4.z * r * g2), h3 = from_f32<TH>(t4.w * r * g3);
    TH* d = ht + static_cast<size_t>(m) * D + e;
    TH* o = ht_out ? ht_out + static_cast<size_t>(m) * D + e : nullptr;
    if constexpr (sizeof(TH) == 2) {  // one 8-byte store per four values (e is a multiple of 4)
      const uint2 pk = make_uint2(pack_bf16x2(to_f32<TH>(h0), to_f32<TH>(h1)), pack_bf16x2(to_f32<TH>(h2), to_f32<TH>(h3)));
      *reinterpret_cast<uint2*>(d) = pk;
      if (o) *reinterpret_cast<uint2*>(o) = pk;
    } else {
      d[0] = h0;
      d[1] = h1;
      d[2] = h2;
      d[3] = h3;
      if (o) {
        o[0] = h0;
        o[1] = h1;
        o[2] = h2;
        o[3] = h3;
      }
    }
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i) {
      const int v = threadIdx.x + i * nthr;
      if (v < nv) store(v, y[i]);
    }
  } else {
    for (int v = threadIdx.x; v < nv; v += nthr) store(v, row_sum(v));
  }
}

// ------------------------------------------------------------- fp32 path ----

struct F32Segs {
  const float* a[kMaxSeg];
};

// C[M][N] = [A_0 | A_1 | ...] (each [M][kseg]) x W^T, W [N][K]; 64x64 tiles.
__global__ void __launch_bounds__(256) simt_gemm_f32_kernel(F32Segs segs, int kseg, const float* __restrict__ W,
                                                            int M, int N, int K, float* __restrict__ C) {
  __shared__ float As[16][64 + 1];
  __shared__ float Ws[16][64 + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i % 16, r = i / 16;
      const int k = k0 + kk;
      const int seg = k / kseg;
      As[kk][r] = (m0 + r < M && k < K) ? segs.a[seg][static_cast<size_t>(m0 + r) * kseg + (k - seg * kseg)] : 0.f;
      Ws[kk][r] = (n0 + r < N && k < K) ? W[static_cast<size_t>(n0 + r) * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += As[kk][ty * 4 + i] * Ws[kk][tx * 4 + j];
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) {
      const int r = m0 + ty * 4 + i, c = n0 + tx * 4 + j;
      if (r < M && c < N) C[static_cast<size_t>(r) * N + c] = acc[i][j];
    }
}

// One warp per (row, head of the K/V projection): norm + RoPE for keys, store.
__global__ void __launch_bounds__(256) kv_store_f32_kernel(const float* __restrict__ kv, int M, int L, int Hkv,
                                                           int Bc, int cap, const int2* __restrict__ rowinfo,
                                                           const float2* __restrict__ rope_cs,
                                                           const float* __restrict__ k_gain, float eps,
                                                           float* __restrict__ cache_k, float* __restrict__ cache_v) {
  const int heads = L * 2 * Hkv;
  const long wid = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= static_cast<long>(M) * heads) return;
  const int m = static_cast<int>(wid / heads), hidx = static_cast<int>(wid % heads);
  const int2 ri = rowinfo[m];
  if (ri.x < 0) return;
  const int l = hidx / (2 * Hkv), s = (hidx / Hkv) % 2, h = hidx % Hkv;
  const float* src = kv + static_cast<size_t>(m) * heads * HD + static_cast<size_t>(hidx) * HD;
  float* dst = (s == 0 ? cache_k : cache_v) + (((static_cast<size_t>(l) * Bc + ri.x) * Hkv + h) * cap + ri.y) * HD;
  const int e0 = 2 * lane;
  float x0 = src[e0], x1 = src[e0 + 1], y0 = src[e0 + 64], y1 = src[e0 + 65];
  if (s == 1) {
    dst[e0] = x0;
    dst[e0 + 1] = x1;
    dst[e0 + 64] = y0;
    dst[e0 + 65] = y1;
    return;
  }
  const float ss = warp_sum(x0 * x0 + x1 * x1 + y0 * y0 + y1 * y1);
  const float r = rsqrtf(ss * (1.0f / HD) + eps);
  const float* kg = k_gain ? k_gain + l * HD : nullptr;
  x0 *= r * (kg ? kg[e0] : 1.f);
  x1 *= r * (kg ? kg[e0 + 1] : 1.f);
  y0 *= r * (kg ? kg[e0 + 64] : 1.f);
  y1 *= r * (kg ? kg[e0 + 65] : 1.f);
  const float2 c0 = rope_cs[static_cast<size_t>(e0) * M + m], c1 = rope_cs[static_cast<size_t>(e0 + 1) * M + m];
  dst[e0] = x0 * c0.x - y0 * c0.y;
  dst[e0 + 1] = x1 * c1.x - y1 * c1.y;
  dst[e0 + 64] = y0 * c0.x + x0 * c0.y;
  dst[e0 + 65] = y1 * c1.x + x1 * c1.y;
}

// bf16 cache, few rows: the K/V GEMM leaves stream-K partial sums in slots and
// this kernel finishes them, one warp per (row, head of the K/V projection):
// the sum of the tile's slots, then for keys the per-head RMSNorm * k_gain and
// RoPE, and the bf16 store into the cache.  Lane i holds elements 2i, 2i + 1
// and their RoPE partners 2i + 64, 2i + 65; a warp's slot loads and stores are
// 256 contiguous bytes.  Every load of a warp is issued before any is used:
// the first kMaxKvSlots slots are read whatever the tile's slot count (the
// unused ones are masked out), so the warp waits for memory once; many warps
// per SM overlap those waits, which the GEMM's four epilogue warps cannot.
constexpr int kMaxKvSlots = 4;

__global__ void __launch_bounds__(256) kv_epilogue_kernel(
    const float* __restrict__ part, int slots, const int* __restrict__ pieces, int tile_rows, int n_tiles, int M,
    int L, int Hkv, int Bc, int cap, const int2* __restrict__ rowinfo, const __half2* __restrict__ rope_cs,
    const __nv_bfloat16* __restrict__ k_gain, float eps, __nv_bfloat16* __restrict__ cache_k,
    __nv_bfloat16* __restrict__ cache_v) {
  pdl_wait_primary();  // the partial sums of the K/V GEMM
  pdl_launch_dependents();
  pieces = pdl_fresh(pieces);
  const int heads = L * 2 * Hkv;
  const long wid = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= static_cast<long>(M) * heads) return;
  const int m = static_cast<int>(wid / heads), hidx = static_cast<int>(wid % heads);
  const int l = hidx / (2 * Hkv), s = (hidx / Hkv) % 2, h = hidx % Hkv;
  const size_t N = static_cast<size_t>(heads) * HD;
  const size_t slot = static_cast<size_t>(M) * N;
  const float* src = part + static_cast<size_t>(m) * N + static_cast<size_t>(hidx) * HD;
  const int e0 = 2 * lane;
  // every load up front
  const int2 ri = rowinfo[m];
  const int ns = pieces[(m / tile_rows) * n_tiles + hidx];  // 128-column tiles: tile n = head
  float2 u[kMaxKvSlots], v[kMaxKvSlots];
#pragma unroll
  for (int k = 0; k < kMaxKvSlots; ++k) {
    u[k] = make_float2(0.f, 0.f);
    v[k] = make_float2(0.f, 0.f);
    if (k < slots) {
      u[k] = __ldcg(reinterpret_cast<const float2*>(src + k * slot + e0));
      v[k] = __ldcg(reinterpret_cast<const float2*>(src + k * slot + e0 + 64));
    }
  }
  __half2 cs0 = __floats2half2_rn(1.f, 0.f), cs1 = cs0;
  float g0 = 1.f, g1 = 1.f, g2 = 1.f, g3 = 1.f;  // element loads: the gain vector may be 2-byte aligned
  if (s == 0) {
    // the row's (cos, sin) pairs, row-major: one 8-byte load of frequencies e0, e0 + 1
    const uint2 cs = *reinterpret_cast<const uint2*>(rope_cs + static_cast<size_t>(m) * (HD / 2) + e0);
    cs0 = *reinterpret_cast<const __half2*>(&cs.x);
    cs1 = *reinterpret_cast<const __half2*>(&cs.y);
    if (k_gain) {
      const __nv_bfloat16* kg = k_gain + l * HD;
      g0 = __bfloat162float(kg[e0]);
      g1 = __bfloat162float(kg[e0 + 1]);
      g2 = __bfloat162float(kg[e0 + 64]);
      g3 = __bfloat162float(kg[e0 + 65]);
    }
  }
  float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMaxKvSlots; ++k)
    if (k < ns) {
      a.x += u[k].x;
      a.y += u[k].y;
      b.x += v[k].x;
      b.y += v[k].y;
    }
  for (int k = kMaxKvSlots; k < ns; ++k) {  // more slots than kept in registers
    const float2 x = __ldcg(reinterpret_cast<const float2*>(src + k * slot + e0));
    const float2 y = __ldcg(reinterpret_cast<const float2*>(src + k * slot + e0 + 64));
    a.x += x.x;
    a.y += x.y;
    b.x += y.x;
    b.y += y.y;
  }
  // the slots' lines of this (row, head) are read by this warp only: drop them
  // from L2 (4 lines of 128 bytes per slot) rather than let them be written back
  __syncwarp();
  const int nread = max(ns, min(slots, kMaxKvSlots));
  for (int i = lane; i < 4 * nread; i += 32) discard_l2_line(src + (i / 4) * slot + (i % 4) * 32);
  if (s == 0) {
    const float ss = warp_sum(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
    const float r = rsqrtf(ss * (1.0f / HD) + eps);
    const float x0 = a.x * r * g0, x1 = a.y * r * g1, y0 = b.x * r * g2, y1 = b.y * r * g3;
    const float2 c0 = __half22float2(cs0), c1 = __half22float2(cs1);
    a = make_float2(x0 * c0.x - y0 * c0.y, x1 * c1.x - y1 * c1.y);
    b = make_float2(y0 * c0.x + x0 * c0.y, y1 * c1.x + x1 * c1.y);
  }
  if (ri.x < 0) return;  // row flagged by the row map: nothing is stored
  __nv_bfloat16* dst =
      (s == 0 ? cache_k : cache_v) + (((static_cast<size_t>(l) * Bc + ri.x) * Hkv + h) * cap + ri.y) * HD;
  reinterpret_cast<uint32_t*>(dst)[lane] = pack_bf16x2(a.x, a.y);
  reinterpret_cast<uint32_t*>(dst + 64)[lane] = pack_bf16x2(b.x, b.y);
}

// ------------------------------------------------------------- planning -----

// A few new rows (M <= 256, weight-bound): the fusion GEMM takes 256-row by
// 128-column units (each W_c tile read once) split along K to about one unit
// per SM, and the K/V GEMM 128 x 128 units of one head (enough units to fill
// the SMs).  Larger M (tensor-bound): 128 x 256 units for both, the N = 256
// MMA doing twice the work of N = 128 for 1.6x its time.  When the fusion
// GEMM's tiles do not fill whole waves of kSplitTarget CTAs, the whole waves
// run tile by tile and the remaining tiles are balanced by stream-K over
// kSplitTarget shares, with as many partial-sum slots as the most shares
// meeting one tile.
struct FusePlan {
  int fuse_mt, fuse_bn, fuse_m_tiles, fuse_n_tiles, k_splits, kv_bn, stream_k, shares, dp_tiles;
  int kv_mt, kv_m_tiles, kv_n_tiles, kv_shares;  // K/V GEMM: stream-K over kv_shares CTAs
  int kv_split;  // M <= 256: partial sums left in kv_slots slots, finished by kv_epilogue_kernel;
  int kv_slots;  // otherwise the GEMM's own epilogue finishes them (fixup)
};


FusePlan plan(int M, int D, int num_kb, int n_kv) {
  FusePlan f;
  f.fuse_bn = M <= 2 * kBM ? 128 : 256;
  f.fuse_n_tiles = D / f.fuse_bn;
  // 256-row units read each activation tile half as often; they fill all of
  // tensor memory (no second accumulator to overlap an epilogue with the next
  // unit), so they are taken only while every CTA has at most about one unit
  const int m256 = (M + 2 * kBM - 1) / (2 * kBM);
  f.fuse_mt = (M <= 2 * kBM || m256 * f.fuse_n_tiles <= kSplitTarget) ? 2 : 1;
  f.fuse_m_tiles = (M + f.fuse_mt * kBM - 1) / (f.fuse_mt * kBM);
  const int tiles = f.fuse_m_tiles * f.fuse_n_tiles;
  f.stream_k = M > 2 * kBM && tiles % kSplitTarget != 0;
  f.shares = 0;
  f.dp_tiles = 0;
  f.k_splits = std::max(1, std::min(16, kSplitTarget / std::max(1, tiles)));
  if (f.stream_k) {
    f.dp_tiles = tiles / kSplitTarget * kSplitTarget;
    const long tot = static_cast<long>(tiles - f.dp_tiles) * num_kb;
    f.shares = static_cast<int>(std::min<long>(kSplitTarget, tot));  // every share non-empty
    auto share = [&](long x) { return ((x + 1) * f.shares - 1) / tot; };
    f.k_splits = 1;
    for (long t = 0; t < tiles - f.dp_tiles; ++t)
      f.k_splits = std::max(f.k_splits, static_cast<int>(share((t + 1) * num_kb - 1) - share(t * num_kb) + 1));
  }
  f.kv_bn = M <= 2 * kBM ? 128 : 256;
  f.kv_mt = M <= 2 * kBM ? 2 : 1;
  f.kv_m_tiles = (M + f.kv_mt * kBM - 1) / (f.kv_mt * kBM);
  f.kv_n_tiles = n_kv / f.kv_bn;
  f.kv_shares = fixup_shares(f.kv_m_tiles * f.kv_n_tiles, D / kBK);
  f.kv_split = M <= 2 * kBM;
  f.kv_slots = sk_max_count(static_cast<long>(f.kv_m_tiles) * f.kv_n_tiles, D / kBK, f.kv_shares);
  return f;
}


}  // namespace

size_t fuse_ws_bytes(int M, int J, int dt_width, int D, int L, int Hkv, dflash_dtype dt) {
  const int Ntot = L * 2 * Hkv * HD;
  size_t s = align256(static_cast<size_t>(M) * sizeof(int2)) +
             align256(static_cast<size_t>(M) * (HD / 2) * sizeof(float2));
  if (dt == DFLASH_BF16) {
    const FusePlan f = plan(M, D, J * dt_width / kBK, Ntot);
    s += (f.kv_split ? align256(static_cast<size_t>(f.kv_slots) * M * Ntot * sizeof(float)) +
                           align256(static_cast<size_t>(f.kv_m_tiles) * f.kv_n_tiles * sizeof(int))
                     : fixup_ws_bytes<256, 1>(f.kv_shares)) +
         align256(static_cast<size_t>(f.k_splits) * M * D * sizeof(float)) +
         align256(static_cast<size_t>(M) * D * sizeof(__nv_bfloat16)) +
         align256(static_cast<size_t>(f.fuse_m_tiles) * f.fuse_n_tiles * sizeof(int));
  } else {
    s += align256(static_cast<size_t>(M) * D * sizeof(float)) * 2 +
         align256(static_cast<size_t>(M) * Ntot * sizeof(float));
  }
  return s + 256;
}

dflash_status launch_fuse_context(int J, const void* const* taps, int dt_width, const int32_t* cu_new,
                                  int B, int M, const void* w_fuse, const void* g_fuse, int D,
                                  const void* w_kv, const void* k_gain, float theta, float eps,
                                  const dflash_kv_cache& c, void* h_t_out, void* ws, cudaStream_t st,
                                  const DeviceInfo& dev) {
  const int L = c.num_layers, Hkv = c.num_kv_heads;
  const int Ntot = L * 2 * Hkv * HD;
  InvFreq inv;
  for (int e = 0; e < HD / 2; ++e) inv.v[e] = std::pow(static_cast<double>(theta), -2.0 * e / HD);
  WsCarver w(ws);
  int2* rowinfo = w.take<int2>(M);
  float2* rope_cs = w.take<float2>(static_cast<size_t>(M) * (HD / 2));

  if (c.dtype == DFLASH_F32) {
    float* Y = w.take<float>(static_cast<size_t>(M) * D);
    float* H = w.take<float>(static_cast<size_t>(M) * D);
    float* KV = w.take<float>(static_cast<size_t>(M) * Ntot);
    F32Segs segs{};
    for (int j = 0; j < J; ++j) segs.a[j] = static_cast<const float*>(taps[j]);
    simt_gemm_f32_kernel<<<dim3((D + 63) / 64, (M + 63) / 64), 256, 0, st>>>(
        segs, dt_width, static_cast<const float*>(w_fuse), M, D, J * dt_width, Y);
    fuse_rownorm_kernel<float, float><<<M, kNormThreads, 0, st>>>(
        Y, 1, nullptr, kBM, D, 1, M, D, static_cast<const float*>(g_fuse), eps, H, static_cast<float*>(h_t_out), cu_new, c.seq_len, B,
        c.capacity, c.ring, inv, rowinfo, rope_cs, 0, nullptr, 0, nullptr, 0, 0, 0, dev.status);
    F32Segs hs{};
    hs.a[0] = H;
    simt_gemm_f32_kernel<<<dim3((Ntot + 63) / 64, (M + 63) / 64), 256, 0, st>>>(
        hs, D, static_cast<const float*>(w_kv), M, Ntot, D, KV);
    const long warps = static_cast<long>(M) * L * 2 * Hkv;
    kv_store_f32_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
        KV, M, L, Hkv, c.batch, c.capacity, rowinfo, const_cast<const float2*>(rope_cs), static_cast<const float*>(k_gain), eps,
        static_cast<float*>(c.k), static_cast<float*>(c.v));
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "fp32 fusion launch");
  }

  const FusePlan f = plan(M, D, J * dt_width / kBK, Ntot);
  if (L * HD > 4 * 32 * kStgRow)  // the K/V epilogue keeps every layer's K gains in shared memory
    return fail(DFLASH_ERR_UNSUPPORTED, "fusion: at most 36 draft layers");
  if (D % 4 != 0) return fail(DFLASH_ERR_UNSUPPORTED, "fusion: d_model must be a multiple of 4");
  float* Ypart = w.take<float>(static_cast<size_t>(f.k_splits) * M * D);
  auto* H = w.take<__nv_bfloat16>(static_cast<size_t>(M) * D);
  int* tile_pieces = w.take<int>(static_cast<size_t>(f.fuse_m_tiles) * f.fuse_n_tiles);
  GemmArgs k{};
  float* KVpart = nullptr;
  if (f.kv_split) {
    KVpart = w.take<float>(static_cast<size_t>(f.kv_slots) * M * Ntot);
    k.pieces = w.take<int>(static_cast<size_t>(f.kv_m_tiles) * f.kv_n_tiles);
    k.stream_k = f.kv_shares;
    k.dp_tiles = 0;
    k.k_splits = f.kv_slots;
    k.out_f32 = KVpart;
  } else {
    fixup_take<256, 1>(w, f.kv_shares, k);
  }

  // 1. fusion GEMM: A = the J taps (one tensor map each), B = W_c [D][J*dt]
  TmapPack am{};
  for (int j = 0; j < J; ++j) {
    dflash_status s = make_tmap_bf16_2d(&am.a[j], taps[j], static_cast<uint64_t>(M), dt_width, kBM, kBK);
    if (s) return s;
  }
  CUtensorMap bm;
  dflash_status s =
      make_tmap_bf16_2d(&bm, w_fuse, static_cast<uint64_t>(D), static_cast<uint64_t>(J) * dt_width, f.fuse_bn, kBK);
  if (s) return s;
  GemmArgs a{};
  a.M = M;
  a.N = D;
  a.num_kb = J * dt_width / kBK;
  a.kb_per_seg = dt_width / kBK;
  a.k_splits = f.stream_k ? f.k_splits : std::min(f.k_splits, a.num_kb);
  a.stream_k = f.stream_k ? f.shares : 0;
  a.dp_tiles = f.dp_tiles;
  a.pieces = tile_pieces;
  a.m_tiles = f.fuse_m_tiles;
  a.n_tiles = f.fuse_n_tiles;
  a.epi = 0;
  a.pdl = 1;  // its CTAs may start while the preceding kernel finishes; the taps are loaded after it has,
  a.prefetch_b = 1;  // the weights (which no kernel of the chain writes) before
  a.out_f32 = Ypart;
  a.status = dev.status;
  s = f.fuse_bn == 128  ? launch_gemm<128, 4, 2>(am, bm, a, st, dev)
      : f.fuse_mt == 2 ? launch_gemm<256, 3, 2>(am, bm, a, st, dev)
                       : launch_gemm<256, 4, 1>(am, bm, a, st, dev);
  if (s) return s;

  // 2. row map + split-K sum + RMSNorm -> H_t (bf16), a programmatic dependent
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    // one or two float4 of the row per thread; at least 65 threads (the
    // RoPE angles and the row map)
    cfg.blockDim = dim3(static_cast<unsigned>(
        std::min(kNormMaxThreads, std::max(96, ((D / 4 + kNormSlots - 1) / kNormSlots + 31) / 32 * 32))));
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le = cudaLaunchKernelEx(&cfg, fuse_rownorm_kernel<__nv_bfloat16, __nv_bfloat16>,
                                        static_cast<const float*>(Ypart), a.k_splits,
                                        static_cast<const int*>(f.stream_k ? tile_pieces : nullptr), f.fuse_mt * kBM,
                                        f.fuse_bn, f.fuse_n_tiles, M, D,
                                        static_cast<const __nv_bfloat16*>(g_fuse), eps, H,
                                        static_cast<__nv_bfloat16*>(h_t_out), cu_new, c.seq_len, B, c.capacity,
                                        c.ring, inv, rowinfo, rope_cs, f.kv_split ? 1 : 0, k.fix_flag,
                                        f.kv_split ? 0 : f.kv_shares,
                                        c.block_table, c.max_pages, c.page_size, c.num_pages, dev.status);
    if (le != cudaSuccess) return cuda_fail(le, "fuse_rownorm_kernel launch");
  }

  // 3. K/V GEMM with the cache epilogue
  TmapPack hm{};
  s = make_tmap_bf16_2d(&hm.a[0], H, static_cast<uint64_t>(M), D, kBM, kBK);
  if (s) return s;
  CUtensorMap wm;
  s = make_tmap_bf16_2d(&wm, w_kv, static_cast<uint64_t>(Ntot), D, f.kv_bn, kBK);
  if (s) return s;
  k.M = M;
  k.N = Ntot;
  k.num_kb = D / kBK;
  k.kb_per_seg = k.num_kb;
  k.m_tiles = f.kv_m_tiles;
  k.n_tiles = f.kv_n_tiles;
  k.epi = f.kv_split ? 0 : 1;
  k.pdl = 1;
  k.prefetch_b = 1;
  k.cache_k = static_cast<__nv_bfloat16*>(c.k);
  k.cache_v = static_cast<__nv_bfloat16*>(c.v);
  k.L = L;
  // a cache slab per (layer, x, head) of R rows: x = sequence and R = capacity
  // (linear, ring) or x = page and R = page size (paged)
  const int slabs = c.block_table ? c.num_pages : c.batch;
  const int slab_rows = c.block_table ? c.page_size : c.capacity;
  k.Bc = slabs;
  k.Hkv = Hkv;
  k.cap = slab_rows;
  k.rowinfo = rowinfo;
  k.rope_cs = reinterpret_cast<const __half2*>(rope_cs);
  k.k_gain = static_cast<const __nv_bfloat16*>(k_gain);
  k.eps = eps;
  k.status = dev.status;
  if (!f.kv_split) return launch_gemm<256, 4, 1>(hm, wm, k, st, dev);
  s = launch_gemm<128, 4, 2>(hm, wm, k, st, dev);
  if (s) return s;

  // 4. the K/V epilogue over the partial sums, a programmatic dependent
  cudaLaunchConfig_t cfg = {};
  const long warps = static_cast<long>(M) * L * 2 * Hkv;
  cfg.gridDim = dim3(static_cast<unsigned>((warps * 32 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, kv_epilogue_kernel, static_cast<const float*>(KVpart), f.kv_slots,
                                      static_cast<const int*>(k.pieces), f.kv_mt * kBM, f.kv_n_tiles, M, L, Hkv,
                                      slabs, slab_rows, static_cast<const int2*>(rowinfo),
                                      reinterpret_cast<const __half2*>(rope_cs), static_cast<const __nv_bfloat16*>(k_gain),
                                      eps, static_cast<__nv_bfloat16*>(c.k), static_cast<__nv_bfloat16*>(c.v));
  return le == cudaSuccess ? DFLASH_OK : cuda_fail(le, "kv_epilogue_kernel launch");
}

}  // namespace dflash
