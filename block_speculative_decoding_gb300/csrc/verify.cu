// Exact speculative verification over the full vocabulary.
//
// Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash",
// section "Why exact verification preserves the target" (accept with
// min(1, p/q), otherwise draw from the normalised positive residual; greedy:
// accept while the draft equals the target argmax); "DFlash & DFlash2:
// Block-Diffusion LLM-Speedup", 4.4 (same rules) and FAQ Q3 (temperature
// applied to both rows before the ratio).
//
// Kernels (one stream, no inter-CTA waiting):
//   1. stats    -- every logit row (bs target rows, bs-1 draft rows per
//                  sequence) is cut into 16384-logit chunks; each CTA streams
//                  one chunk with 16-byte loads and writes (max, sum 2^x) of
//                  x = logit * log2(e)/T, or (max, first argmax) when T == 0.
//   2. decide   -- (T == 0) one warp per sequence: the target argmax of every
//                  row against the draft tokens.
//   2. finish   -- (T > 0) one CTA per (sequence, chunk), launched as a
//                  programmatic dependent of the stats pass; four fit on an
//                  SM, so the whole grid is resident at once.  Before waiting
//                  for the stats pass the CTA loads the draft tokens and their
//                  target and draft logits and draws the Philox words; then
//                  its warps merge the sequence's chunk partials into
//                  log-normalisers and one warp evaluates
//                  alpha_k = min(1, p(x)/q(x)) and finds the first rejection n
//                  (every CTA of the sequence takes the same decision).  The
//                  CTA sums max(0, p - q) (the bonus row: p) over its chunk of
//                  row n; the last CTA of the sequence to finish (an atomic
//                  count) runs the inverse-CDF search for the first index
//                  whose cumulative mass exceeds v * S.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "dflash_device.cuh"
#include "dflash_internal.h"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 16384;                 // logits per CTA chunk
constexpr int kPerThread = kChunk / kThreads;  // 64 logits per thread
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kFinishChunks = 1;              // chunks per CTA of the finish kernel
constexpr int kResidParts = 2;                // passes per warp over its residual segment
constexpr int kSeg = 2048;                    // logits per residual-mass segment (one warp's share of a chunk)
constexpr int kSegsPerChunk = kChunk / kSeg;

struct Decision {
  int n;            // accepted drafts; the correction/bonus comes from row n
  uint32_t vbits;   // Philox word for the draw at row n
  float lzp;        // log2 normaliser of p (row n), in units of logit*scale
  float lzq;        // log2 normaliser of q (row n); unused for the bonus row
};

// 16-byte vector loaders: 8 bf16, 4 fp32, or one scalar.
template <typename T, int VEC>
struct Vec;
template <>
struct Vec<__nv_bfloat16, 8> {
  using type = uint4;
  static __device__ __forceinline__ void unpack(const type& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  }
};
template <>
struct Vec<float, 4> {
  using type = float4;
  static __device__ __forceinline__ void unpack(const type& v, float* f) {
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <typename T>
struct Vec<T, 1> {
  using type = T;
  static __device__ __forceinline__ void unpack(const type& v, float* f) { f[0] = to_f32<T>(v); }
};

// (m, s) represents s * 2^m; merges tolerate empty (-inf) sides.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mn = fmaxf(m, m2);
  s = s * exp2f(m - mn) + s2 * exp2f(m2 - mn);
  m = mn;
}

__device__ __forceinline__ void amax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Raw 16-byte vectors of this thread's 64 logits of chunk [e0, e1): vector i
// covers elements e0 + (i*256 + t)*VEC ...; `live` marks in-range vectors.
template <typename T, int VEC>
__device__ __forceinline__ void load_raw(const T* __restrict__ row, int e0, int e1,
                                         typename Vec<T, VEC>::type (&v)[kPerThread / VEC], bool (&live)[kPerThread / VEC]) {
  using VT = typename Vec<T, VEC>::type;
#pragma unroll
  for (int i = 0; i < kPerThread / VEC; ++i) {
    const int e = e0 + (i * kThreads + threadIdx.x) * VEC;
    live[i] = e < e1;
    if (live[i]) v[i] = __ldcs(reinterpret_cast<const VT*>(row + e));
  }
}

// Raw vectors of lane `lane`'s N * VEC logits of one warp's contiguous span
// starting at s0 (in-range below s1): vector i covers elements
// s0 + (i*32 + lane)*VEC ...
template <typename T, int VEC, int N>
__device__ __forceinline__ void load_seg(const T* __restrict__ row, int s0, int s1, int lane,
                                         typename Vec<T, VEC>::type (&v)[N], bool (&live)[N]) {
  using VT = typename Vec<T, VEC>::type;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int e = s0 + (i * 32 + lane) * VEC;
    live[i] = e < s1;
    if (live[i]) v[i] = __ldcg(reinterpret_cast<const VT*>(row + e));
  }
}

// Resident CTAs per SM of the stats pass: six for the bf16 sampling pass (40
// registers, 48 KB of loads in flight per SM more than with four), four where
// more live values would spill.
template <typename T, int VEC, bool GREEDY>
constexpr int stats_ctas_per_sm() {
  return (sizeof(T) == 2 && VEC == 8 && !GREEDY) ? 6 : 4;
}

// The stats pass zeroes the per-sequence counters of the finish kernel.
template <typename T, int VEC, bool GREEDY>
__global__ void __launch_bounds__(kThreads, (stats_ctas_per_sm<T, VEC, GREEDY>())) verify_stats_kernel(const T* __restrict__ lt,
                                                                   const T* __restrict__ ld, int B,
                                                                   int bs, int V, int nchunk,
                                                                   float scale,
                                                                   float2* __restrict__ part,
                                                                   int* __restrict__ counters) {
  // launched as a programmatic dependent of the preceding kernel: nothing is
  // read or written before that grid has completed, and the finish kernel
  // (which loads the draft tokens' logits before its own wait) is released
  // only after that
  pdl_wait_primary();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && counters)
    for (int i = threadIdx.x; i < B; i += kThreads) counters[i] = 0;
  const int c = blockIdx.x % nchunk;
  const int r = blockIdx.x / nchunk;
  const T* row = (r < B * bs) ? lt + static_cast<size_t>(r) * V
                              : ld + static_cast<size_t>(r - B * bs) * V;
  const int e0 = c * kChunk;
  const int e1 = min(V, e0 + kChunk);
  constexpr int NV = kPerThread / VEC;
  typename Vec<T, VEC>::type v[NV];
  bool live[NV];
  load_raw<T, VEC>(row, e0, e1, v, live);

  float a, b;  // GREEDY: (value, index-as-bits); else (max, sum)
  if constexpr (GREEDY) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < NV; ++i) {  // slots visit this thread's logits in index order
      if (!live[i]) continue;
      float f[VEC];
      Vec<T, VEC>::unpack(v[i], f);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const int e = e0 + (i * kThreads + threadIdx.x) * VEC + j;
        if (bi == INT_MAX || f[j] > bv) {
          bv = f[j];
          bi = e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      amax_merge(bv, bi, v2, i2);
    }
    a = bv;
    b = __int_as_float(bi);
  } else {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (!live[i]) continue;
      float f[VEC];
      Vec<T, VEC>::unpack(v[i], f);
#pragma unroll
      for (int j = 0; j < VEC; ++j) mx = fmaxf(mx, f[j]);
    }
    float m = mx * scale;  // scale > 0
    float sum = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        if (!live[i]) continue;
        float f[VEC];
        Vec<T, VEC>::unpack(v[i], f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) sum += ex2_approx(fmaf(f[j], scale, -m));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      lse_merge(m, sum, m2, s2);
    }
    a = m;
    b = sum;
  }
  __shared__ float2 red[kThreads / 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  if (threadIdx.x == 0) {
    float2 acc = red[0];
    for (int w = 1; w < kThreads / 32; ++w) {
      if constexpr (GREEDY) {
        int ai = __float_as_int(acc.y);
        amax_merge(acc.x, ai, red[w].x, __float_as_int(red[w].y));
        acc.y = __int_as_float(ai);
      } else {
        lse_merge(acc.x, acc.y, red[w].x, red[w].y);
      }
    }
    part[static_cast<size_t>(r) * nchunk + c] = acc;
  }
}

// Merge the chunk partials of one row across the warp; every lane gets the result.
template <bool GREEDY>
__device__ __forceinline__ float2 merge_row(const float2* __restrict__ part, int nchunk) {
  float a = -INFINITY, b = GREEDY ? __int_as_float(INT_MAX) : 0.f;
  for (int c = threadIdx.x % 32; c < nchunk; c += 32) {
    const float2 p = part[c];
    if constexpr (GREEDY) {
      int bi = __float_as_int(b);
      amax_merge(a, bi, p.x, __float_as_int(p.y));
      b = __int_as_float(bi);
    } else {
      lse_merge(a, b, p.x, p.y);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a2 = __shfl_xor_sync(0xffffffffu, a, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, b, o);
    if constexpr (GREEDY) {
      int bi = __float_as_int(b);
      amax_merge(a, bi, a2, __float_as_int(b2));
      b = __int_as_float(bi);
    } else {
      lse_merge(a, b, a2, b2);
    }
  }
  return make_float2(a, b);
}

// The decision for sequence b, taken by one warp (lane k: block position k):
// log-normalisers of the rows, the acceptance test of every draft, the first
// rejection n.  Every lane returns the same Decision.  With `acc` / `out` it
// also writes the accepted length and the tokens: the accepted drafts, -1 after
// row n, and at row n the target argmax (greedy) or nothing (the correction is
// drawn later).
template <typename T, bool GREEDY>
__device__ __forceinline__ Decision decide_seq(const T* __restrict__ lt, const T* __restrict__ ld,
                                               const int32_t* __restrict__ x, int b, int B, int bs, int V,
                                               int nchunk, float scale, const float2* __restrict__ part,
                                               uint32_t k0, uint32_t k1, uint32_t c_lo, uint32_t c_hi,
                                               int32_t* __restrict__ acc, int32_t* __restrict__ out,
                                               unsigned* status, const float* s_lz = nullptr,
                                               const float2* pre = nullptr, const uint2* words = nullptr,
                                               const int* xk_pre = nullptr) {
  const int lane = threadIdx.x % 32;
  int xk = -1;
  if (lane < bs - 1) xk = xk_pre ? *xk_pre : x[b * (bs - 1) + lane];
  // pre, words, xk_pre (optional): lane k's target and draft logits of its
  // token, its two Philox words (acceptance, draw) and its token, obtained earlier
  float lzp = 0.f, lzq = 0.f;
  int amax = 0;
  if constexpr (GREEDY) {
    for (int k = 0; k < bs; ++k) {
      const float2 pt = merge_row<true>(part + static_cast<size_t>(b * bs + k) * nchunk, nchunk);
      const int i = __float_as_int(pt.y);
      if (lane == k) amax = (i == INT_MAX) ? 0 : i;
    }
  } else {
    // normalisers precomputed by the block (row_normalisers)
    if (lane < bs) lzp = s_lz[lane];
    if (lane < bs - 1) lzq = s_lz[bs + lane];
  }
  bool rejected = false;
  uint32_t vbits = 0;
  if (lane < bs) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (!GREEDY) {
      if (words) {
        w.x = words->x;
        w.y = words->y;
      } else {
        w = philox4x32_10(make_uint4(lane, b, c_lo, c_hi), k0, k1);
      }
    }
    vbits = w.y;
    if (lane < bs - 1) {
      if (xk < 0 || xk >= V) {
        if (out) raise_status(status, DFLASH_DEV_BAD_TOKEN);
        rejected = true;
      } else if constexpr (GREEDY) {
        rejected = (amax != xk);
      } else {
        const float rt = pre ? pre->x : to_f32<T>(lt[static_cast<size_t>(b * bs + lane) * V + xk]);
        const float rd = pre ? pre->y : to_f32<T>(ld[static_cast<size_t>(b * (bs - 1) + lane) * V + xk]);
        const float lp = rt * scale - lzp;
        const float lq = rd * scale - lzq;
        const float alpha = fminf(1.f, exp2f(lp - lq));
        rejected = !(uniform24(w.x) < alpha);
      }
    }
  }
  const unsigned mask = __ballot_sync(0xffffffffu, rejected);
  const int n = mask ? (__ffs(mask) - 1) : (bs - 1);
  const int amax_n = __shfl_sync(0xffffffffu, amax, n);
  Decision d;
  d.n = n;
  d.vbits = __shfl_sync(0xffffffffu, vbits, n);
  d.lzp = __shfl_sync(0xffffffffu, lzp, n);
  d.lzq = __shfl_sync(0xffffffffu, lzq, n);
  if (out && lane < bs && (GREEDY || lane != n)) out[b * bs + lane] = lane < n ? xk : (lane == n ? amax_n : -1);
  if (acc && lane == 0) acc[b] = n;
  return d;
}

// Greedy decoding: one warp per sequence.
template <typename T>
__global__ void __launch_bounds__(128) verify_decide_kernel(
    const T* __restrict__ lt, const int32_t* __restrict__ x, int B, int bs, int V, int nchunk,
    const float2* __restrict__ part, int32_t* __restrict__ acc, int32_t* __restrict__ out, unsigned* status) {
  pdl_launch_dependents();
  const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (b >= B) return;
  decide_seq<T, true>(lt, lt, x, b, B, bs, V, nchunk, 1.f, part, 0u, 0u, 0u, 0u, acc, out, status);
}

// Residual weight of one logit pair (or of p alone for the bonus row).
__device__ __forceinline__ float resid_weight(float xt, float xd, const Decision& d, bool has_q,
                                              float& pw) {
  pw = ex2_approx(xt - d.lzp);
  if (!has_q) return pw;
  const float qw = ex2_approx(xd - d.lzq);
  return fmaxf(0.f, pw - qw);
}

// log2 normaliser of every row of sequence b (target rows 0..bs-1, then the
// draft rows), from the chunk partials: the warps of the block take the rows in
// turn.  With at most 32 chunks a row (lane c: chunk c), a warp issues the loads
// of all its rows before merging any.
__device__ __forceinline__ void row_normalisers(const float2* __restrict__ part, int b, int B, int bs, int nchunk,
                                                float* s_lz) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int kWarps = kThreads / 32;
  const int nrows = 2 * bs - 1;
  auto part_row = [&](int r) {
    return r < bs ? static_cast<size_t>(b * bs + r) : static_cast<size_t>(B * bs + b * (bs - 1) + r - bs);
  };
  if (nchunk <= 32) {
    constexpr int kRows = (2 * 32 - 1 + kWarps - 1) / kWarps;  // rows per warp for blocks of up to 32
    float2 v[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = warp + kWarps * i;
      v[i] = (r < nrows && lane < nchunk) ? part[part_row(r) * nchunk + lane] : make_float2(-INFINITY, 0.f);
    }
    // per row: the largest chunk maximum first (a max tree), then the chunk
    // sums rescaled to it, one exponential per lane (an add tree)
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = warp + kWarps * i;
      if (r >= nrows) break;
      float M = v[i].x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float sum = (v[i].x == -INFINITY) ? 0.f : v[i].y * exp2f(v[i].x - M);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) s_lz[r] = M + log2f(sum);
    }
    return;
  }
  for (int r = warp; r < nrows; r += kWarps) {
    const float2 st = merge_row<false>(part + part_row(r) * nchunk, nchunk);
    if (lane == 0) s_lz[r] = st.x + log2f(st.y);
  }
}

// Resident CTAs per SM of the finish kernel: four for 16-byte bf16 loads (64
// registers), two where the wider live values would spill.
template <typename T, int VEC>
constexpr int finish_ctas_per_sm() {
  return (sizeof(T) == 2 && VEC == 8) ? 4 : 2;
}

// Non-greedy verification after the stats pass; see the file comment.
template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads, (finish_ctas_per_sm<T, VEC>())) verify_finish_kernel(
    const T* __restrict__ lt, const T* __restrict__ ld, const int32_t* __restrict__ x, int B, int bs, int V,
    int nchunk, float scale, const float2* __restrict__ part, uint32_t k0, uint32_t k1, uint32_t c_lo,
    uint32_t c_hi, int32_t* __restrict__ acc, int32_t* __restrict__ out, float2* __restrict__ rpart,
    int* __restrict__ counters, unsigned* status) {
  pdl_launch_dependents();  // a following call's first kernel may become resident; it waits for this grid
  const int ncb = (nchunk + kFinishChunks - 1) / kFinishChunks;  // CTAs per sequence
  const int b = blockIdx.x / ncb, cb = blockIdx.x % ncb;
  // the draft tokens' logits and the Philox words do not depend on the stats
  // pass: fetch and draw them first
  float2 pre = make_float2(0.f, 0.f);
  uint2 words = make_uint2(0u, 0u);
  int xk = -1;
  if (threadIdx.x < bs - 1) {
    xk = x[b * (bs - 1) + threadIdx.x];
    if (xk >= 0 && xk < V)
      pre = make_float2(to_f32<T>(lt[static_cast<size_t>(b * bs + threadIdx.x) * V + xk]),
                        to_f32<T>(ld[static_cast<size_t>(b * (bs - 1) + threadIdx.x) * V + xk]));
  }
  if (threadIdx.x < bs) {
    const uint4 w = philox4x32_10(make_uint4(threadIdx.x, b, c_lo, c_hi), k0, k1);
    words = make_uint2(w.x, w.y);
  }
  pdl_wait_primary();  // the stats pass's partials and cleared counters
  part = pdl_fresh(part);
  __shared__ Decision s_dec;
  __shared__ int s_is_last;
  __shared__ float s_lz[32];
  row_normalisers(part, b, B, bs, nchunk, s_lz);
  __syncthreads();
  if (threadIdx.x < 32) {
    const Decision dw = decide_seq<T, false>(lt, ld, x, b, B, bs, V, nchunk, scale, part, k0, k1, c_lo, c_hi,
                                             cb == 0 ? acc : nullptr, cb == 0 ? out : nullptr, status, s_lz, &pre,
                                             &words, &xk);
    if (threadIdx.x == 0) s_dec = dw;
  }
  __syncthreads();
  const Decision d = s_dec;
  const bool has_q = d.n < bs - 1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nseg = nchunk * kSegsPerChunk;
  const T* prow = lt + static_cast<size_t>(b * bs + d.n) * V;
  const T* qrow = has_q ? ld + static_cast<size_t>(b * (bs - 1) + d.n) * V : nullptr;
  for (int c = cb * kFinishChunks; c < min(nchunk, (cb + 1) * kFinishChunks); ++c) {
    // masses of max(0, p - q) and of p over this warp's segment of row n, in
    // kResidParts passes: fewer live registers, so that four CTAs fit on an
    // SM and the whole grid is resident at once
    constexpr int NP = kPerThread / VEC / kResidParts;
    const int s0 = c * kChunk + warp * kSeg, s1 = min(V, s0 + kSeg);
    float sr = 0.f, sp = 0.f;
#pragma unroll 1
    for (int h = 0; h < kResidParts; ++h) {
      typename Vec<T, VEC>::type vt[NP], vq[NP];
      bool live[NP];
      const int h0 = s0 + h * NP * 32 * VEC;
      load_seg<T, VEC, NP>(prow, h0, s1, lane, vt, live);
      if (has_q) load_seg<T, VEC, NP>(qrow, h0, s1, lane, vq, live);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        if (!live[i]) continue;
        float ft[VEC], fq[VEC];
        Vec<T, VEC>::unpack(vt[i], ft);
        if (has_q) Vec<T, VEC>::unpack(vq[i], fq);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          if (ft[j] == -INFINITY) continue;  // a -inf logit: zero mass
          float pw;
          const float r = resid_weight(ft[j] * scale, has_q ? fq[j] * scale : 0.f, d, has_q, pw);
          sr += r;
          sp += pw;
        }
      }
    }
    sr = warp_sum(sr);
    sp = warp_sum(sp);
    if (lane == 0 && s0 < V) rpart[static_cast<size_t>(b) * nseg + c * kSegsPerChunk + warp] = make_float2(sr, sp);
  }
  if (lane == 0) __threadfence();  // this warp's masses, visible before the CTA's count below
  __syncthreads();
  // The count is an acquire-release add: the last CTA's thread 0 then sees
  // every other CTA's masses, and the barrier passes that on to its threads.
  if (threadIdx.x == 0) s_is_last = atom_add_acq_rel_gpu(counters + b, 1) == ncb - 1;
  __syncthreads();
  if (!s_is_last) return;
  // the last CTA of the sequence: inverse-CDF search over row n, first over
  // the segment masses (one warp, vocabulary order), then inside the segment
  __shared__ int s_seg;
  __shared__ int s_use_p;
  __shared__ float s_target;
  __shared__ float s_wsum[kThreads / 32];
  __shared__ int s_pick;
  __shared__ int s_last;
  const int nseg_live = (V + kSeg - 1) / kSeg;
  if (warp == 0) {
    const float2* rp = rpart + static_cast<size_t>(b) * nseg;
    int cs = -1;
    float excl_cs = 0.f, t = 0.f;
    bool use_p = false;
    constexpr int kKeep = 8;  // segment masses per lane held in registers (V up to 32 * kKeep * kSeg)
    if (nseg_live <= 32 * kKeep) {
      // lane l holds the k contiguous segments l*k .. l*k + k - 1: one warp
      // scan of the lane totals finds the lane, a scan of its k masses the segment
      const int k = (nseg_live + 31) / 32;
      float wr[kKeep], wp[kKeep];
      float lr = 0.f, lp = 0.f;
#pragma unroll
      for (int j = 0; j < kKeep; ++j) {
        const int g = lane * k + j;
        const float2 v = (j < k && g < nseg_live) ? __ldcg(rp + g) : make_float2(0.f, 0.f);
        wr[j] = v.x;
        wp[j] = v.y;
        lr += v.x;
        lp += v.y;
      }
      float ir = lr, ip = lp;  // inclusive scans of the lane totals
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float ur = __shfl_up_sync(0xffffffffu, ir, o);
        const float up = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
          ir += ur;
          ip += up;
        }
      }
      use_p = !(__shfl_sync(0xffffffffu, ir, 31) > 0.f);
      t = uniform24(d.vbits) * __shfl_sync(0xffffffffu, use_p ? ip : ir, 31);
      const float L = use_p ? lp : lr;
      const float ex = (use_p ? ip : ir) - L;  // mass of the lanes ahead
      const unsigned hit = __ballot_sync(0xffffffffu, L > 0.f && ex + L > t);
      const unsigned pos = __ballot_sync(0xffffffffu, L > 0.f);
      // the first lane whose segments reach t; if rounding left t past the
      // end, the last lane holding mass (and in it its last positive segment)
      const int lsel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
      int pick = -1;
      float excl = 0.f;
      if (lane == lsel) {
        float run = ex, ex_last = 0.f;
        int last = -1;
#pragma unroll
        for (int j = 0; j < kKeep; ++j) {
          const float w = use_p ? wp[j] : wr[j];
          if (j < k && w > 0.f) {
            if (pick < 0 && hit && run + w > t) {
              pick = j;
              excl = run;
            }
            last = j;
            ex_last = run;
          }
          run += w;
        }
        if (pick < 0) {
          pick = last;
          excl = ex_last;
        }
      }
      if (lsel >= 0) {
        pick = __shfl_sync(0xffffffffu, pick, lsel);
        excl = __shfl_sync(0xffffffffu, excl, lsel);
        cs = lsel * k + max(pick, 0);
        excl_cs = pick >= 0 ? excl : 0.f;
      } else {
        cs = 0;
      }
    } else {  // longer rows: groups of 32 segments in turn, read again for the scan
      float sr = 0.f, sp = 0.f;
      for (int g = lane; g < nseg_live; g += 32) {
        const float2 v = __ldcg(rp + g);
        sr += v.x;
        sp += v.y;
      }
      sr = warp_sum(sr);
      sp = warp_sum(sp);
      use_p = !(sr > 0.f);
      t = uniform24(d.vbits) * (use_p ? sp : sr);
      float before = 0.f;  // mass of the segments ahead of this group of 32
      int last_pos = -1;
      float excl_last = 0.f;
      for (int g0 = 0; g0 < nseg_live && cs < 0; g0 += 32) {
        const int g = g0 + lane;
        float w = 0.f;
        if (g < nseg_live) {
          const float2 v = __ldcg(rp + g);
          w = use_p ? v.y : v.x;
        }
        float inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += u;
        }
        const float ex = before + (inc - w);
        const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && ex + w > t);
        const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
        if (hit) {
          const int l = __ffs(hit) - 1;
          cs = g0 + l;
          excl_cs = __shfl_sync(0xffffffffu, ex, l);
        }
        if (pos) {
          const int l = 31 - __clz(pos);
          last_pos = g0 + l;
          excl_last = __shfl_sync(0xffffffffu, ex, l);
        }
        before += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (cs < 0) {  // rounding left the threshold at the very end
        cs = max(last_pos, 0);
        excl_cs = last_pos >= 0 ? excl_last : 0.f;
      }
    }
    if (lane == 0) {
      s_seg = cs;
      s_use_p = use_p;
      s_target = fmaxf(0.f, t - excl_cs);
      s_pick = INT_MAX;
      s_last = -1;
    }
  }
  __syncthreads();
  const bool use_p = s_use_p != 0;
  const float target = s_target;
  const int seg0 = s_seg * kSeg;
  // kSeg / kThreads = 8 consecutive logits per thread, in vocabulary order
  constexpr int kEach = kSeg / kThreads;
  const int q0 = seg0 + threadIdx.x * kEach;
  float w[kEach];
  {
    const bool with_q = has_q && !use_p;
    constexpr int NV = kEach / VEC;
    using VT = typename Vec<T, VEC>::type;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = q0 + i * VEC;
      float fp[VEC], fq[VEC];
      const bool in = e < V;
      if (in) {
        Vec<T, VEC>::unpack(*reinterpret_cast<const VT*>(prow + e), fp);
        if (with_q) Vec<T, VEC>::unpack(*reinterpret_cast<const VT*>(qrow + e), fq);
      }
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        float pw;
        w[i * VEC + j] = (!in || fp[j] == -INFINITY) ? 0.f
                         : with_q ? resid_weight(fp[j] * scale, fq[j] * scale, d, true, pw)
                                  : ex2_approx(fp[j] * scale - d.lzp);
      }
    }
  }
  float mine = 0.f;
  int last_pos = -1;
#pragma unroll
  for (int i = 0; i < kEach; ++i) {
    if (w[i] > 0.f) last_pos = q0 + i;
    mine += w[i];
  }
  // exclusive scan of the threads' masses: within the warp, then across warps
  float inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) s_wsum[warp] = inc;
  if (last_pos >= 0) atomicMax(&s_last, last_pos);
  __syncthreads();
  float wbefore = 0.f;
  for (int i = 0; i < warp; ++i) wbefore += s_wsum[i];
  const float excl = wbefore + (inc - mine);
  if (mine > 0.f && excl <= target && target < excl + mine) {
    float run = excl;
    int pick = -1;
    bool done = false;
#pragma unroll
    for (int i = 0; i < kEach; ++i) {
      if (!done && w[i] > 0.f) {
        pick = q0 + i;  // last positive so far: fallback if rounding runs out
        run += w[i];
        done = run > target;
      }
    }
    if (pick >= 0) atomicMin(&s_pick, pick);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int y = s_pick;
    if (y == INT_MAX) y = s_last >= 0 ? s_last : seg0;
    out[b * bs + d.n] = y;
  }
}

int pick_vec(dflash_dtype dt, int V, const void* a, const void* b) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b);
  if (dt == DFLASH_BF16) return (V % 8 == 0 && (al & 15) == 0) ? 8 : 1;
  return (V % 4 == 0 && (al & 15) == 0) ? 4 : 1;
}

template <typename T, int VEC>
dflash_status run(const T* lt, const T* ld, const int32_t* x, int B, int bs, int V, float Temp,
                  uint64_t seed, uint64_t cycle, int32_t* acc, int32_t* out, void* ws,
                  cudaStream_t st, const DeviceInfo& dev) {
  const int nchunk = (V + kChunk - 1) / kChunk;
  const bool greedy = (Temp == 0.0f);
  const int R = greedy ? B * bs : B * bs + B * (bs - 1);
  WsCarver w(ws);
  float2* part = w.take<float2>(static_cast<size_t>(2 * B * bs) * nchunk);
  float2* rpart = w.take<float2>(static_cast<size_t>(B) * nchunk * kSegsPerChunk);
  int* counters = w.take<int>(B);
  const float scale = greedy ? 1.f : kLog2e / Temp;
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  const uint32_t c0 = static_cast<uint32_t>(cycle), c1 = static_cast<uint32_t>(cycle >> 32);
  const unsigned g1 = static_cast<unsigned>(nchunk) * static_cast<unsigned>(R);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t sc = {};  // the stats pass, a programmatic dependent of the preceding kernel
  sc.gridDim = dim3(g1);
  sc.blockDim = dim3(kThreads);
  sc.stream = st;
  sc.attrs = attr;
  sc.numAttrs = 1;
  if (greedy) {
    cudaError_t le = cudaLaunchKernelEx(&sc, verify_stats_kernel<T, VEC, true>, lt, ld, B, bs, V, nchunk, scale, part,
                                        static_cast<int*>(nullptr));
    if (le != cudaSuccess) return cuda_fail(le, "verify_stats_kernel launch");
    verify_decide_kernel<T><<<(B + 3) / 4, 128, 0, st>>>(lt, x, B, bs, V, nchunk, part, acc, out, dev.status);
  } else {
    cudaError_t le0 = cudaLaunchKernelEx(&sc, verify_stats_kernel<T, VEC, false>, lt, ld, B, bs, V, nchunk, scale, part,
                                         counters);
    if (le0 != cudaSuccess) return cuda_fail(le0, "verify_stats_kernel launch");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((nchunk + kFinishChunks - 1) / kFinishChunks) * static_cast<unsigned>(B));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le = cudaLaunchKernelEx(&cfg, verify_finish_kernel<T, VEC>, lt, ld, x, B, bs, V, nchunk, scale,
                                        static_cast<const float2*>(part), k0, k1, c0, c1, acc, out, rpart, counters,
                                        dev.status);
    if (le != cudaSuccess) return cuda_fail(le, "verify_finish_kernel launch");
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "verify kernel launch");
}

}  // namespace

size_t verify_ws_bytes(int B, int bs, int V) {
  const size_t nchunk = (static_cast<size_t>(V) + kChunk - 1) / kChunk;
  return align256(2 * static_cast<size_t>(B) * bs * nchunk * sizeof(float2)) +
         align256(static_cast<size_t>(B) * nchunk * kSegsPerChunk * sizeof(float2)) +
         align256(static_cast<size_t>(B) * sizeof(int)) + 256;
}

dflash_status launch_verify(const void* lt, const void* ld, dflash_dtype dt, const int32_t* x, int B,
                            int bs, int V, float T, uint64_t seed, uint64_t cycle, int32_t* acc,
                            int32_t* out, void* ws, cudaStream_t st, const DeviceInfo& dev) {
  const bool greedy = (T == 0.0f);
  const double rows = greedy ? double(B) * bs : double(B) * (2 * bs - 1);
  if (rows * ((V + kChunk - 1) / kChunk) >= 2147483647.0)
    return fail(DFLASH_ERR_UNSUPPORTED, "verify: too many logit chunks for one launch");
  if (greedy) ld = lt;  // draft rows are never read under greedy decoding
  const int vec = pick_vec(dt, V, lt, ld);
  if (dt == DFLASH_BF16) {
    auto* a = static_cast<const __nv_bfloat16*>(lt);
    auto* b = static_cast<const __nv_bfloat16*>(ld);
    return vec == 8 ? run<__nv_bfloat16, 8>(a, b, x, B, bs, V, T, seed, cycle, acc, out, ws, st, dev)
                    : run<__nv_bfloat16, 1>(a, b, x, B, bs, V, T, seed, cycle, acc, out, ws, st, dev);
  }
  auto* a = static_cast<const float*>(lt);
  auto* b = static_cast<const float*>(ld);
  return vec == 4 ? run<float, 4>(a, b, x, B, bs, V, T, seed, cycle, acc, out, ws, st, dev)
                  : run<float, 1>(a, b, x, B, bs, V, T, seed, cycle, acc, out, ws, st, dev);
}

}  // namespace dflash
