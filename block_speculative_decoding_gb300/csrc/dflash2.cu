// DFlash2 variants: the local depthwise convolution along the draft block and
// the candidate path selector's per-position statistics.
//
// Page: "DFlash & DFlash2: Block-Diffusion LLM-Speedup", section 5 (DFlash2
// innovations): 5.1 depthwise 1D convolutions of kernel width k in {3, 5}
// between the drafter's attention and feed-forward sub-layers,
// ConvOutput_t = sum_j W_conv,j (.) H_{t-j} + b_conv; 5.2 the draft head's
// top-m candidates per block position and the path score
// S = sum_j log P_draft(x_j^(m_j)) + lambda * Entropy(P_draft(x_j)).
//
// Kernels:
//   block_conv_kernel  one thread per (sequence, 4 channels): the block's rows
//                      of those channels in registers, the causal depthwise
//                      sum, bf16 out (in place allowed).
//   topm_chunk_kernel  one CTA per (row, 16384-logit chunk; four per SM): the chunk's
//                      (max, sum e^(s-max), sum e^(s-max) (s-max)) of s = l / T
//                      and its m best logits (ties to the lower index).
//   topm_merge_kernel  one CTA per sequence, one warp per row: the row's
//                      log-normaliser and entropy from the chunk triples, its
//                      m best candidates from the chunks' candidates, their
//                      log-probabilities, and the sequence's best-path score.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <climits>

#include "dflash_device.cuh"
#include "dflash_internal.h"

namespace dflash {
namespace {

constexpr int kConvMaxBlock = 16;
constexpr int kConvMaxK = 8;

// h, out [B * bs, D] bf16 (sequence-major rows, out may be h); w [k, D] bf16;
// bias [D] bf16 or null.  out_t = sum_{j < k, j <= t} w_j * h_{t-j} + b
// (+ h_t if residual), t the row's position in its block.  One thread per
// (sequence, 4 channels).
__global__ void __launch_bounds__(256) block_conv_kernel(const __nv_bfloat16* h, int B, int bs, int D, int k,
                                                         const __nv_bfloat16* __restrict__ w,
                                                         const __nv_bfloat16* __restrict__ bias, int residual,
                                                         __nv_bfloat16* out) {
  const int groups = D / 4;
  const long t = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<long>(B) * groups) return;
  const int b = static_cast<int>(t / groups), c0 = static_cast<int>(t % groups) * 4;
  float x[kConvMaxBlock][4];
#pragma unroll
  for (int r = 0; r < kConvMaxBlock; ++r) {
    if (r >= bs) continue;
    const uint2 v = *reinterpret_cast<const uint2*>(h + (static_cast<size_t>(b) * bs + r) * D + c0);
    x[r][0] = bf16_lo(v.x);
    x[r][1] = bf16_hi(v.x);
    x[r][2] = bf16_lo(v.y);
    x[r][3] = bf16_hi(v.y);
  }
  float wk[kConvMaxK][4];
#pragma unroll
  for (int j = 0; j < kConvMaxK; ++j) {
    if (j >= k) continue;
    const uint2 v = *reinterpret_cast<const uint2*>(w + static_cast<size_t>(j) * D + c0);
    wk[j][0] = bf16_lo(v.x);
    wk[j][1] = bf16_hi(v.x);
    wk[j][2] = bf16_lo(v.y);
    wk[j][3] = bf16_hi(v.y);
  }
  float bv[4] = {0.f, 0.f, 0.f, 0.f};
  if (bias) {
    const uint2 v = *reinterpret_cast<const uint2*>(bias + c0);
    bv[0] = bf16_lo(v.x);
    bv[1] = bf16_hi(v.x);
    bv[2] = bf16_lo(v.y);
    bv[3] = bf16_hi(v.y);
  }
  // every input row is in registers before the first store, so out may be h
#pragma unroll
  for (int r = 0; r < kConvMaxBlock; ++r) {
    if (r >= bs) continue;
    float acc[4] = {bv[0], bv[1], bv[2], bv[3]};
#pragma unroll
    for (int j = 0; j < kConvMaxK; ++j) {
      if (j >= k || j > r) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(wk[j][i], x[r - j][i], acc[i]);
    }
    if (residual) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += x[r][i];
    }
    *reinterpret_cast<uint2*>(out + (static_cast<size_t>(b) * bs + r) * D + c0) =
        make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
  }
}

constexpr int kTopmThreads = 256;
constexpr int kTopmChunk = 16384;                       // logits per chunk CTA
constexpr int kTopmVecs = kTopmChunk / (kTopmThreads * 8);  // 8 vectors of 8 bf16 per thread
constexpr int kMaxM = 8;
constexpr int kTopmBuf = 128;                            // compacted candidates per warp
constexpr int kTopmVecCap = 32;                          // staged 8-logit vectors per warp

// (value, index) order of the candidates: larger logit first, then lower index.
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Warp-wide best (value, index); every lane gets it.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Bitonic sort of the warp's 32 keys, best first (lane 0 ends with the best):
// in every compare-exchange the lower lane of a best-first run keeps the
// better key, of a worst-first run the worse one.
__device__ __forceinline__ void warp_sort_best_first(float& v, int& i, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oi = __shfl_xor_sync(0xffffffffu, i, j);
      const bool best_first = (lane & k) == 0 || k == 32;
      const bool lower = (lane & j) == 0;
      const bool take = (lower == best_first) ? better(ov, oi, v, i) : better(v, i, ov, oi);
      if (take) {
        v = ov;
        i = oi;
      }
    }
  }
}

// One CTA per (row, chunk).  stats[row][c] = (max s, sum e^(s - max),
// sum e^(s - max) (s - max), 0) over the chunk's finite logits, s = l * inv_t;
// cand[row][c][r] = (logit bits, index) of the chunk's r-th best logit.
__global__ void __launch_bounds__(kTopmThreads, 4) topm_chunk_kernel(const __nv_bfloat16* __restrict__ logits, int V,
                                                                 int nchunk, float inv_t, int m,
                                                                 float4* __restrict__ stats, int2* __restrict__ cand) {
  const int row = blockIdx.x / nchunk, c = blockIdx.x % nchunk;
  const __nv_bfloat16* lr = logits + static_cast<size_t>(row) * V;
  const int e0 = c * kTopmChunk;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  uint4 raw[kTopmVecs];
#pragma unroll
  for (int i = 0; i < kTopmVecs; ++i) {
    const int e = e0 + (i * kTopmThreads + tid) * 8;
    raw[i] = e < V ? __ldcs(reinterpret_cast<const uint4*>(lr + e)) : make_uint4(0xFF80FF80u, 0xFF80FF80u,
                                                                                0xFF80FF80u, 0xFF80FF80u);
  }
  // per vector, the largest of its 8 logits (packed bf16 maxima); this lane's
  // best key (value, lowest index with it) from the first vector holding it
  float vmax[kTopmVecs];
  float mv = -INFINITY;
#pragma unroll
  for (int i = 0; i < kTopmVecs; ++i) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&raw[i].x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&raw[i].y));
    const __nv_bfloat162 c2 = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&raw[i].z),
                                      *reinterpret_cast<const __nv_bfloat162*>(&raw[i].w));
    const __nv_bfloat162 d2 = __hmax2(a, c2);
    vmax[i] = fmaxf(__low2float(d2), __high2float(d2));
    mv = fmaxf(mv, vmax[i]);
  }
  int mi = INT_MAX;
#pragma unroll
  for (int i = 0; i < kTopmVecs; ++i) {
    if (mi == INT_MAX && vmax[i] == mv) {
      const uint32_t u[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
      const int e = e0 + (i * kTopmThreads + tid) * 8;
#pragma unroll
      for (int j = 7; j >= 0; --j)
        if (((j & 1) ? bf16_hi(u[j / 2]) : bf16_lo(u[j / 2])) == mv) mi = e + j;
    }
  }
  if (mv == -INFINITY) {  // all of the lane's logits are -inf: its key is its lowest index (none past V)
    const int first = e0 + tid * 8;
    mi = first < V ? first : INT_MAX;
  }
  const float mx = mv;
  // the warp's threshold tau: the m-th best of the 32 lane keys.  At least m
  // of the warp's elements have a key >= tau (in the total order of
  // better(): larger logit, then lower index), so its m best are among them.
  float tv = mv;
  int ti = mi;
  warp_sort_best_first(tv, ti, lane);
  tv = __shfl_sync(0xffffffffu, tv, m - 1);
  ti = __shfl_sync(0xffffffffu, ti, m - 1);
  // the warp's keys >= tau, appended to shared memory by the lanes holding
  // them (only vectors whose maximum reaches tau are looked into); few pass:
  // an all-equal row passes (m - 1) * 8 + 1 of them
  __shared__ int2 s_buf[kTopmThreads / 32][kTopmBuf];
  __shared__ int2 s_wcand[kTopmThreads / 32][kMaxM];
  __shared__ int s_cnt[kTopmThreads / 32];
  __shared__ uint4 s_vec[kTopmThreads / 32][kTopmVecCap];
  __shared__ int s_vbase[kTopmThreads / 32][kTopmVecCap];
  __shared__ int s_vcnt[kTopmThreads / 32];
  if (lane == 0) {
    s_cnt[warp] = 0;
    s_vcnt[warp] = 0;
  }
  __syncwarp();
  // stage the vectors whose maximum reaches tau (few), then test them with
  // eight lanes per vector, four vectors per step
#pragma unroll
  for (int i = 0; i < kTopmVecs; ++i) {
    if (vmax[i] >= tv) {
      const int k = atomicAdd(&s_vcnt[warp], 1);
      if (k < kTopmVecCap) {
        s_vec[warp][k] = raw[i];
        s_vbase[warp][k] = e0 + (i * kTopmThreads + tid) * 8;
      }
    }
  }
  __syncwarp();
  const int nvec = s_vcnt[warp];
  if (nvec <= kTopmVecCap) {
    for (int k0 = 0; k0 < nvec; k0 += 4) {
      const int k = k0 + lane / 8, j = lane % 8;
      if (k < nvec) {
        const uint4 q = s_vec[warp][k];
        const uint32_t w2 = j < 2 ? q.x : j < 4 ? q.y : j < 6 ? q.z : q.w;
        const float v = (j & 1) ? bf16_hi(w2) : bf16_lo(w2);
        const int idx = s_vbase[warp][k] + j;
        if (idx < V && !better(tv, ti, v, idx)) {
          const int pos = atomicAdd(&s_cnt[warp], 1);
          if (pos < kTopmBuf) s_buf[warp][pos] = make_int2(__float_as_int(v), idx);
        }
      }
    }
  } else {  // many vectors reach tau: every lane tests its own
#pragma unroll
    for (int i = 0; i < kTopmVecs; ++i) {
      if (vmax[i] >= tv) {
        const uint32_t u[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float v = (j & 1) ? bf16_hi(u[j / 2]) : bf16_lo(u[j / 2]);
          const int idx = e0 + (i * kTopmThreads + tid) * 8 + j;
          if (idx < V && !better(tv, ti, v, idx)) {
            const int pos = atomicAdd(&s_cnt[warp], 1);
            if (pos < kTopmBuf) s_buf[warp][pos] = make_int2(__float_as_int(v), idx);
          }
        }
      }
    }
  }
  __syncwarp();
  const int cnt = s_cnt[warp];
  // the warp's m best: one sort when they fit a warp, else m rounds over the
  // buffer, else (overflow) over the registers
  if (cnt <= 32) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (lane < cnt) {
      const int2 e = s_buf[warp][lane];
      bv = __int_as_float(e.x);
      bi = e.y;
    }
    warp_sort_best_first(bv, bi, lane);
    if (lane < m) s_wcand[warp][lane] = make_int2(__float_as_int(bv), bi);
  } else if (cnt <= kTopmBuf) {
    for (int r = 0; r < m; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX, bk = -1;
      for (int k = lane; k < cnt; k += 32) {
        const int2 e = s_buf[warp][k];
        if (better(__int_as_float(e.x), e.y, bv, bi)) {
          bv = __int_as_float(e.x);
          bi = e.y;
          bk = k;
        }
      }
      float wv = bv;
      int wi = bi;
      warp_best(wv, wi);
      if (bk >= 0 && bi == wi) s_buf[warp][bk] = make_int2(__float_as_int(-INFINITY), INT_MAX);
      if (lane == 0) s_wcand[warp][r] = make_int2(__float_as_int(wv), wi);
      __syncwarp();
    }
  } else {
    float pv = INFINITY;  // the previous round's winner: this round takes the best key after it
    int pi = -1;
    for (int r = 0; r < m; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      // (rare) re-read the lane's vectors rather than keep them live in registers
#pragma unroll 1
      for (int i = 0; i < kTopmVecs; ++i) {
        const int e = e0 + (i * kTopmThreads + tid) * 8;
        if (e >= V) continue;
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(lr + e));
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float v = (j & 1) ? bf16_hi(u[j / 2]) : bf16_lo(u[j / 2]);
          const int idx = e + j;
          if (better(pv, pi, v, idx) && better(v, idx, bv, bi)) {
            bv = v;
            bi = idx;
          }
        }
      }
      warp_best(bv, bi);
      if (lane == 0) s_wcand[warp][r] = make_int2(__float_as_int(bv), bi);
      pv = bv;
      pi = bi;
    }
  }
  __shared__ float s_red[kTopmThreads / 32][2];
  // the chunk's maximum of s = l * inv_t (inv_t > 0 keeps the order)
  float wm = warp_max(mx);
  if (lane == 0) s_red[warp][0] = wm;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kTopmThreads / 32; ++w) M = fmaxf(M, s_red[w][0]);
  const float Ms = M * inv_t;
  float S = 0.f, W = 0.f;
  if (M != -INFINITY) {
    // in base 2 and without branches: d2 = (s - max) log2(e), clamped so that a
    // -inf logit (zero probability, also the padding past V) adds e = 0 and
    // e * d2 = 0; W is converted back to natural units below
    const float k2 = inv_t * 1.4426950408889634f, m2 = Ms * 1.4426950408889634f;
#pragma unroll
    for (int i = 0; i < kTopmVecs; ++i) {
      const uint32_t u[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v = (j & 1) ? bf16_hi(u[j / 2]) : bf16_lo(u[j / 2]);
        const float d2 = fmaxf(fmaf(v, k2, -m2), -1.0e30f);
        const float e = ex2_approx(d2);
        S += e;
        W = fmaf(e, d2, W);
      }
    }
    W *= 0.6931471805599453f;
  }
  S = warp_sum(S);
  W = warp_sum(W);
  __syncthreads();  // every thread has read s_red[.][0]
  if (lane == 0) {
    s_red[warp][0] = S;
    s_red[warp][1] = W;
  }
  __syncthreads();
  if (tid == 0) {
    float St = 0.f, Wt = 0.f;
    for (int w = 0; w < kTopmThreads / 32; ++w) {
      St += s_red[w][0];
      Wt += s_red[w][1];
    }
    stats[static_cast<size_t>(row) * nchunk + c] = make_float4(Ms, St, Wt, 0.f);
  }
  // the chunk's m best from the warps' m best each: warp 0 sorts warps 0-3's
  // and warps 4-7's candidates (32 each), and a bitonic merge of the first
  // list with the reversed second keeps the 32 best in order
  __syncthreads();
  if (warp == 0) {
    constexpr int kW = kTopmThreads / 32;
    static_assert(kW == 8 && kMaxM == 8, "two lists of four warps' eight candidates");
    const int w_a = lane / kMaxM, r_a = lane % kMaxM;
    int2 ea = r_a < m ? s_wcand[w_a][r_a] : make_int2(__float_as_int(-INFINITY), INT_MAX);
    int2 eb = r_a < m ? s_wcand[w_a + 4][r_a] : make_int2(__float_as_int(-INFINITY), INT_MAX);
    float av = __int_as_float(ea.x), bvv = __int_as_float(eb.x);
    int ai = ea.y, bii = eb.y;
    warp_sort_best_first(av, ai, lane);
    warp_sort_best_first(bvv, bii, lane);
    // lane l pairs a[l] with b[31 - l]: the better of each pair forms a bitonic sequence of the 32 best
    const float rv = __shfl_sync(0xffffffffu, bvv, 31 - lane);
    const int ri = __shfl_sync(0xffffffffu, bii, 31 - lane);
    if (better(rv, ri, av, ai)) {
      av = rv;
      ai = ri;
    }
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, av, j);
      const int oi = __shfl_xor_sync(0xffffffffu, ai, j);
      const bool lower = (lane & j) == 0;
      if (lower ? better(ov, oi, av, ai) : better(av, ai, ov, oi)) {
        av = ov;
        ai = oi;
      }
    }
    if (lane < m) cand[(static_cast<size_t>(row) * nchunk + c) * m + lane] = make_int2(__float_as_int(av), ai);
  }
}

// One CTA per sequence, one warp per draft row r < R: the row's
// log-normaliser logZ = max + ln S and entropy ln S - W / S from the chunk
// triples, its m best candidates from the chunks' candidates with
// logp = l * inv_t - logZ, and the sequence's best-path score
// sum_r (logp of the first candidate) + lambda * sum_r entropy.
__global__ void __launch_bounds__(512) topm_merge_kernel(const float4* __restrict__ stats,
                                                        const int2* __restrict__ cand, int R, int nchunk, int m,
                                                        float inv_t, float lambda, int32_t* __restrict__ idx_out,
                                                        float* __restrict__ logp_out, float* __restrict__ ent_out,
                                                        float* __restrict__ score_out) {
  pdl_wait_primary();
  pdl_launch_dependents();
  stats = pdl_fresh(stats);
  cand = pdl_fresh(cand);
  const int b = blockIdx.x, warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __shared__ float s_part[16];
  if (warp < R) {
    const int row = b * R + warp;
    // log-normaliser and entropy: rescale every chunk's sums to the row maximum
    float M = -INFINITY;
    for (int c = lane; c < nchunk; c += 32) M = fmaxf(M, stats[static_cast<size_t>(row) * nchunk + c].x);
    M = warp_max(M);
    float S = 0.f, W = 0.f;
    if (M != -INFINITY) {
      for (int c = lane; c < nchunk; c += 32) {
        const float4 t = stats[static_cast<size_t>(row) * nchunk + c];
        if (t.x == -INFINITY) continue;
        const float f = __expf(t.x - M);
        S = fmaf(f, t.y, S);
        W = fmaf(f, t.z + (t.x - M) * t.y, W);
      }
    }
    S = warp_sum(S);
    W = warp_sum(W);
    const float logz = M + logf(S);
    const float ent = S > 0.f ? logf(S) - W / S : 0.f;
    // the m best of the nchunk * m chunk candidates (each lane holds up to
    // kMaxCand of them), m rounds of a warp arg-best with exclusion
    constexpr int kMaxCand = 8;  // nchunk * m <= 256
    float cv[kMaxCand];
    int ci[kMaxCand];
    const int ncand = nchunk * m;
#pragma unroll
    for (int q = 0; q < kMaxCand; ++q) {
      const int k = lane + 32 * q;
      cv[q] = -INFINITY;
      ci[q] = INT_MAX;
      if (k < ncand) {
        const int2 e = cand[static_cast<size_t>(row) * ncand + k];
        if (e.y != INT_MAX) {
          cv[q] = __int_as_float(e.x);
          ci[q] = e.y;
        }
      }
    }
    float first = 0.f;
    for (int r = 0; r < m; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int q = 0; q < kMaxCand; ++q)
        if (better(cv[q], ci[q], bv, bi)) {
          bv = cv[q];
          bi = ci[q];
        }
      warp_best(bv, bi);
#pragma unroll
      for (int q = 0; q < kMaxCand; ++q)
        if (ci[q] == bi) {
          cv[q] = -INFINITY;
          ci[q] = INT_MAX;
        }
      const float lp = (bi == INT_MAX || logz == -INFINITY) ? -INFINITY : bv * inv_t - logz;  // -inf row: no mass
      if (r == 0) first = lp;
      if (lane == 0) {
        idx_out[static_cast<size_t>(row) * m + r] = bi == INT_MAX ? -1 : bi;
        logp_out[static_cast<size_t>(row) * m + r] = lp;
      }
    }
    if (lane == 0) {
      ent_out[row] = ent;
      s_part[warp] = first + lambda * ent;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float sc = 0.f;
    for (int r = 0; r < R; ++r) sc += s_part[r];
    score_out[b] = sc;
  }
}

}  // namespace

dflash_status launch_block_conv(const void* h, int B, int bs, int D, int k, const void* w, const void* bias,
                                int residual, void* out, cudaStream_t st) {
  const long threads = static_cast<long>(B) * (D / 4);
  block_conv_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(h), B, bs, D, k, static_cast<const __nv_bfloat16*>(w),
      static_cast<const __nv_bfloat16*>(bias), residual, static_cast<__nv_bfloat16*>(out));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "block_conv_kernel launch");
}

size_t topm_ws_bytes(int B, int R, int V, int m) {
  const size_t rows = static_cast<size_t>(B) * R;
  const size_t nchunk = (static_cast<size_t>(V) + kTopmChunk - 1) / kTopmChunk;
  return align256(rows * nchunk * sizeof(float4)) + align256(rows * nchunk * m * sizeof(int2)) + 256;
}

int topm_max_m() { return kMaxM; }
int topm_max_chunks_times_m() { return 32 * 8; }

dflash_status launch_draft_topm(const void* logits, int B, int R, int V, int m, float T, float lambda,
                                int32_t* idx, float* logp, float* ent, float* score, void* ws, cudaStream_t st) {
  const int nchunk = (V + kTopmChunk - 1) / kTopmChunk;
  WsCarver w(ws);
  float4* stats = w.take<float4>(static_cast<size_t>(B) * R * nchunk);
  int2* cand = w.take<int2>(static_cast<size_t>(B) * R * nchunk * m);
  const float inv_t = 1.0f / T;
  topm_chunk_kernel<<<static_cast<unsigned>(static_cast<long>(B) * R * nchunk), kTopmThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(logits), V, nchunk, inv_t, m, stats, cand);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "topm_chunk_kernel launch");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(static_cast<unsigned>(32 * R));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topm_merge_kernel, static_cast<const float4*>(stats), static_cast<const int2*>(cand),
                         R, nchunk, m, inv_t, lambda, idx, logp, ent, score);
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "topm_merge_kernel launch");
}

}  // namespace dflash

