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
//               query head and block key, rounded to the storage dtype.
//   main     -- split-KV, memory-bound: a persistent grid walks work items
//               (sequence, KV head, key split).  A producer warp streams 64-key
//               K and V tiles of the cache with TMA (128-byte swizzle) through
//               a ring of shared-memory stages; four consumer warps compute
//               S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 -> fp32) for
//               all Hq/Hkv query heads x bs block rows of the KV head at once,
//               with an online softmax reduced by warp shuffles.  The last split
//               of each (sequence, KV head) also takes the bs block keys.
//   combine  -- log-sum-exp merge of the per-split partial outputs.
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
constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfTileBytes = kTile * 64 * 2;  // 64 keys x 64 dims bf16 = 8 KB (one TMA box)
constexpr int kStageBytes = 4 * kHalfTileBytes; // K (2 boxes) + V (2 boxes) = 32 KB
constexpr int kMergeSlotFloats = 16 * HD + 32;  // O[16][128], m[16], l[16]
constexpr int kMaxBatch = 4096;
constexpr double kTwoPi = 6.283185307179586476925286766559;

struct InvFreq {
  double v[HD / 2];
};

struct AttnParams {
  int B, bs, G, Hkv, Hq, cap, layer, window, chunk, max_splits, rows, n_mt, n_wg;
  const int32_t* seq_len;
  const __nv_bfloat16* qh;   // [B, Hq, bs, 128]   prologue output
  const __nv_bfloat16* kbh;  // [B, Hkv, bs, 128]  prologue output
  const __nv_bfloat16* vb;   // [B, Hkv, bs, 128]  block values (input)
  __nv_bfloat16* out;        // [B, Hq, bs, 128]
  float* opart;              // [B, Hkv, max_splits, rows, 128] normalised partial outputs
  float2* mlpart;            // [B, Hkv, max_splits, rows]      (max, sum) in log2 units
  float scale_log2;          // log2(e) / sqrt(128)
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
    unsigned* status) {
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
// main split-KV kernel (bf16)
// --------------------------------------------------------------------------

struct Item {
  int b, g, s, nsplit, kstart, kend, ntiles;
  bool last;
};

__device__ __forceinline__ Item decode_item(int w, const int* s_prefix, const int* s_n, const AttnParams& p) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {  // largest b with prefix[b] <= w
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= w) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.b = lo;
  const int n = s_n[lo];
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int ncache = n - first;
  it.nsplit = n_splits(ncache, p.chunk);
  const int r = w - s_prefix[lo];
  it.g = r / it.nsplit;
  it.s = r % it.nsplit;
  it.kstart = first + it.s * p.chunk;
  it.kend = first + min(ncache, (it.s + 1) * p.chunk);
  it.ntiles = it.kend > it.kstart ? (it.kend - it.kstart + kTile - 1) / kTile : 0;
  it.last = it.s == it.nsplit - 1;
  return it;
}

// Swizzled byte offset of (key row, 16-byte chunk c in 0..15) inside a K or V
// stage: two TMA boxes of 64 dims each, rows of 128 bytes, chunk ^= row & 7.
__device__ __forceinline__ uint32_t tile_off(int key, int c) {
  return static_cast<uint32_t>((c >> 3) * kHalfTileBytes + key * 128 + (((c & 7) ^ (key & 7)) << 4));
}

struct SoftmaxState {
  float m[2], l[2];
  float o[16][4];
};

// Online-softmax update of one warp's 16 rows with an S tile of NT*8 keys.
// s[j][0..1] belong to row lane/4, s[j][2..3] to row lane/4 + 8.  On return
// s holds p = 2^(s - m) (fp32) and the running state is rescaled.
template <int NT>
__device__ __forceinline__ void softmax_update(SoftmaxState& st, float (&s)[NT][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < NT; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * h], s[j][2 * h + 1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mnew = fmaxf(st.m[h], mx);
    const float muse = mnew == -INFINITY ? 0.f : mnew;
    const float corr = exp2f(st.m[h] - muse);
    st.m[h] = mnew;
    float rs = 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      s[j][2 * h] = exp2f(s[j][2 * h] - muse);
      s[j][2 * h + 1] = exp2f(s[j][2 * h + 1] - muse);
      rs += s[j][2 * h] + s[j][2 * h + 1];
    }
    st.l[h] = st.l[h] * corr + rs;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      st.o[n][2 * h] *= corr;
      st.o[n][2 * h + 1] *= corr;
    }
  }
}

// A fragments (m16 x k16) of P for keys [16*kk, 16*kk+16): P = hi + lo, both
// bf16, so the P V product keeps ~16 mantissa bits of each weight.
__device__ __forceinline__ void p_fragments(const float (&e)[4], const float (&o)[4], uint32_t (&hi)[4],
                                            uint32_t (&lo)[4]) {
  const float* src[4] = {&e[0], &e[2], &o[0], &o[2]};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float a = src[r][0], b = src[r][1];
    hi[r] = pack_bf16x2(a, b);
    lo[r] = pack_bf16x2(a - bf16_lo(hi[r]), b - bf16_hi(hi[r]));
  }
}

// One 64-key cache tile from shared memory.
__device__ __forceinline__ void process_cache_tile(SoftmaxState& st, const uint32_t (&qa)[8][4],
                                                   uint32_t kst, uint32_t vst, int nvalid,
                                                   float scale_log2, int lane) {
  float s[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  const int mi = lane >> 3;  // which 8x8 matrix this lane addresses
#pragma unroll
  for (int np = 0; np < 4; ++np) {
    const int key = 16 * np + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(kst + tile_off(key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
      mma_bf16_16816(s[2 * np], qa[kk], b0, b1);
      mma_bf16_16816(s[2 * np + 1], qa[kk], b2, b3);
    }
  }
  const int kc = 2 * (lane & 3);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = 8 * j + kc + (e & 1);
      s[j][e] = key < nvalid ? s[j][e] * scale_log2 : -INFINITY;
    }
  }
  softmax_update<8>(st, s);
#pragma unroll
  for (int kk2 = 0; kk2 < 4; ++kk2) {
    uint32_t ph[4], pl[4];
    p_fragments(s[2 * kk2], s[2 * kk2 + 1], ph, pl);
    const int key = 16 * kk2 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(vst + tile_off(key, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
      mma_bf16_16816(st.o[2 * dp], ph, b0, b1);
      mma_bf16_16816(st.o[2 * dp + 1], ph, b2, b3);
      mma_bf16_16816(st.o[2 * dp], pl, b0, b1);
      mma_bf16_16816(st.o[2 * dp + 1], pl, b2, b3);
    }
  }
}

// The bs (<= 16) block keys, read straight from global memory.
__device__ __forceinline__ void process_block_keys(SoftmaxState& st, const uint32_t (&qa)[8][4],
                                                   const __nv_bfloat16* __restrict__ kbh,
                                                   const __nv_bfloat16* __restrict__ vb, int bs,
                                                   float scale_log2, int lane) {
  float s[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  const int kc = 2 * (lane & 3);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int key = 8 * j + (lane >> 2);
    const uint32_t* kr = reinterpret_cast<const uint32_t*>(kbh + static_cast<size_t>(key) * HD);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t b0 = key < bs ? kr[(16 * kk + kc) / 2] : 0u;
      const uint32_t b1 = key < bs ? kr[(16 * kk + 8 + kc) / 2] : 0u;
      mma_bf16_16816(s[j], qa[kk], b0, b1);
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = 8 * j + kc + (e & 1);
      s[j][e] = key < bs ? s[j][e] * scale_log2 : -INFINITY;
    }
  }
  softmax_update<2>(st, s);
  uint32_t ph[4], pl[4];
  p_fragments(s[0], s[1], ph, pl);
  const unsigned short* vr = reinterpret_cast<const unsigned short*>(vb);
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) {
    const int dim = 8 * dn + (lane >> 2);
    const int k0 = kc, k1 = kc + 8;
    auto ld = [&](int key) -> uint32_t { return key < bs ? vr[static_cast<size_t>(key) * HD + dim] : 0u; };
    const uint32_t b0 = ld(k0) | (ld(k0 + 1) << 16);
    const uint32_t b1 = ld(k1) | (ld(k1 + 1) << 16);
    mma_bf16_16816(st.o[dn], ph, b0, b1);
    mma_bf16_16816(st.o[dn], pl, b0, b1);
  }
}

template <int STAGES>
__global__ void __launch_bounds__(kAttnThreads) attn_main_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap,
                                                                 const AttnParams p, int total_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  // layout: [stages x 32 KB][merge slots][prefix B+1][n B][full STAGES][empty STAGES]
  float* merge = reinterpret_cast<float*>(gbase + STAGES * kStageBytes);
  int* s_prefix = reinterpret_cast<int*>(merge + 4 * kMergeSlotFloats);
  int* s_n = s_prefix + (p.B + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(s_n + p.B) + 7) & ~uintptr_t(7));
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, p.n_mt);
    }
    mbar_fence_init();
  }
  if (warp == 0) {  // per-sequence lengths and the work-item prefix
    for (int b = lane; b < p.B; b += 32) s_n[b] = clamp_seq(p.seq_len[b], p.cap, p.status);
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int b = 0; b < p.B; ++b) {
        s_prefix[b] = acc;
        const int first = p.window > 0 ? max(0, s_n[b] - p.window) : 0;
        acc += n_splits(s_n[b] - first, p.chunk) * p.Hkv;
      }
      s_prefix[p.B] = acc;
    }
  }
  __syncthreads();
  const int n_items = min(total_items, s_prefix[p.B]);  // items that exist for these lengths

  if (warp == kConsumerWarps) {
    // ---------------- producer: TMA K/V tiles into the stage ring ----------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      const uint64_t pol = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
        const Item it = decode_item(w, s_prefix, s_n, p);
        const int rowbase = ((p.layer * p.B + it.b) * p.Hkv + it.g) * p.cap;
        for (int t = 0; t < it.ntiles; ++t) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.status)) return;
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint32_t dst = base + stage * kStageBytes;
          const int y = rowbase + it.kstart + t * kTile;
          tma_load_2d_hint(dst, &kmap, fb, 0, y, pol);
          tma_load_2d_hint(dst + kHalfTileBytes, &kmap, fb, 64, y, pol);
          tma_load_2d_hint(dst + 2 * kHalfTileBytes, &vmap, fb, 0, y, pol);
          tma_load_2d_hint(dst + 3 * kHalfTileBytes, &vmap, fb, 64, y, pol);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    return;  // the producer takes no part in the consumers' named barriers
  }

  // ---------------- consumers ------------------------------------------------
  const int mt = warp % p.n_mt;
  const int wg = warp / p.n_mt;
  const bool active = warp < p.n_mt * p.n_wg;
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    const Item it = decode_item(w, s_prefix, s_n, p);
    SoftmaxState st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
    uint32_t qa[8][4];
    {
      const size_t qrow0 = (static_cast<size_t>(it.b) * p.Hq + it.g * p.G) * p.bs;
      const int r0 = mt * 16 + (lane >> 2), r1 = r0 + 8;
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(p.qh + (qrow0 + r0) * HD);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(p.qh + (qrow0 + r1) * HD);
      const int kc = 2 * (lane & 3);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = r0 < p.rows ? q0[(16 * kk + kc) / 2] : 0u;
        qa[kk][1] = r1 < p.rows ? q1[(16 * kk + kc) / 2] : 0u;
        qa[kk][2] = r0 < p.rows ? q0[(16 * kk + 8 + kc) / 2] : 0u;
        qa[kk][3] = r1 < p.rows ? q1[(16 * kk + 8 + kc) / 2] : 0u;
      }
    }
    for (int t = 0; t < it.ntiles; ++t) {
      if (active && ok && (t % p.n_wg) == wg) {
        ok = mbar_wait(full0 + 8 * stage, phase, p.status);
        if (ok) {
          const uint32_t kst = base + stage * kStageBytes;
          const int nvalid = min(kTile, it.kend - (it.kstart + t * kTile));
          process_cache_tile(st, qa, kst, kst + 2 * kHalfTileBytes, nvalid, p.scale_log2, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      }
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (it.last && active && wg == 0) {
      const size_t kb0 = (static_cast<size_t>(it.b) * p.Hkv + it.g) * p.bs * HD;
      process_block_keys(st, qa, p.kbh + kb0, p.vb + kb0, p.bs, p.scale_log2, lane);
    }
    // ---- merge the warp groups' partial softmax states through shared memory
    named_barrier_sync(1, kConsumerWarps * 32);
    if (active) {
      float* slot = merge + (wg * p.n_mt + mt) * kMergeSlotFloats;
      float l0 = st.l[0], l1 = st.l[1];
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      const int r0 = lane >> 2, kc = 2 * (lane & 3);
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        slot[r0 * HD + 8 * n + kc] = st.o[n][0];
        slot[r0 * HD + 8 * n + kc + 1] = st.o[n][1];
        slot[(r0 + 8) * HD + 8 * n + kc] = st.o[n][2];
        slot[(r0 + 8) * HD + 8 * n + kc + 1] = st.o[n][3];
      }
      if ((lane & 3) == 0) {
        slot[16 * HD + r0] = st.m[0];
        slot[16 * HD + r0 + 8] = st.m[1];
        slot[16 * HD + 16 + r0] = l0;
        slot[16 * HD + 16 + r0 + 8] = l1;
      }
    }
    named_barrier_sync(1, kConsumerWarps * 32);
    const bool single = it.nsplit == 1;
    const size_t part_row0 = ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.max_splits + it.s) * p.rows;
    const size_t out_row0 = (static_cast<size_t>(it.b) * p.Hq + it.g * p.G) * p.bs;
    for (int idx = threadIdx.x; idx < p.rows * HD; idx += kConsumerWarps * 32) {
      const int row = idx / HD, e = idx % HD;
      const int rmt = row / 16, rr = row % 16;
      float M = -INFINITY;
      for (int g2 = 0; g2 < p.n_wg; ++g2)
        M = fmaxf(M, merge[(g2 * p.n_mt + rmt) * kMergeSlotFloats + 16 * HD + rr]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f, O = 0.f;
      for (int g2 = 0; g2 < p.n_wg; ++g2) {
        const float* sl = merge + (g2 * p.n_mt + rmt) * kMergeSlotFloats;
        const float f = exp2f(sl[16 * HD + rr] - Mu);
        L += sl[16 * HD + 16 + rr] * f;
        O += sl[rr * HD + e] * f;
      }
      const float val = L > 0.f ? O / L : 0.f;
      if (single) {
        p.out[(out_row0 + row) * HD + e] = __float2bfloat16_rn(val);
      } else {
        p.opart[(part_row0 + row) * HD + e] = val;
        if (e == 0) p.mlpart[part_row0 + row] = make_float2(M, L);
      }
    }
  }
}

constexpr int kCombineThreads = 256;

// Log-sum-exp merge of the split partials of one (sequence, KV head): one warp
// per output row, each lane owning 4 of the 128 dims.
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const AttnParams p) {
  const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
  const int n = min(max(p.seq_len[b], 0), p.cap);
  const int first = p.window > 0 ? max(0, n - p.window) : 0;
  const int ns = n_splits(n - first, p.chunk);
  if (ns <= 1) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t part0 = (static_cast<size_t>(b) * p.Hkv + g) * p.max_splits * p.rows;
  const size_t out_row0 = (static_cast<size_t>(b) * p.Hq + g * p.G) * p.bs;
  for (int row = warp; row < p.rows; row += kCombineThreads / 32) {
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.mlpart[part0 + static_cast<size_t>(s) * p.rows + row].x);
    M = warp_max(M);
    const float Mu = M == -INFINITY ? 0.f : M;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
#pragma unroll 4
    for (int s = 0; s < ns; ++s) {
      const size_t r = part0 + static_cast<size_t>(s) * p.rows + row;
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
    uint2 packed = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    reinterpret_cast<uint2*>(p.out + (out_row0 + row) * HD)[lane] = packed;
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

constexpr int kStages = 4;

size_t attn_main_smem(int B) {
  return 1024 + static_cast<size_t>(kStages) * kStageBytes + 4 * kMergeSlotFloats * sizeof(float) +
         (2 * static_cast<size_t>(B) + 1) * sizeof(int) + 8 + 16 * kStages;
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
         align256(static_cast<size_t>(B) * Hkv * max_splits * rows * sizeof(float2));
  return s + 256;
}

dflash_status launch_block_attn(int layer, int B, int bs, int Hq, const void* q, const void* kb,
                                const void* vb, const void* qg, const void* kg, float theta,
                                float eps, const dflash_kv_cache& c, int window, void* out, void* ws,
                                cudaStream_t st, const DeviceInfo& dev) {
  if (B > kMaxBatch) return fail(DFLASH_ERR_UNSUPPORTED, "block_attn: batch must be <= 4096");
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
        static_cast<const float*>(kg), c.seq_len, B, bs, Hq, Hkv, c.capacity, eps, inv, qh, kbh,
        dev.status);
    attn_f32_kernel<<<B * Hq, 128, 0, st>>>(qh, kbh, static_cast<const float*>(vb),
                                            static_cast<const float*>(c.k), static_cast<const float*>(c.v),
                                            c.seq_len, B, bs, Hq, Hkv, c.capacity, layer, window, scale,
                                            static_cast<float*>(out));
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "fp32 block attention launch");
  }
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
  p.n_mt = (p.rows + 15) / 16;
  p.n_wg = p.n_mt == 3 ? 1 : 4 / p.n_mt;
  p.seq_len = c.seq_len;
  auto* qh = w.take<__nv_bfloat16>(static_cast<size_t>(B) * Hq * bs * HD);
  auto* kbh = w.take<__nv_bfloat16>(static_cast<size_t>(B) * Hkv * bs * HD);
  p.qh = qh;
  p.kbh = kbh;
  p.vb = static_cast<const __nv_bfloat16*>(vb);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.opart = w.take<float>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows * HD);
  p.mlpart = w.take<float2>(static_cast<size_t>(B) * Hkv * p.max_splits * p.rows);
  p.scale_log2 = 1.4426950408889634f * scale;
  p.status = dev.status;

  CUtensorMap kmap, vmap;
  const uint64_t rows = static_cast<uint64_t>(c.num_layers) * c.batch * Hkv * c.capacity;
  dflash_status s = make_tmap_bf16_2d(&kmap, c.k, rows, HD, kTile, 64);
  if (s) return s;
  s = make_tmap_bf16_2d(&vmap, c.v, rows, HD, kTile, 64);
  if (s) return s;

  attn_prologue_kernel<__nv_bfloat16><<<B * bs, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kb),
      static_cast<const __nv_bfloat16*>(qg), static_cast<const __nv_bfloat16*>(kg), c.seq_len, B, bs,
      Hq, Hkv, c.capacity, eps, inv, qh, kbh, dev.status);

  const size_t smem = attn_main_smem(B);
  if (smem > dev.max_smem_optin) return fail(DFLASH_ERR_UNSUPPORTED, "block_attn: shared memory");
  static int configured_device = -1;
  if (configured_device != dev.device) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_kernel<kStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(dev.max_smem_optin));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_main_kernel)");
    configured_device = dev.device;
  }
  const long upper = static_cast<long>(B) * Hkv * p.max_splits;
  const int grid = static_cast<int>(std::min<long>(upper, dev.num_sms));
  attn_main_kernel<kStages><<<grid, kAttnThreads, smem, st>>>(kmap, vmap, p, static_cast<int>(upper));
  attn_combine_kernel<<<B * Hkv, kCombineThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "block attention launch");
}

}  // namespace dflash
