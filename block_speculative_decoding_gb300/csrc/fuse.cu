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
// bf16 path, three launches chained as programmatic dependents:
//   1. gemm_tc (fusion)  Y = [taps] W_c^T on tcgen05 tensor cores: a unit is
//      MT x 128 rows by 128 columns of Y over a range of K blocks; TMA loads
//      128x64 A tiles (taken from the tap that owns the K block -- the concat is
//      never materialised) and the 128x64 W_c tile into a ring, one thread
//      issues tcgen05.mma (M=128, N=128, K=16) into MT accumulators in tensor
//      memory, four epilogue warps drain them.  A few new rows (M <= 256) take
//      MT = 2, so each W_c tile is read once, and split K over ~one unit per
//      SM; the fp32 partial sums stay in the workspace.
//   2. rownorm           row -> (sequence, cache position) and its RoPE table
//      (before waiting for the GEMM), then H_t = bf16(sum_splits(Y) *
//      rsqrt(mean(Y^2) + eps) * g)
//   3. gemm_tc (K/V)     [K|V] = H_t W_kv^T, one head (128 columns) per unit, with
//      a fused epilogue: a K head is RMS-normalised (gain k_gain[l]) and rotated
//      at its cache position, a V head copied, both stored as bf16 cache rows.
//      Its producer loads the first W_kv tiles before waiting for H_t.
// fp32 path: the same steps as plain SIMT kernels (parity path).
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
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kGemmThreads = 192;  // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr int kMaxSeg = 8;
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
constexpr int kSplitTarget = 152;  // work units aimed for when splitting K (one per SM)

struct InvFreq {
  double v[HD / 2];
};

struct TmapPack {
  CUtensorMap a[kMaxSeg];
};

struct GemmArgs {
  int M, N, num_kb, kb_per_seg, k_splits, m_tiles, n_tiles;
  int stream_k;            // > 0: the number of shares (CTAs); CTA c takes the c-th near-equal share of the
                           // (tile, K block) space
  int dp_tiles;            // stream_k: leading tiles scheduled whole, a multiple of the share count
  int* pieces;             // stream_k: [m_tiles * n_tiles] number of slots written for the tile
  int epi;                 // 0: fp32 partial store, 1: K/V cache epilogue
  int pdl;                 // launched as a programmatic dependent (waits for the preceding grid before any load)
  int prefetch_b;          // the B operand (weights) may be loaded before that wait
  float* out_f32;          // epi 0: [k_splits][M][N]
  __nv_bfloat16* cache_k;  // epi 1
  __nv_bfloat16* cache_v;
  int L, Bc, Hkv, cap;
  const int2* rowinfo;     // [M] (sequence, cache row) or (-1, -1)
  const float2* rope_cs;   // [64][M] (cos, sin), element-major: a warp's rows read it coalesced
  const __nv_bfloat16* k_gain;  // [L][128] or null
  float eps;
  unsigned* status;
};

// A unit is MT x 128 rows by BN columns (over a range of K blocks); its MT
// accumulators of BN fp32 columns sit side by side in tensor memory, twice
// over (double-buffered) when that fits the 512 columns.
template <int BN, int MT>
__host__ __device__ constexpr int stage_bytes() {
  return MT * kBM * kBK * 2 + BN * kBK * 2;
}

template <int BN, int MT>
__host__ __device__ constexpr int num_acc() {
  return 2 * MT * BN <= 512 ? 2 : 1;
}

template <int BN, int STAGES, int MT>
constexpr size_t gemm_smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * stage_bytes<BN, MT>() + 8 * (2 * STAGES + 4) + 16;
}

__device__ __forceinline__ void unit_coords(int u, const GemmArgs& p, int& m, int& n, int& kb0, int& kb1,
                                            int& ks) {
  n = u % p.n_tiles;
  m = (u / p.n_tiles) % p.m_tiles;
  ks = u / (p.n_tiles * p.m_tiles);
  kb0 = static_cast<int>((static_cast<long>(ks) * p.num_kb) / p.k_splits);
  kb1 = static_cast<int>((static_cast<long>(ks + 1) * p.num_kb) / p.k_splits);
}

// The i-th K block a unit of N tile n works on: the range [kb0, kb1) rotated by
// a start spread over the N tiles, so the CTAs that share A blocks (the same
// rows, other N tiles) do not all request the same block at the same time.
// The sum is the same; only its rounding order differs.
__device__ __forceinline__ int kb_at(int i, int kb0, int kb1, int n, const GemmArgs& p) {
  const int nk = kb1 - kb0;
  const int rot = static_cast<int>((static_cast<long>(n) * nk) / p.n_tiles);
  int j = i + rot;
  if (j >= nk) j -= nk;
  return kb0 + j;
}

// The pieces of work of this CTA, in order.  Plain schedule: units
// blockIdx.x, blockIdx.x + gridDim.x, ... (a unit: one tile over one K split,
// its partial sum in slot = split index).  Stream-K schedule: the first
// dp_tiles tiles (a whole number of waves) go round-robin as whole tiles;
// the K blocks of the remaining tiles, laid end to end (tile-major, N tiles
// fastest), are cut into gridDim.x near-equal, non-empty contiguous shares
// [c tot / P, (c+1) tot / P), so K block x belongs to share ((x+1) P - 1) / tot.
// A tile met by shares c0..c1 gets one partial sum per share, in slot c - c0;
// the piece in slot 0 records the tile's slot count c1 - c0 + 1.  Keeping the
// leading waves whole keeps the CTAs in step along K (operand tiles shared in
// L2); only the tiles left over after the whole waves are balanced.
__device__ __forceinline__ long share_of(long x, long tot, long P) { return ((x + 1) * P - 1) / tot; }

struct Pieces {
  long cur, end;  // plain: unit cursor and count; stream-K: cursor in the balanced K-block range
  int dp_next;    // stream-K: next whole tile of this CTA
  int count = 1;  // stream-K, slot 0: the tile's slot count
  __device__ __forceinline__ explicit Pieces(const GemmArgs& p) {
    dp_next = blockIdx.x;
    if (p.stream_k) {
      const long tot = (static_cast<long>(p.m_tiles) * p.n_tiles - p.dp_tiles) * p.num_kb;
      cur = tot * blockIdx.x / gridDim.x;
      end = tot * (blockIdx.x + 1) / gridDim.x;
    } else {
      cur = blockIdx.x;
      end = static_cast<long>(p.m_tiles) * p.n_tiles * p.k_splits;
    }
  }
  __device__ __forceinline__ bool next(const GemmArgs& p, int& m, int& n, int& kb0, int& kb1, int& slot) {
    if (p.stream_k && dp_next < p.dp_tiles) {
      n = dp_next % p.n_tiles;
      m = dp_next / p.n_tiles;
      kb0 = 0;
      kb1 = p.num_kb;
      slot = 0;
      count = 1;
      dp_next += gridDim.x;
      return true;
    }
    if (cur >= end) return false;
    if (p.stream_k) {
      const long tr = cur / p.num_kb;  // tile index within the balanced range
      const long t = p.dp_tiles + tr;
      kb0 = static_cast<int>(cur - tr * p.num_kb);
      kb1 = static_cast<int>(min(static_cast<long>(p.num_kb), kb0 + (end - cur)));
      n = static_cast<int>(t % p.n_tiles);
      m = static_cast<int>(t / p.n_tiles);
      const long tot = (static_cast<long>(p.m_tiles) * p.n_tiles - p.dp_tiles) * p.num_kb;
      const long c0 = share_of(tr * p.num_kb, tot, gridDim.x);
      slot = static_cast<int>(blockIdx.x - c0);
      if (slot == 0) count = static_cast<int>(share_of((tr + 1) * p.num_kb - 1, tot, gridDim.x) - c0 + 1);
      cur += kb1 - kb0;
    } else {
      unit_coords(static_cast<int>(cur), p, m, n, kb0, kb1, slot);
      cur += gridDim.x;
    }
    return true;
  }
};

// Eight gains from element e of a head's [128] gain vector (ones without one),
// one 16-byte load when the vector is 16-byte aligned.
__device__ __forceinline__ void gain8(const __nv_bfloat16* kg, bool vec, int e, float (&g)[8]) {
  if (kg == nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 1.f;
  } else if (vec) {
    const uint4 u = *reinterpret_cast<const uint4*>(kg + e);
    g[0] = bf16_lo(u.x); g[1] = bf16_hi(u.x); g[2] = bf16_lo(u.y); g[3] = bf16_hi(u.y);
    g[4] = bf16_lo(u.z); g[5] = bf16_hi(u.z); g[6] = bf16_lo(u.w); g[7] = bf16_hi(u.w);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = __bfloat162float(kg[e + i]);
  }
}

// Epilogue of one 128-column head of the K/V projection for this thread's row.
__device__ __forceinline__ void kv_head_epilogue(uint32_t taddr, int col0, int row, const GemmArgs& p) {
  const int hidx = col0 / HD;
  const int l = hidx / (2 * p.Hkv);
  const int s = (hidx / p.Hkv) % 2;
  const int h = hidx % p.Hkv;
  int2 ri = make_int2(-1, -1);
  if (row < p.M) ri = p.rowinfo[row];
  const bool valid = ri.x >= 0;
  __nv_bfloat16* dst = (s == 0 ? p.cache_k : p.cache_v) +
                       ((((static_cast<size_t>(l) * p.Bc + (valid ? ri.x : 0)) * p.Hkv + h) * p.cap) +
                        (valid ? ri.y : 0)) * HD;
  uint32_t r[32];
  if (s == 1) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tmem_ld_32cols(taddr + c * 32, r);
      tmem_ld_wait();
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
      }
    }
    return;
  }
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    tmem_ld_32cols(taddr + c * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float v = __uint_as_float(r[i]);
      ss += v * v;
    }
  }
  const float rinv = rsqrtf(ss * (1.0f / HD) + p.eps);
  const __nv_bfloat16* kg = p.k_gain ? p.k_gain + l * HD : nullptr;
  const bool kg_vec = kg && (reinterpret_cast<uintptr_t>(kg) & 15u) == 0;
  const float2* cs = p.rope_cs + (valid ? row : 0);
  const size_t cs_stride = static_cast<size_t>(p.M);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int e0 = half * 32;
    uint32_t r2[32];
    tmem_ld_32cols(taddr + e0, r);
    tmem_ld_32cols(taddr + 64 + e0, r2);
    tmem_ld_wait();
    uint32_t o1[16], o2[16];
#pragma unroll
    for (int j8 = 0; j8 < 32; j8 += 8) {
      float g1[8], g2[8];
      gain8(kg, kg_vec, e0 + j8, g1);
      gain8(kg, kg_vec, 64 + e0 + j8, g2);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        float a[2], b[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j8 + i + k;
          const float y1 = __uint_as_float(r[j]) * rinv * g1[i + k];
          const float y2 = __uint_as_float(r2[j]) * rinv * g2[i + k];
          const float2 c = valid ? cs[(e0 + j) * cs_stride] : make_float2(1.f, 0.f);
          a[k] = y1 * c.x - y2 * c.y;
          b[k] = y2 * c.x + y1 * c.y;
        }
        o1[(j8 + i) / 2] = pack_bf16x2(a[0], a[1]);
        o2[(j8 + i) / 2] = pack_bf16x2(b[0], b[1]);
      }
    }
    if (valid) {
      uint4* d1 = reinterpret_cast<uint4*>(dst + e0);
      uint4* d2 = reinterpret_cast<uint4*>(dst + 64 + e0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        d1[i] = make_uint4(o1[4 * i], o1[4 * i + 1], o1[4 * i + 2], o1[4 * i + 3]);
        d2[i] = make_uint4(o2[4 * i], o2[4 * i + 1], o2[4 * i + 2], o2[4 * i + 3]);
      }
    }
  }
}

template <int BN, int STAGES, int MT>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_tc_kernel(const __grid_constant__ TmapPack amaps,
                                                                  const __grid_constant__ CUtensorMap bmap,
                                                                  const GemmArgs p) {
  constexpr int A_BYTES = kBM * kBK * 2;   // one 128-row A box
  constexpr int STAGE = stage_bytes<BN, MT>();
  constexpr int NACC = num_acc<BN, MT>();
  constexpr int ACC_COLS = MT * BN;
  constexpr uint32_t IDESC = umma_idesc_bf16(kBM, BN);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), NACC * ACC_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------ TMA producer
      for (int s = 0; s < kMaxSeg; ++s)
        if (s * p.kb_per_seg < p.num_kb) tma_prefetch_desc(&amaps.a[s]);
      tma_prefetch_desc(&bmap);
      // The B operand (weights) does not depend on the previous kernel: as a
      // programmatic dependent, fill the ring's B halves first, then wait.
      int pre = 0;
      Pieces first(p);
      int m, n, kb0, kb1, ks;
      if (p.prefetch_b && first.next(p, m, n, kb0, kb1, ks)) {
        for (; pre < STAGES && kb0 + pre < kb1; ++pre) {
          const int kbp = kb_at(pre, kb0, kb1, n, p);
          const uint32_t fb = full0 + 8 * pre;
          mbar_arrive_expect_tx(fb, STAGE);
          tma_load_2d(base + pre * STAGE + MT * A_BYTES, &bmap, fb, kbp * kBK, n * BN);
        }
      }
      pdl_wait_primary();
      // The next kernel (the row norm) reads its inputs before its own wait:
      // release it only once the grid this one depends on has completed.
      pdl_launch_dependents();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Pieces pcs(p);
      for (bool head = true; ok && pcs.next(p, m, n, kb0, kb1, ks); head = false) {
        for (int i = 0; i < kb1 - kb0; ++i) {
          const int kb = kb_at(i, kb0, kb1, n, p);
          const bool b_done = head && i < pre;
          if (!b_done && !(ok = mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.status))) break;
          const uint32_t fb = full0 + 8 * stage;
          if (!b_done) mbar_arrive_expect_tx(fb, STAGE);
          const uint32_t sa = base + stage * STAGE;
          const int seg = kb / p.kb_per_seg;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            tma_load_2d(sa + mt * A_BYTES, &amaps.a[seg], fb, (kb - seg * p.kb_per_seg) * kBK, (m * MT + mt) * kBM);
          if (!b_done) tma_load_2d(sa + MT * A_BYTES, &bmap, fb, kb * kBK, n * BN);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      Pieces pcs(p);
      int m, n, kb0, kb1, ks;
      while (ok && pcs.next(p, m, n, kb0, kb1, ks)) {
        if (!(ok = mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, p.status))) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int i = 0; i < kb1 - kb0; ++i) {
          if (!(ok = mbar_wait(full0 + 8 * stage, phase, p.status))) break;
          tc_fence_after_sync();
          const uint32_t sa = base + stage * STAGE;
          const uint64_t bd = umma_desc_kmajor_sw128(sa + MT * A_BYTES);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint64_t ad = umma_desc_kmajor_sw128(sa + mt * A_BYTES);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              umma_bf16(d_tmem + mt * BN, ad + 2 * k, bd + 2 * k, IDESC, (i > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(tfull0 + 8 * acc);
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else {  // -------------------------------------------- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    Pieces pcs(p);
    int m, n, kb0, kb1, ks;
    while (pcs.next(p, m, n, kb0, kb1, ks)) {
      if (!mbar_wait(tfull0 + 8 * acc, acc_phase, p.status)) break;
      if (p.stream_k && ks == 0 && warp == 2 && lane == 0) p.pieces[m * p.n_tiles + n] = pcs.count;
      tc_fence_after_sync();
#pragma unroll 1
      for (int i = 0; i < MT; ++i) {
        const int row = (m * MT + i) * kBM + q * 32 + lane;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS + i * BN;
        if (p.epi == 0) {
          float* dst = p.out_f32 + (static_cast<size_t>(ks) * p.M + row) * p.N + n * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(taddr + c * 32, r);
            tmem_ld_wait();
            if (row < p.M) {
              float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                    __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
          }
        } else {
#pragma unroll 1
          for (int hh = 0; hh < BN / HD; ++hh) kv_head_epilogue(taddr + hh * HD, n * BN + hh * HD, row, p);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, NACC * ACC_COLS);
  }
}

// One CTA per new row m:
//   * row -> (sequence, cache position) and the RoPE (cos, sin) table of the row
//     (used by the K/V epilogue);
//   * H_t[m] = the sum of the split-K partials of Y[m], RMS-normalised with
//     gain g, stored as TH (workspace copy for the K/V GEMM) and optionally as
//     the caller's copy.  Each thread keeps its float4 slots of the row in
//     registers (rows up to 4096 wide), so the partials are read once.
constexpr int kNormThreads = 256;
constexpr int kNormSlots = 4;  // float4 slots per thread

template <typename TG, typename TH>
__global__ void __launch_bounds__(kNormThreads) fuse_rownorm_kernel(
    const float* __restrict__ part, int k_splits, const int* __restrict__ pieces, int tile_rows, int tile_cols,
    int n_tiles, int M, int D, const TG* __restrict__ g, float eps,
    TH* __restrict__ ht, TH* __restrict__ ht_out, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ seq_len, int B, int cap, int ring, InvFreq inv, int2* __restrict__ rowinfo,
    float2* __restrict__ rope_cs, unsigned* status) {
  const int m = blockIdx.x;
  if (threadIdx.x <= HD / 2) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {  // largest b with cu_new[b] <= m
      const int mid = (lo + hi + 1) >> 1;
      if (cu_new[mid] <= m) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
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
      rope_cs[static_cast<size_t>(threadIdx.x) * M + m] = make_float2(cv, sv);
    } else {
      rowinfo[m] = valid ? make_int2(b, ring ? pos % cap : pos) : make_int2(-1, -1);  // (sequence, cache row)
      if (!valid) raise_status(status, seq_ok ? DFLASH_DEV_CAPACITY : DFLASH_DEV_BAD_SEQLEN);
    }
  }
  pdl_launch_dependents();
  pdl_wait_primary();  // the partials of the fusion GEMM
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
  const bool in_regs = nv <= kNormThreads * kNormSlots;
  float4 y[kNormSlots];
  float ss = 0.f;
  if (in_regs) {
    // slots outermost, so the loads of a thread's float4 slots are independent
    int ns[kNormSlots];
    int ns_max = 0;
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i) {
      const int v = threadIdx.x + i * kNormThreads;
      y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      ns[i] = v < nv ? (prow_pieces ? prow_pieces[(4 * v) / tile_cols] : k_splits) : 0;
      ns_max = max(ns_max, ns[i]);
      if (v < nv) y[i] = prow[v];
    }
    for (int s0 = 1; s0 < ns_max; s0 += 2) {
      float4 t[2][kNormSlots];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int i = 0; i < kNormSlots; ++i)
          if (s0 + u < ns[i]) t[u][i] = prow[(s0 + u) * split_stride + threadIdx.x + i * kNormThreads];
#pragma unroll
      for (int u = 0; u < 2; ++u)
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
    for (int v = threadIdx.x; v < nv; v += kNormThreads) {
      const float4 t4 = row_sum(v);
      ss += t4.x * t4.x + t4.y * t4.y + t4.z * t4.z + t4.w * t4.w;
    }
  }
  ss = warp_sum(ss);
  __shared__ float red[kNormThreads / 32];
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float r = rsqrtf(tot / static_cast<float>(D) + eps);
  auto store = [&](int v, float4 t4) {
    const int e = 4 * v;
    const float g0 = g ? to_f32<TG>(g[e]) : 1.f, g1 = g ? to_f32<TG>(g[e + 1]) : 1.f;
    const float g2 = g ? to_f32<TG>(g[e + 2]) : 1.f, g3 = g ? to_f32<TG>(g[e + 3]) : 1.f;
    const TH h0 = from_f32<TH>(t4.x * r * g0), h1 = from_f32<TH>(t4.y * r * g1);
    const TH h2 = from_f32<TH>(t4.z * r * g2), h3 = from_f32<TH>(t4.w * r * g3);
    TH* d = ht + static_cast<size_t>(m) * D + e;
    d[0] = h0;
    d[1] = h1;
    d[2] = h2;
    d[3] = h3;
    if (ht_out) {
      TH* o = ht_out + static_cast<size_t>(m) * D + e;
      o[0] = h0;
      o[1] = h1;
      o[2] = h2;
      o[3] = h3;
    }
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kNormSlots; ++i) {
      const int v = threadIdx.x + i * kNormThreads;
      if (v < nv) store(v, y[i]);
    }
  } else {
    for (int v = threadIdx.x; v < nv; v += kNormThreads) store(v, row_sum(v));
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
};

FusePlan plan(int M, int D, int num_kb) {
  FusePlan f;
  f.fuse_mt = M <= 2 * kBM ? 2 : 1;
  f.fuse_m_tiles = (M + f.fuse_mt * kBM - 1) / (f.fuse_mt * kBM);
  f.fuse_bn = M <= 2 * kBM ? 128 : 256;
  f.fuse_n_tiles = D / f.fuse_bn;
  const int tiles = f.fuse_m_tiles * f.fuse_n_tiles;
  f.stream_k = f.fuse_mt == 1 && tiles % kSplitTarget != 0;
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
  return f;
}

template <int BN, int STAGES, int MT>
dflash_status launch_gemm(const TmapPack& am, const CUtensorMap& bm, const GemmArgs& a, cudaStream_t st,
                          const DeviceInfo& dev) {
  const size_t smem = gemm_smem_bytes<BN, STAGES, MT>();
  if (smem > dev.max_smem_optin) return fail(DFLASH_ERR_UNSUPPORTED, "gemm_tc: shared memory");
  static int configured = -1;
  if (configured != dev.device) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, STAGES, MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemm_tc_kernel)");
    configured = dev.device;
  }
  const int units = a.m_tiles * a.n_tiles * a.k_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.stream_k ? a.stream_k : std::min(units, dev.num_sms)));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t le = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, STAGES, MT>, am, bm, a);
  if (le != cudaSuccess) return cuda_fail(le, "gemm_tc_kernel launch");
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "gemm_tc_kernel launch");
}

}  // namespace

size_t fuse_ws_bytes(int M, int J, int dt_width, int D, int L, int Hkv, dflash_dtype dt) {
  const int Ntot = L * 2 * Hkv * HD;
  size_t s = align256(static_cast<size_t>(M) * sizeof(int2)) +
             align256(static_cast<size_t>(M) * (HD / 2) * sizeof(float2));
  if (dt == DFLASH_BF16) {
    const FusePlan f = plan(M, D, J * dt_width / kBK);
    s += align256(static_cast<size_t>(f.k_splits) * M * D * sizeof(float)) +
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
        c.capacity, c.ring, inv, rowinfo, rope_cs, dev.status);
    F32Segs hs{};
    hs.a[0] = H;
    simt_gemm_f32_kernel<<<dim3((Ntot + 63) / 64, (M + 63) / 64), 256, 0, st>>>(
        hs, D, static_cast<const float*>(w_kv), M, Ntot, D, KV);
    const long warps = static_cast<long>(M) * L * 2 * Hkv;
    kv_store_f32_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
        KV, M, L, Hkv, c.batch, c.capacity, rowinfo, rope_cs, static_cast<const float*>(k_gain), eps,
        static_cast<float*>(c.k), static_cast<float*>(c.v));
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "fp32 fusion launch");
  }

  const FusePlan f = plan(M, D, J * dt_width / kBK);
  if (D % 4 != 0) return fail(DFLASH_ERR_UNSUPPORTED, "fusion: d_model must be a multiple of 4");
  float* Ypart = w.take<float>(static_cast<size_t>(f.k_splits) * M * D);
  auto* H = w.take<__nv_bfloat16>(static_cast<size_t>(M) * D);
  int* tile_pieces = w.take<int>(static_cast<size_t>(f.fuse_m_tiles) * f.fuse_n_tiles);

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
  a.pdl = 1;  // its CTAs may start while the preceding kernel finishes; nothing is loaded before it has
  a.out_f32 = Ypart;
  a.status = dev.status;
  s = f.fuse_mt == 2 ? launch_gemm<128, 4, 2>(am, bm, a, st, dev) : launch_gemm<256, 4, 1>(am, bm, a, st, dev);
  if (s) return s;

  // 2. row map + split-K sum + RMSNorm -> H_t (bf16), a programmatic dependent
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(kNormThreads);
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
                                        c.ring, inv, rowinfo, rope_cs, dev.status);
    if (le != cudaSuccess) return cuda_fail(le, "fuse_rownorm_kernel launch");
  }

  // 3. K/V GEMM with the cache epilogue
  TmapPack hm{};
  s = make_tmap_bf16_2d(&hm.a[0], H, static_cast<uint64_t>(M), D, kBM, kBK);
  if (s) return s;
  CUtensorMap wm;
  s = make_tmap_bf16_2d(&wm, w_kv, static_cast<uint64_t>(Ntot), D, f.kv_bn, kBK);
  if (s) return s;
  GemmArgs k{};
  k.M = M;
  k.N = Ntot;
  k.num_kb = D / kBK;
  k.kb_per_seg = k.num_kb;
  k.k_splits = 1;
  k.m_tiles = (M + kBM - 1) / kBM;
  k.n_tiles = Ntot / f.kv_bn;
  k.epi = 1;
  k.pdl = 1;
  k.prefetch_b = 1;
  k.cache_k = static_cast<__nv_bfloat16*>(c.k);
  k.cache_v = static_cast<__nv_bfloat16*>(c.v);
  k.L = L;
  k.Bc = c.batch;
  k.Hkv = Hkv;
  k.cap = c.capacity;
  k.rowinfo = rowinfo;
  k.rope_cs = rope_cs;
  k.k_gain = static_cast<const __nv_bfloat16*>(k_gain);
  k.eps = eps;
  k.status = dev.status;
  return f.kv_bn == 256 ? launch_gemm<256, 4, 1>(hm, wm, k, st, dev) : launch_gemm<128, 6, 1>(hm, wm, k, st, dev);
}

}  // namespace dflash
