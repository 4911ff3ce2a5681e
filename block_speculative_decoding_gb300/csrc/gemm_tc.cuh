// The warp-specialised tcgen05 GEMM shared by the fusion, the drafter's
// head and the draft-layer remainder: a TMA producer warp, one MMA-issuing
// thread, four epilogue warps;
// operands staged by TMA in a shared-memory ring (128-byte swizzle, K-major),
// accumulators in tensor memory (double-buffered when they fit), plain or
// stream-K schedules (the partial sums of a tile either left in slots for the
// next kernel or added in by the share that holds the tile's first K block),
// and three epilogues (fp32 sums, the K/V cache rows of the fusion, the
// drafter's logits with the draft race).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
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
constexpr int kSplitTarget = 152;  // work units aimed for when splitting K (one per SM)
constexpr int kStgRow = 36;        // fp32 staging row of an epilogue warp: 32 columns + 4 of padding
constexpr int kStgBytes = 32 * kStgRow * 4;
constexpr int kBarBytes = 512;     // mbarriers and the tensor-memory address
constexpr int kFixGroupF4 = 4 * 8 * kBM;         // float4 of one partial sum over a 128-column group
constexpr int kFixGroupBytes = kFixGroupF4 * 16;  // 64 KB

struct TmapPack {
  CUtensorMap a[kMaxSeg];
};

struct GemmArgs {
  int M, N, num_kb, kb_per_seg, k_splits, m_tiles, n_tiles;
  int stream_k;            // > 0: the number of shares (CTAs); CTA c takes the c-th near-equal share of the
                           // (tile, K block) space
  int dp_tiles;            // stream_k: leading tiles scheduled whole, a multiple of the share count
  int* pieces;             // stream_k without fixup: [m_tiles * n_tiles] number of slots written for the tile
  int fixup;               // stream_k: a share that holds a tile's first K block adds the other shares'
                           // partial sums before the epilogue (which then sees the whole sum)
  float4* fix_part;        // fixup: [shares][MT * BN * 32] float4, the partial sum of a share's first piece
                           // in the accumulator's own order (column chunk, 4-column group, row)
  int* fix_flag;           // fixup: [shares], zero at launch; 4 once the share's partial sum is stored
  int epi;                 // 0: fp32 partial store, 1: K/V cache epilogue, 2: drafter logits + draft race
  int a4d_bs;              // > 0: A is an attention output [B][Hq][a4d_bs][128] read through a 4D map
                           // (row b * bs + j, K index h * 128 + e); 0: A is a row-major 2D tensor
  int pdl;                 // launched as a programmatic dependent (waits for the preceding grid before any load)
  int prefetch_b;          // the B operand (weights) may be loaded before that wait
  float* out_f32;          // epi 0: [k_splits][M][N]
  __nv_bfloat16* cache_k;  // epi 1
  __nv_bfloat16* cache_v;
  int L, Bc, Hkv, cap;
  const int2* rowinfo;     // [M] (sequence, cache row) or (-1, -1)
  const __half2* rope_cs;  // [64][M] (cos, sin) in fp16, element-major: a warp's rows read it coalesced
  const __nv_bfloat16* k_gain;  // [L][128] or null
  float eps;
  // epi 2 (drafter head): rows are (sequence b, proposal row k) with k < rows_per_seq
  __nv_bfloat16* logits;   // [M][N] bf16
  float2* race;            // [M][n_tiles] best (key, column as int bits) of each N tile
  float inv_temp;          // 1 / T; 0: greedy (key = logit)
  int rows_per_seq;
  uint32_t seed_lo, seed_hi, cycle_lo, cycle_hi;
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
  static_assert(8 * (2 * STAGES + 5) + 16 <= kBarBytes, "mbarrier block");
  return 1024 + static_cast<size_t>(STAGES) * stage_bytes<BN, MT>() + kBarBytes + 4 * kStgBytes;
}

template <int BN, int MT>
__host__ __device__ constexpr int fix_part_float4() {
  return MT * BN * kBM / 4;
}

// Where the epilogue reads this thread's row of a unit: tensor memory, plus
// (fixup) the partial sums of nfix later shares of the same tile.  A partial
// sum is stored as float4 [column chunk of 32][group of 4 columns][row of the
// 128-row block], so the 32 rows of a warp read and write 512 contiguous bytes.
struct AccSrc {
  uint32_t taddr;        // tensor memory of the 128-column group (lane quarter and accumulator applied)
  const float4* fix;     // the first later share's partial sum (this thread's row applied), in global
                         // memory or staged in shared memory
  int nfix;
  int fix_stride;        // float4 between two shares' partial sums
  int col_base;          // column of the group in the layout fix points into
  bool smem;             // fix points into shared memory
};

// Adds the later shares' partial sums of columns col .. col + 31 (col a
// multiple of 32) of this thread's row to r.
__device__ __forceinline__ void acc_add32(const AccSrc& s, int col, uint32_t (&r)[32]) {
  const float4* src = s.fix + static_cast<size_t>((s.col_base + col) >> 5) * 8 * kBM;
  for (int k = 0; k < s.nfix; ++k, src += s.fix_stride) {
    float4 v[8];
    if (s.smem) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = src[j * kBM];
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + j * kBM);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v[j].x);
      r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v[j].y);
      r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v[j].z);
      r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v[j].w);
    }
  }
}

// 32 accumulator columns from col (a multiple of 32) of this thread's row.
__device__ __forceinline__ void acc_ld32(const AccSrc& s, int col, uint32_t (&r)[32]) {
  tmem_ld_32cols(s.taddr + col, r);
  tmem_ld_wait();
  acc_add32(s, col, r);
}

// Two 32-column blocks, both tensor-memory loads in flight before one wait.
__device__ __forceinline__ void acc_ld32x2(const AccSrc& s, int ca, uint32_t (&ra)[32], int cb, uint32_t (&rb)[32]) {
  tmem_ld_32cols(s.taddr + ca, ra);
  tmem_ld_32cols(s.taddr + cb, rb);
  tmem_ld_wait();
  acc_add32(s, ca, ra);
  acc_add32(s, cb, rb);
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

// Eight gains from element e of a head's [128] gain vector, held as fp32 in
// shared memory (nullptr: ones).
__device__ __forceinline__ void gain8(const float* kg, int e, float (&g)[8]) {
  if (kg == nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 1.f;
  } else {
    const float4 a = *reinterpret_cast<const float4*>(kg + e);
    const float4 b = *reinterpret_cast<const float4*>(kg + e + 4);
    g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
  }
}

// Epilogue of the drafter's head for this thread's row, BN columns from col0:
// the logits rounded to bf16 and stored, and the best key of the draft race
// over those columns (a draw from softmax(logits / T) is the argmax of
// logit / T - ln(-ln U); T == 0: the argmax of the logits), ties to the lowest
// column.  U comes from one Philox-4x32-10 block per four columns, counter
// (col / 4, (b << 5) | k, cycle_lo, cycle_hi | tag), word col % 4,
// U = ((w >> 8) + 1) * 2^-24.
template <int BN>
__device__ __forceinline__ void head_epilogue(uint32_t taddr, int col0, int row, int n_tile, const GemmArgs& p) {
  const bool live = row < p.M;
  const int b = row / p.rows_per_seq, k = row % p.rows_per_seq;
  const uint32_t c1 = (static_cast<uint32_t>(b) << 5) | static_cast<uint32_t>(k);
  const uint32_t c3 = p.cycle_hi | 0x80000000u;
  const bool greedy = p.inv_temp == 0.f;
  float best = -INFINITY;
  int best_col = INT_MAX;
  __nv_bfloat16* dst = p.logits + static_cast<size_t>(live ? row : 0) * p.N + col0;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32cols(taddr + c * 32, r);
    tmem_ld_wait();
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    if (live) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) d4[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
    }
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) {  // four columns per Philox block
      const int colg = col0 + c * 32 + 4 * g4;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (!greedy) w = philox4x32_10(make_uint4(static_cast<uint32_t>(colg) >> 2, c1, p.cycle_lo, c3), p.seed_lo, p.seed_hi);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int j = 4 * g4 + t;
        const uint32_t h = packed[j / 2];
        const float lg = (j & 1) ? bf16_hi(h) : bf16_lo(h);  // the stored (rounded) logit
        float key = lg;
        if (!greedy) {
          const float u = static_cast<float>((ws[t] >> 8) + 1u) * (1.0f / 16777216.0f);
          key = fmaf(lg, p.inv_temp, -__logf(-__logf(u)));
        }
        if (key > best) {
          best = key;
          best_col = colg + t;
        }
      }
    }
  }
  if (live) p.race[static_cast<size_t>(row) * p.n_tiles + n_tile] = make_float2(best, __int_as_float(best_col));
}

// fp32 sums of one 128-column group from column col0 into out_f32 slot ks,
// staged through this warp's shared-memory rows so that each store instruction
// writes four whole 128-byte row segments; row0 is the warp's first row.
__device__ __forceinline__ void f32_group(const AccSrc& src, float* stg, int ks, int row0, int col0, int lane,
                                          const GemmArgs& p) {
  float* dst = p.out_f32 + static_cast<size_t>(ks) * p.M * p.N + col0 + (lane & 7) * 4;
#pragma unroll 1
  for (int c2 = 0; c2 < 4; c2 += 2) {
    uint32_t r[2][32];
    acc_ld32x2(src, c2 * 32, r[0], c2 * 32 + 32, r[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(stg + lane * kStgRow + 4 * j) =
            make_float4(__uint_as_float(r[h][4 * j]), __uint_as_float(r[h][4 * j + 1]),
                        __uint_as_float(r[h][4 * j + 2]), __uint_as_float(r[h][4 * j + 3]));
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int rl = it * 4 + (lane >> 3);
        const float4 v = *reinterpret_cast<const float4*>(stg + rl * kStgRow + (lane & 7) * 4);
        if (row0 + rl < p.M)
          *reinterpret_cast<float4*>(dst + static_cast<size_t>(row0 + rl) * p.N + (c2 + h) * 32) = v;
      }
    }
  }
}

// Epilogue of one 128-column head of the K/V projection for this thread's row.
__device__ __forceinline__ void kv_head_epilogue(const AccSrc& src, int hcol, int col0, int row, const float* kgain,
                                                 const GemmArgs& p) {
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
    uint32_t rv[2][32];
#pragma unroll 1
    for (int c = 0; c < 4; c += 2) {
      acc_ld32x2(src, hcol + c * 32, rv[0], hcol + c * 32 + 32, rv[1]);
      if (valid) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + (c + h2) * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pack_bf16x2(__uint_as_float(rv[h2][8 * i]), __uint_as_float(rv[h2][8 * i + 1])),
                               pack_bf16x2(__uint_as_float(rv[h2][8 * i + 2]), __uint_as_float(rv[h2][8 * i + 3])),
                               pack_bf16x2(__uint_as_float(rv[h2][8 * i + 4]), __uint_as_float(rv[h2][8 * i + 5])),
                               pack_bf16x2(__uint_as_float(rv[h2][8 * i + 6]), __uint_as_float(rv[h2][8 * i + 7])));
        }
      }
    }
    return;
  }
  // all 64 rotation pairs of the row are requested before the accumulator is
  // read (unconditionally: rows past the end read row 0 and store nothing),
  // so their global-memory latency overlaps it
  const __half2* cs = p.rope_cs + (row < p.M ? row : 0);
  const size_t cs_stride = static_cast<size_t>(p.M);
  __half2 csh[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) csh[j] = __ldg(cs + j * cs_stride);
  float ss = 0.f;
  uint32_t r2[32];
#pragma unroll 1
  for (int c = 0; c < 4; c += 2) {
    acc_ld32x2(src, hcol + c * 32, r, hcol + c * 32 + 32, r2);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float v = __uint_as_float(r[i]), v2 = __uint_as_float(r2[i]);
      ss += v * v + v2 * v2;
    }
  }
  const float rinv = rsqrtf(ss * (1.0f / HD) + p.eps);
  const float* kg = kgain ? kgain + l * HD : nullptr;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int e0 = half * 32;
    acc_ld32x2(src, hcol + e0, r, hcol + 64 + e0, r2);
    uint32_t o1[16], o2[16];
#pragma unroll
    for (int j8 = 0; j8 < 32; j8 += 8) {
      float g1[8], g2[8];
      gain8(kg, e0 + j8, g1);
      gain8(kg, 64 + e0 + j8, g2);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        float a[2], b[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j8 + i + k;
          const float y1 = __uint_as_float(r[j]) * rinv * g1[i + k];
          const float y2 = __uint_as_float(r2[j]) * rinv * g2[i + k];
          const float2 c = __half22float2(csh[e0 + j]);
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  float* stg_all = reinterpret_cast<float*>(gbase + STAGES * STAGE + kBarBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t fixbar = tempty0 + 16;  // staged partial sums of a fixup

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
    mbar_init(fixbar, 1);
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
          for (int mt = 0; mt < MT; ++mt) {
            if (p.a4d_bs > 0)  // K block kb = (head kb / 2, dims (kb % 2) * 64 ..), rows = (sequence, block row)
              tma_load_4d(sa + mt * A_BYTES, &amaps.a[0], fb, (kb & 1) * 64, 0, kb >> 1,
                          (m * MT + mt) * kBM / p.a4d_bs);
            else
              tma_load_2d(sa + mt * A_BYTES, &amaps.a[seg], fb, (kb - seg * p.kb_per_seg) * kBK, (m * MT + mt) * kBM);
          }
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
    float* stg = stg_all + q * (32 * kStgRow);
    constexpr int FIX = fix_part_float4<BN, MT>();
    // K/V epilogue: every layer's K gains, as fp32, in the staging area (which
    // only the fp32 epilogue uses otherwise)
    const float* kgain = nullptr;
    if (p.epi == 1 && p.k_gain != nullptr && p.L * HD <= 4 * 32 * kStgRow) {
      for (int i = threadIdx.x - 64; i < p.L * HD; i += 128) stg_all[i] = __bfloat162float(p.k_gain[i]);
      named_barrier_sync(1, 128);
      kgain = stg_all;
    }
    const int rowl = q * 32 + lane;  // row within a 128-row block
    uint32_t fphase = 0;             // parity of the staged-partials barrier
    while (pcs.next(p, m, n, kb0, kb1, ks)) {
      if (!mbar_wait(tfull0 + 8 * acc, acc_phase, p.status)) break;
      if (p.stream_k && !p.fixup && ks == 0 && warp == 2 && lane == 0) p.pieces[m * p.n_tiles + n] = pcs.count;
      tc_fence_after_sync();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS;
      if (p.fixup && ks > 0) {
        // a later share of the tile: store the partial sum, then raise this share's flag
        float4* dst = p.fix_part + static_cast<size_t>(blockIdx.x) * FIX + rowl;
#pragma unroll 1
        for (int cc = 0; cc < MT * BN / 32; ++cc) {
          uint32_t r[32];
          tmem_ld_32cols(tacc + cc * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            __stcg(dst + (cc * 8 + j) * kBM, make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                         __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(p.fix_flag + blockIdx.x, 1);
        }
      } else {
        // the tile's first share adds the later shares' partial sums (shares
        // blockIdx.x + 1 ..).  This is the share's last piece, so once its
        // accumulator is complete the operand ring is idle: up to three
        // partial sums are staged there, one 128-column group at a time, by
        // bulk copies; more are read from global memory as they are used.
        const int nfix = (p.fixup && pcs.count > 1) ? pcs.count - 1 : 0;
        const bool staged = nfix > 0 && nfix * kFixGroupBytes <= STAGES * STAGE;
        if (nfix > 0 && !staged) {
          if (lane == 0)
            for (int k = 1; k <= nfix; ++k)
              if (!wait_counter_at_least(p.fix_flag + blockIdx.x + k, 4, p.status)) break;
          __syncwarp();
        }
        bool first_group = true;
#pragma unroll 1
        for (int i = 0; i < MT; ++i) {
          const int row = (m * MT + i) * kBM + rowl;
          if (p.epi == 2) {
            head_epilogue<BN>(tacc + i * BN, n * BN, row, n, p);
            continue;
          }
#pragma unroll 1
          for (int grp = 0; grp < BN / 128; ++grp) {
            AccSrc src;
            src.taddr = tacc + i * BN + grp * 128;
            src.nfix = nfix;
            if (staged) {
              named_barrier_sync(1, 128);  // the previous group's staged sums have been read
              if (warp == 2 && lane == 0) {
                if (first_group)
                  for (int k = 1; k <= nfix; ++k)
                    if (!wait_counter_at_least(p.fix_flag + blockIdx.x + k, 4, p.status)) break;
                fence_proxy_async_all();
                mbar_arrive_expect_tx(fixbar, nfix * kFixGroupBytes);
                for (int k = 0; k < nfix; ++k)
                  bulk_load(base + k * kFixGroupBytes,
                            p.fix_part + static_cast<size_t>(blockIdx.x + 1 + k) * FIX +
                                static_cast<size_t>(i * (BN / 128) + grp) * kFixGroupF4,
                            kFixGroupBytes, fixbar);
              }
              mbar_wait(fixbar, fphase, p.status);
              fphase ^= 1u;
              src.fix = reinterpret_cast<const float4*>(gbase) + rowl;
              src.fix_stride = kFixGroupF4;
              src.col_base = 0;
              src.smem = true;
            } else {
              src.fix = p.fix_part + static_cast<size_t>(blockIdx.x + 1) * FIX + rowl;
              src.fix_stride = FIX;
              src.col_base = i * BN + grp * 128;
              src.smem = false;
            }
            first_group = false;
            const int col0 = n * BN + grp * 128;
            if (p.epi == 0)
              f32_group(src, stg, ks, row - lane, col0, lane, p);
            else
              kv_head_epilogue(src, 0, col0, row, kgain, p);
          }
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

// The most stream-K shares that meet one tile when `tiles` tiles of num_kb K
// blocks are cut into `shares` near-equal shares (the slots a tile needs).
inline int sk_max_count(long tiles, long num_kb, long shares) {
  const long tot = tiles * num_kb;
  auto share = [&](long x) { return ((x + 1) * shares - 1) / tot; };
  int c = 1;
  for (long t = 0; t < tiles; ++t)
    c = std::max(c, static_cast<int>(share((t + 1) * num_kb - 1) - share(t * num_kb) + 1));
  return c;
}

// Stream-K with fixup over all of a GEMM's tiles: as many shares as SMs
// (every share non-empty); each share's partial-sum area and its flag.
inline int fixup_shares(int tiles, int num_kb) {
  return static_cast<int>(std::min<long>(kSplitTarget, static_cast<long>(tiles) * num_kb));
}

template <int BN, int MT>
size_t fixup_ws_bytes(int shares) {
  return align256(static_cast<size_t>(shares) * fix_part_float4<BN, MT>() * sizeof(float4)) +
         align256(static_cast<size_t>(shares) * sizeof(int));
}

template <int BN, int MT>
void fixup_take(WsCarver& w, int shares, GemmArgs& a) {
  a.fix_part = w.take<float4>(static_cast<size_t>(shares) * fix_part_float4<BN, MT>());
  a.fix_flag = w.take<int>(static_cast<size_t>(shares));
  a.fixup = 1;
  a.stream_k = shares;
  a.dp_tiles = 0;
  a.k_splits = 1;
}

template <int BN, int STAGES, int MT>
dflash_status launch_gemm(const TmapPack& am, const CUtensorMap& bm, const GemmArgs& a, cudaStream_t st,
                          const DeviceInfo& dev) {
  const size_t smem = gemm_smem_bytes<BN, STAGES, MT>();
  if (smem > dev.max_smem_optin) return fail(DFLASH_ERR_UNSUPPORTED, "gemm_tc: shared memory");
  dflash_status ss = smem_limit_once<gemm_tc_kernel<BN, STAGES, MT>>(dev.device, static_cast<int>(smem),
                                                                      "cudaFuncSetAttribute(gemm_tc_kernel)");
  if (ss) return ss;
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
}  // namespace dflash
