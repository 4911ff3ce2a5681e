// A draft layer around its attention: before it, the input RMSNorm and the
// block rows' q/k/v projections; after it, the output projection and
// residual, post-attention RMSNorm, SwiGLU MLP and residual.
//
// Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash",
// section "The parameter count exposes the real cost" (a Qwen3-style layer:
// q/k/v/o projections, a gated MLP, two RMSNorms; the MLP's intermediate size
// 5120 closes the printed parameter count) and "The released serving cycle"
// (the drafter runs its layers over the block).
//
// Six launches chained as programmatic dependents (M = B * bs block rows):
//   1. gemm_tc   Y = o W_o^T, split K; the attention output [B][Hq][bs][128]
//                is read through a 4D tensor map (rows (b, j), K = (h, e)),
//                never copied -> fp32 partial slots
//   2. resnorm   x1 = bf16(x + sum of the slots), written back to x;
//                h = bf16(RMSNorm(x1) * g_post)
//   3. gemm_tc   [gate | up] = h [W_gate | W_up]^T, stream-K over all SMs ->
//                fp32 slots; the weight rows are interleaved in 64-row blocks,
//                so each 128-column tile holds the gate and up values of the
//                same 64 outputs
//   4. swiglu    act = bf16(silu(gate) * up) from the slots, one thread per
//                four outputs (the GEMM's four epilogue warps per SM cannot
//                hide the latency of this work; a full grid can)
//   5. gemm_tc   Y = act W_down^T, split K -> slots
//   6. resnorm   x2 = bf16(x1 + sum of the slots) -> x
//
// The q/k/v projections, three launches:
//   1. resnorm   h = bf16(RMSNorm(x) * g_in) (no slots; x left as it is)
//   2. gemm_tc   [q | k | v] = h W_qkv^T, stream-K over all SMs -> fp32 slots;
//                a 128-column tile is one head
//   3. qkv_scatter  the sum of each tile's slots, rounded to bf16 and stored
//                in the block attention's [B][heads][bs][128] layouts
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "dflash_device.cuh"
#include "dflash_internal.h"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

constexpr int kResMaxThreads = 512;
constexpr int kResSlots = 2;      // float4 of the row per thread: rows up to 4096 wide
constexpr int kMaxKSplits = 16;   // partial sums per output (split-K slots)
constexpr int kResBatch = 8;      // slots loaded together

// One CTA per row m: x1 = bf16(x + sum_s part[s]) (written to x if write_x); with g_mode,
// h = bf16(x1 * rsqrt(mean(x1^2) + eps) * g), g == nullptr meaning ones.
// Each thread owns kResSlots float4 of the row and requests up to kResBatch
// slots of each before adding any, so its loads are in flight together.
__global__ void __launch_bounds__(kResMaxThreads) resnorm_kernel(const float* __restrict__ part, int k_splits, int M,
                                                                int D, __nv_bfloat16* __restrict__ x, int write_x,
                                                                int g_mode,
                                                                const __nv_bfloat16* __restrict__ g, float eps,
                                                                __nv_bfloat16* __restrict__ h,
                                                                int* __restrict__ zero_flags, int n_zero) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  const int nthr = blockDim.x;
  // the fixup flags of the GEMM that follows (every earlier grid has completed)
  if (m == 0)
    for (int i = threadIdx.x; i < n_zero; i += nthr) zero_flags[i] = 0;
  const int nv = D / 4;
  const float4* pr = reinterpret_cast<const float4*>(part + static_cast<size_t>(m) * D);
  const size_t stride = static_cast<size_t>(M) * D / 4;
  uint2* xr = reinterpret_cast<uint2*>(x + static_cast<size_t>(m) * D);
  float4 t[kResSlots];
  uint2 xv[kResSlots];
#pragma unroll
  for (int i = 0; i < kResSlots; ++i) {
    const int v = threadIdx.x + i * nthr;
    t[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    xv[i] = make_uint2(0u, 0u);
    if (v < nv) xv[i] = xr[v];
  }
  for (int s0 = 0; s0 < k_splits; s0 += kResBatch) {
    float4 u[kResSlots][kResBatch];
#pragma unroll
    for (int i = 0; i < kResSlots; ++i)
#pragma unroll
      for (int b = 0; b < kResBatch; ++b) {
        const int v = threadIdx.x + i * nthr;
        u[i][b] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < nv && s0 + b < k_splits) u[i][b] = __ldcg(pr + (s0 + b) * stride + v);
      }
#pragma unroll
    for (int i = 0; i < kResSlots; ++i)
#pragma unroll
      for (int b = 0; b < kResBatch; ++b) {
        t[i].x += u[i][b].x;
        t[i].y += u[i][b].y;
        t[i].z += u[i][b].z;
        t[i].w += u[i][b].w;
      }
  }
  // the row's slot lines are read by this CTA only (a 128-byte line by eight
  // consecutive threads of one warp): drop them from L2 once the warp has them
  if (D % 32 == 0) {
    __syncwarp();
    if (threadIdx.x % 8 == 0)
#pragma unroll
      for (int i = 0; i < kResSlots; ++i) {
        const int v = threadIdx.x + i * nthr;
        if (v < nv)
          for (int s = 0; s < k_splits; ++s) discard_l2_line(pr + s * stride + v);
      }
  }
  float4 y[kResSlots];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kResSlots; ++i) {
    const int v = threadIdx.x + i * nthr;
    y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v < nv) {
      const uint32_t lo = pack_bf16x2(bf16_lo(xv[i].x) + t[i].x, bf16_hi(xv[i].x) + t[i].y);
      const uint32_t hi = pack_bf16x2(bf16_lo(xv[i].y) + t[i].z, bf16_hi(xv[i].y) + t[i].w);
      if (write_x) xr[v] = make_uint2(lo, hi);
      y[i] = make_float4(bf16_lo(lo), bf16_hi(lo), bf16_lo(hi), bf16_hi(hi));  // the stored x1
      ss += y[i].x * y[i].x + y[i].y * y[i].y + y[i].z * y[i].z + y[i].w * y[i].w;
    }
  }
  if (!g_mode) return;
  ss = warp_sum(ss);
  __shared__ float red[kResMaxThreads / 32];
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nthr / 32; ++w) tot += red[w];
  const float r = rsqrtf(tot / static_cast<float>(D) + eps);
  uint2* hr = reinterpret_cast<uint2*>(h + static_cast<size_t>(m) * D);
#pragma unroll
  for (int i = 0; i < kResSlots; ++i) {
    const int v = threadIdx.x + i * nthr;
    if (v >= nv) continue;
    float g4[4] = {1.f, 1.f, 1.f, 1.f};
    if (g) {
      const uint2 gv = reinterpret_cast<const uint2*>(g)[v];
      g4[0] = bf16_lo(gv.x);
      g4[1] = bf16_hi(gv.x);
      g4[2] = bf16_lo(gv.y);
      g4[3] = bf16_hi(gv.y);
    }
    hr[v] = make_uint2(pack_bf16x2(y[i].x * r * g4[0], y[i].y * r * g4[1]),
                       pack_bf16x2(y[i].z * r * g4[2], y[i].w * r * g4[3]));
  }
}

// act[m][j] = bf16(silu(gate) * up) from the gate/up GEMM's stream-K partial
// sums: in 128-column tile t of the GEMM output, columns 0..63 are the gate
// values and 64..127 the up values of outputs 64 t .. 64 t + 63.  One thread
// per four outputs; the first kMaxGuSlots slots of both halves are requested
// together whatever the tile's slot count (unused ones are masked out).
constexpr int kMaxGuSlots = 4;

__global__ void __launch_bounds__(256) swiglu_kernel(const float* __restrict__ part, int slots,
                                                     const int* __restrict__ pieces, int tile_rows, int n_tiles,
                                                     int M, int I, __nv_bfloat16* __restrict__ act) {
  pdl_wait_primary();  // the partial sums of the gate/up GEMM
  pdl_launch_dependents();
  pieces = pdl_fresh(pieces);
  const long t = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int q4 = I / 4;
  if (t >= static_cast<long>(M) * q4) return;
  const int m = static_cast<int>(t / q4), j = static_cast<int>(t % q4) * 4;
  const int tile = j / 64;
  const size_t N = static_cast<size_t>(2) * I;
  const size_t slot = static_cast<size_t>(M) * N;
  const float* g = part + static_cast<size_t>(m) * N + static_cast<size_t>(tile) * 128 + (j % 64);
  const int ns = pieces[(m / tile_rows) * n_tiles + tile];
  float4 gu[kMaxGuSlots], uu[kMaxGuSlots];
#pragma unroll
  for (int k = 0; k < kMaxGuSlots; ++k) {
    gu[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    uu[k] = gu[k];
    if (k < slots) {
      gu[k] = __ldcg(reinterpret_cast<const float4*>(g + k * slot));
      uu[k] = __ldcg(reinterpret_cast<const float4*>(g + k * slot + 64));
    }
  }
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
#pragma unroll
  for (int k = 0; k < kMaxGuSlots; ++k)
    if (k < ns) {
      a.x += gu[k].x; a.y += gu[k].y; a.z += gu[k].z; a.w += gu[k].w;
      b.x += uu[k].x; b.y += uu[k].y; b.z += uu[k].z; b.w += uu[k].w;
    }
  for (int k = kMaxGuSlots; k < ns; ++k) {  // more slots than kept in registers
    const float4 x = __ldcg(reinterpret_cast<const float4*>(g + k * slot));
    const float4 y = __ldcg(reinterpret_cast<const float4*>(g + k * slot + 64));
    a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
  }
  // the gate and up lines (eight threads of this warp each) are read for the
  // last time: a whole warp drops them from L2 rather than let them be written back
  if (((t | 31) < static_cast<long>(M) * q4)) {
    __syncwarp();
    if (j % 32 == 0) {
      const int nread = max(ns, min(slots, kMaxGuSlots));
      for (int k = 0; k < nread; ++k) {
        discard_l2_line(g + k * slot);
        discard_l2_line(g + k * slot + 64);
      }
    }
  }
  // silu(g) = g / (1 + e^-g) with the approximate divide (relative error a
  // few units in the last place); it gives 0 once e^-g exceeds 2^126
  auto silu = [](float x) { return __fdividef(x, 1.0f + __expf(-x)); };
  reinterpret_cast<uint2*>(act + static_cast<size_t>(m) * I + j)[0] =
      make_uint2(pack_bf16x2(silu(a.x) * b.x, silu(a.y) * b.y), pack_bf16x2(silu(a.z) * b.z, silu(a.w) * b.w));
}

// q/k/v of the block rows from the projection's stream-K partial sums: one
// thread per four consecutive outputs of a row (a warp covers one 128-wide
// head row, 256 contiguous bytes stored); 128-column tile t of the GEMM output
// is head t: query heads first, then key heads, then value heads.  The first
// kMaxQkvSlots slots are requested together whatever the tile's slot count
// (unused ones are masked out), then the lines are dropped from L2.
constexpr int kMaxQkvSlots = 4;

__global__ void __launch_bounds__(256) qkv_scatter_kernel(const float* __restrict__ part, int slots,
                                                          const int* __restrict__ pieces, int tile_rows, int M,
                                                          int bs, int Hq, int Hkv, __nv_bfloat16* __restrict__ q,
                                                          __nv_bfloat16* __restrict__ kb,
                                                          __nv_bfloat16* __restrict__ vb) {
  pdl_wait_primary();  // the partial sums of the projection
  pdl_launch_dependents();
  pieces = pdl_fresh(pieces);
  const int heads = Hq + 2 * Hkv;
  const int q4 = heads * 32;  // four outputs per thread
  const long t = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<long>(M) * q4) return;
  const int m = static_cast<int>(t / q4), c = static_cast<int>(t % q4) * 4;
  const int head = c / 128, e = c % 128;
  const size_t N = static_cast<size_t>(heads) * 128;
  const size_t slot = static_cast<size_t>(M) * N;
  const float* src = part + static_cast<size_t>(m) * N + c;
  const int ns = pieces[(m / tile_rows) * heads + head];
  float4 u[kMaxQkvSlots];
#pragma unroll
  for (int k = 0; k < kMaxQkvSlots; ++k) {
    u[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < slots) u[k] = __ldcg(reinterpret_cast<const float4*>(src + k * slot));
  }
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMaxQkvSlots; ++k)
    if (k < ns) {
      a.x += u[k].x; a.y += u[k].y; a.z += u[k].z; a.w += u[k].w;
    }
  for (int k = kMaxQkvSlots; k < ns; ++k) {  // more slots than kept in registers
    const float4 x = __ldcg(reinterpret_cast<const float4*>(src + k * slot));
    a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
  }
  // a 128-byte line of a slot is read by eight consecutive threads of this
  // warp, for the last time: the first of them drops it from L2
  if ((t | 31) < static_cast<long>(M) * q4) {
    __syncwarp();
    if (e % 32 == 0) {
      const int nread = max(ns, min(slots, kMaxQkvSlots));
      for (int k = 0; k < nread; ++k) discard_l2_line(src + k * slot);
    }
  }
  const int b = m / bs, j = m % bs;
  __nv_bfloat16* dst;
  if (head < Hq)
    dst = q + ((static_cast<size_t>(b) * Hq + head) * bs + j) * 128;
  else if (head < Hq + Hkv)
    dst = kb + ((static_cast<size_t>(b) * Hkv + (head - Hq)) * bs + j) * 128;
  else
    dst = vb + ((static_cast<size_t>(b) * Hkv + (head - Hq - Hkv)) * bs + j) * 128;
  reinterpret_cast<uint2*>(dst + e)[0] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
}

struct TailPlan {
  int mt, m_tiles, ks_o, ks_down;
  int gu_shares, gu_slots;  // gate/up: stream-K over gu_shares CTAs into gu_slots slots
};

TailPlan tail_plan(int M, int D, int Kq, int I) {
  TailPlan t;
  t.mt = M <= 2 * kBM ? 2 : 1;
  t.m_tiles = (M + t.mt * kBM - 1) / (t.mt * kBM);
  const int tiles = t.m_tiles * (D / 128);
  const int ks = std::max(1, std::min(kMaxKSplits, kSplitTarget / std::max(1, tiles)));
  t.ks_o = std::min(ks, Kq / kBK);
  t.ks_down = std::min(ks, I / kBK);
  t.gu_shares = fixup_shares(t.m_tiles * (2 * I / 128), D / kBK);
  t.gu_slots = sk_max_count(static_cast<long>(t.m_tiles) * (2 * I / 128), D / kBK, t.gu_shares);
  return t;
}

dflash_status launch_resnorm(const float* part, int k_splits, int M, int D, __nv_bfloat16* x, int write_x, int g_mode,
                             const __nv_bfloat16* g, float eps, __nv_bfloat16* h, int* zero_flags, int n_zero,
                             cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  const int nv = D / 4;
  cfg.blockDim = dim3(static_cast<unsigned>(std::min(kResMaxThreads, ((nv + kResSlots - 1) / kResSlots + 31) / 32 * 32)));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, resnorm_kernel, part, k_splits, M, D, x, write_x, g_mode, g, eps, h,
                                     zero_flags, n_zero);
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "resnorm_kernel launch");
}

template <int MT>
dflash_status run_gemm(const TmapPack& am, const CUtensorMap& bm, const GemmArgs& a, cudaStream_t st,
                       const DeviceInfo& dev) {
  return MT == 2 ? launch_gemm<128, 4, 2>(am, bm, a, st, dev) : launch_gemm<128, 6, 1>(am, bm, a, st, dev);
}

}  // namespace

// fp32 partial sums: the output projection's and the down projection's split-K
// slots, and the gate/up GEMM's stream-K slots, share one buffer (each set is
// read before the next GEMM's epilogue writes, the launches being chained).
size_t tail_part_floats(const TailPlan& t, int M, int D, int I) {
  return std::max(static_cast<size_t>(std::max(t.ks_o, t.ks_down)) * M * D,
                  static_cast<size_t>(t.gu_slots) * M * 2 * I);
}

size_t tail_ws_bytes(int M, int D, int Hq, int I) {
  const TailPlan t = tail_plan(M, D, Hq * 128, I);
  return align256(tail_part_floats(t, M, D, I) * sizeof(float)) +
         align256(static_cast<size_t>(t.m_tiles) * (2 * I / 128) * sizeof(int)) +
         align256(static_cast<size_t>(M) * D * sizeof(__nv_bfloat16)) +
         align256(static_cast<size_t>(M) * I * sizeof(__nv_bfloat16)) + 256;
}

dflash_status launch_layer_tail(void* x, const void* attn_out, int B, int bs, int Hq, int D, int I, const void* w_o,
                                const void* g_post, const void* w_gate_up, const void* w_down, float eps, void* ws,
                                cudaStream_t st, const DeviceInfo& dev) {
  const int M = B * bs, Kq = Hq * 128;
  const TailPlan t = tail_plan(M, D, Kq, I);
  WsCarver w(ws);
  float* part = w.take<float>(tail_part_floats(t, M, D, I));
  int* gu_pieces = w.take<int>(static_cast<size_t>(t.m_tiles) * (2 * I / 128));
  auto* h = w.take<__nv_bfloat16>(static_cast<size_t>(M) * D);
  auto* act = w.take<__nv_bfloat16>(static_cast<size_t>(M) * I);
  auto* xb = static_cast<__nv_bfloat16*>(x);

  // 1. output projection, A through a 4D map of the attention output
  TmapPack am{};
  dflash_status s = make_tmap_bf16_4d(&am.a[0], attn_out, static_cast<uint64_t>(bs), static_cast<uint64_t>(Hq),
                                      static_cast<uint64_t>(B), static_cast<uint32_t>(bs),
                                      static_cast<uint32_t>(kBM / bs));
  if (s) return s;
  CUtensorMap bm;
  s = make_tmap_bf16_2d(&bm, w_o, static_cast<uint64_t>(D), Kq, 128, kBK);
  if (s) return s;
  GemmArgs a{};
  a.M = M;
  a.N = D;
  a.num_kb = Kq / kBK;
  a.kb_per_seg = a.num_kb;
  a.k_splits = t.ks_o;
  a.m_tiles = t.m_tiles;
  a.n_tiles = D / 128;
  a.epi = 0;
  a.a4d_bs = bs;
  a.pdl = 1;  // the attention output is loaded only once the preceding grid has completed;
  a.prefetch_b = 1;  // the weights, which no kernel of the chain writes, before that
  a.out_f32 = part;
  a.status = dev.status;
  s = t.mt == 2 ? run_gemm<2>(am, bm, a, st, dev) : run_gemm<1>(am, bm, a, st, dev);
  if (s) return s;
  // 2. residual + post-attention norm
  s = launch_resnorm(part, t.ks_o, M, D, xb, 1, 1, static_cast<const __nv_bfloat16*>(g_post), eps, h, nullptr, 0, st);
  if (s) return s;
  // 3. gate/up with SwiGLU
  TmapPack hm{};
  s = make_tmap_bf16_2d(&hm.a[0], h, static_cast<uint64_t>(M), D, kBM, kBK);
  if (s) return s;
  CUtensorMap gm;
  s = make_tmap_bf16_2d(&gm, w_gate_up, static_cast<uint64_t>(2) * I, D, 128, kBK);
  if (s) return s;
  GemmArgs gu{};
  gu.M = M;
  gu.N = 2 * I;
  gu.num_kb = D / kBK;
  gu.kb_per_seg = gu.num_kb;
  gu.m_tiles = t.m_tiles;
  gu.n_tiles = 2 * I / 128;
  gu.epi = 0;
  gu.stream_k = t.gu_shares;
  gu.dp_tiles = 0;
  gu.k_splits = t.gu_slots;
  gu.pieces = gu_pieces;
  gu.out_f32 = part;
  gu.pdl = 1;
  gu.prefetch_b = 1;
  gu.status = dev.status;
  s = t.mt == 2 ? run_gemm<2>(hm, gm, gu, st, dev) : run_gemm<1>(hm, gm, gu, st, dev);
  if (s) return s;
  {  // the SwiGLU over the gate/up partial sums
    cudaLaunchConfig_t cfg = {};
    const long threads = static_cast<long>(M) * (I / 4);
    cfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, swiglu_kernel, static_cast<const float*>(part), t.gu_slots,
                                       static_cast<const int*>(gu_pieces), t.mt * kBM, 2 * I / 128, M, I, act);
    if (e != cudaSuccess) return cuda_fail(e, "swiglu_kernel launch");
  }
  // 4. down projection
  TmapPack xm{};
  s = make_tmap_bf16_2d(&xm.a[0], act, static_cast<uint64_t>(M), I, kBM, kBK);
  if (s) return s;
  CUtensorMap dm;
  s = make_tmap_bf16_2d(&dm, w_down, static_cast<uint64_t>(D), I, 128, kBK);
  if (s) return s;
  GemmArgs dn{};
  dn.M = M;
  dn.N = D;
  dn.num_kb = I / kBK;
  dn.kb_per_seg = dn.num_kb;
  dn.k_splits = t.ks_down;
  dn.m_tiles = t.m_tiles;
  dn.n_tiles = D / 128;
  dn.epi = 0;
  dn.pdl = 1;
  dn.prefetch_b = 1;
  dn.out_f32 = part;
  dn.status = dev.status;
  s = t.mt == 2 ? run_gemm<2>(xm, dm, dn, st, dev) : run_gemm<1>(xm, dm, dn, st, dev);
  if (s) return s;
  // 5. residual
  return launch_resnorm(part, t.ks_down, M, D, xb, 1, 0, nullptr, eps, nullptr, nullptr, 0, st);
}

struct QkvPlan {
  int mt, m_tiles, heads, shares, slots;
};

QkvPlan qkv_plan(int M, int D, int Hq, int Hkv) {
  QkvPlan p;
  p.mt = M <= 2 * kBM ? 2 : 1;
  p.m_tiles = (M + p.mt * kBM - 1) / (p.mt * kBM);
  p.heads = Hq + 2 * Hkv;
  p.shares = fixup_shares(p.m_tiles * p.heads, D / kBK);
  p.slots = sk_max_count(static_cast<long>(p.m_tiles) * p.heads, D / kBK, p.shares);
  return p;
}

size_t qkv_ws_bytes(int M, int D, int Hq, int Hkv) {
  const QkvPlan p = qkv_plan(M, D, Hq, Hkv);
  return align256(static_cast<size_t>(p.slots) * M * p.heads * 128 * sizeof(float)) +
         align256(static_cast<size_t>(p.m_tiles) * p.heads * sizeof(int)) +
         align256(static_cast<size_t>(M) * D * sizeof(__nv_bfloat16)) + 256;
}

dflash_status launch_layer_qkv(const void* x, int B, int bs, int D, int Hq, int Hkv, const void* g_in, float eps,
                               const void* w_qkv, void* q, void* kb, void* vb, void* ws, cudaStream_t st,
                               const DeviceInfo& dev) {
  const int M = B * bs;
  const QkvPlan pl = qkv_plan(M, D, Hq, Hkv);
  const int N = pl.heads * 128;
  WsCarver w(ws);
  float* part = w.take<float>(static_cast<size_t>(pl.slots) * M * N);
  int* pieces = w.take<int>(static_cast<size_t>(pl.m_tiles) * pl.heads);
  auto* h = w.take<__nv_bfloat16>(static_cast<size_t>(M) * D);
  // 1. input norm: h = bf16(RMSNorm(x) * g_in); x is only read
  dflash_status s = launch_resnorm(nullptr, 0, M, D, const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(x)),
                                   0, 1, static_cast<const __nv_bfloat16*>(g_in), eps, h, nullptr, 0, st);
  if (s) return s;
  // 2. the projections, stream-K into slots
  TmapPack hm{};
  s = make_tmap_bf16_2d(&hm.a[0], h, static_cast<uint64_t>(M), D, kBM, kBK);
  if (s) return s;
  CUtensorMap wm;
  s = make_tmap_bf16_2d(&wm, w_qkv, static_cast<uint64_t>(N), D, 128, kBK);
  if (s) return s;
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.num_kb = D / kBK;
  a.kb_per_seg = a.num_kb;
  a.m_tiles = pl.m_tiles;
  a.n_tiles = pl.heads;
  a.epi = 0;
  a.stream_k = pl.shares;
  a.dp_tiles = 0;
  a.k_splits = pl.slots;
  a.pieces = pieces;
  a.out_f32 = part;
  a.pdl = 1;
  a.prefetch_b = 1;  // the weights, which no kernel of the chain writes, before the wait
  a.status = dev.status;
  s = pl.mt == 2 ? run_gemm<2>(hm, wm, a, st, dev) : run_gemm<1>(hm, wm, a, st, dev);
  if (s) return s;
  // 3. the heads into the block attention's layouts
  cudaLaunchConfig_t cfg = {};
  const long threads = static_cast<long>(M) * pl.heads * 32;
  cfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, qkv_scatter_kernel, static_cast<const float*>(part), pl.slots,
                                     static_cast<const int*>(pieces), pl.mt * kBM, M, bs, Hq, Hkv,
                                     static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(kb),
                                     static_cast<__nv_bfloat16*>(vb));
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "qkv_scatter_kernel launch");
}

}  // namespace dflash
