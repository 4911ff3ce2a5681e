// The drafter's head: final RMSNorm, LM head and draft sampling.
//
// Pages: "Nemotron 3.5 Bolt E4B: Block-Parallel Speculation with DFlash",
// section "The released serving cycle" (the drafter proposes the block's
// tokens from its final hidden states through its LM head) and section "The
// parameter count exposes the real cost" (the V x D head is most of the
// drafter's weights).
//
// Three launches chained as programmatic dependents:
//   1. head_norm    H = bf16(RMSNorm(x) * g_final), one CTA per proposal row
//   2. gemm_tc      logits = H W_head^T on tcgen05 tensor cores: 256-row by
//                   128-column units (every W_head tile read once for up to
//                   256 rows); the epilogue stores the bf16 logits and, per
//                   row and 128-column tile, the best key of the draft race
//   3. race_reduce  per row, the best key over the tiles -> the draft token
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "dflash_device.cuh"
#include "dflash_internal.h"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

constexpr int kHeadNormThreads = 256;
constexpr int kHeadBN = 128;

// One CTA per row: H[m] = bf16(x[m] * rsqrt(mean(x[m]^2) + eps) * g), with
// 16-byte loads (D % 8 == 0); the row is read twice (the second time from L1).
__global__ void __launch_bounds__(kHeadNormThreads) head_norm_kernel(const __nv_bfloat16* __restrict__ x, int D,
                                                                    const __nv_bfloat16* __restrict__ g, float eps,
                                                                    __nv_bfloat16* __restrict__ h) {
  pdl_wait_primary();  // a programmatic dependent of the preceding kernel: nothing is read before it completed
  pdl_launch_dependents();
  x = pdl_fresh(x);
  g = pdl_fresh(g);
  const int m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * D);
  const int nv = D / 8;
  float ss = 0.f;
  for (int v = threadIdx.x; v < nv; v += kHeadNormThreads) {
    const uint4 u = xr[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
      ss += a * a + b * b;
    }
  }
  ss = warp_sum(ss);
  __shared__ float red[kHeadNormThreads / 32];
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kHeadNormThreads / 32; ++w) tot += red[w];
  const float r = rsqrtf(tot / static_cast<float>(D) + eps);
  uint4* hr = reinterpret_cast<uint4*>(h + static_cast<size_t>(m) * D);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  for (int v = threadIdx.x; v < nv; v += kHeadNormThreads) {
    const uint4 u = xr[v];
    const uint4 gu = g ? gr[v] : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w}, gw[4] = {gu.x, gu.y, gu.z, gu.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_bf16x2(bf16_lo(w[i]) * r * bf16_lo(gw[i]), bf16_hi(w[i]) * r * bf16_hi(gw[i]));
    hr[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// One warp per row: the best (key, column) over the row's tiles, ties to the
// lowest column.
__global__ void __launch_bounds__(256) race_reduce_kernel(const float2* __restrict__ race, int M, int n_tiles,
                                                          int32_t* __restrict__ tokens) {
  pdl_wait_primary();
  pdl_launch_dependents();
  race = pdl_fresh(race);
  const int row = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row >= M) return;
  float best = -INFINITY;
  int col = INT_MAX;
  for (int t = lane; t < n_tiles; t += 32) {
    const float2 v = race[static_cast<size_t>(row) * n_tiles + t];
    const int c = __float_as_int(v.y);
    if (v.x > best || (v.x == best && c < col)) {
      best = v.x;
      col = c;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int c2 = __shfl_xor_sync(0xffffffffu, col, o);
    if (b2 > best || (b2 == best && c2 < col)) {
      best = b2;
      col = c2;
    }
  }
  if (lane == 0) tokens[row] = col == INT_MAX ? 0 : col;
}

dflash_status launch_pdl(const void* fn, dim3 grid, dim3 block, cudaStream_t st, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "draft head launch");
}

}  // namespace

size_t head_ws_bytes(int M, int D, int V) {
  const size_t n_tiles = static_cast<size_t>(V) / kHeadBN;
  return align256(static_cast<size_t>(M) * D * sizeof(__nv_bfloat16)) +
         align256(static_cast<size_t>(M) * n_tiles * sizeof(float2)) + 256;
}

dflash_status launch_draft_head(const void* x, int B, int rows_per_seq, int D, const void* g_final, float eps,
                                const void* w_head, int V, float T, uint64_t seed, uint64_t cycle, void* logits,
                                int32_t* tokens, void* ws, cudaStream_t st, const DeviceInfo& dev) {
  const int M = B * rows_per_seq;
  const int n_tiles = V / kHeadBN;
  WsCarver w(ws);
  auto* H = w.take<__nv_bfloat16>(static_cast<size_t>(M) * D);
  float2* race = w.take<float2>(static_cast<size_t>(M) * n_tiles);

  {  // 1. final norm
    const __nv_bfloat16* xa = static_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* ga = static_cast<const __nv_bfloat16*>(g_final);
    int Da = D;
    float ea = eps;
    void* args[] = {&xa, &Da, &ga, &ea, &H};
    dflash_status s = launch_pdl(reinterpret_cast<const void*>(head_norm_kernel), dim3(M), dim3(kHeadNormThreads),
                                 st, args);
    if (s) return s;
  }
  // 2. LM head with the draft race in its epilogue
  TmapPack am{};
  dflash_status s = make_tmap_bf16_2d(&am.a[0], H, static_cast<uint64_t>(M), D, kBM, kBK);
  if (s) return s;
  CUtensorMap bm;
  s = make_tmap_bf16_2d(&bm, w_head, static_cast<uint64_t>(V), D, kHeadBN, kBK);
  if (s) return s;
  GemmArgs a{};
  a.M = M;
  a.N = V;
  a.num_kb = D / kBK;
  a.kb_per_seg = a.num_kb;
  a.k_splits = 1;
  a.m_tiles = (M + 2 * kBM - 1) / (2 * kBM);
  a.n_tiles = n_tiles;
  a.epi = 2;
  a.pdl = 1;
  a.prefetch_b = 1;  // the head's weights do not depend on the norm kernel
  a.logits = static_cast<__nv_bfloat16*>(logits);
  a.race = race;
  a.inv_temp = T > 0.0f ? 1.0f / T : 0.0f;
  a.rows_per_seq = rows_per_seq;
  a.seed_lo = static_cast<uint32_t>(seed);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  a.cycle_lo = static_cast<uint32_t>(cycle);
  a.cycle_hi = static_cast<uint32_t>(cycle >> 32) & 0x7FFFFFFFu;
  a.status = dev.status;
  s = launch_gemm<kHeadBN, 4, 2>(am, bm, a, st, dev);
  if (s) return s;
  // 3. the draft tokens
  {
    const float2* ra = race;
    int Ma = M, nt = n_tiles;
    int32_t* ta = tokens;
    void* args[] = {&ra, &Ma, &nt, &ta};
    return launch_pdl(reinterpret_cast<const void*>(race_reduce_kernel), dim3((M + 7) / 8), dim3(256), st, args);
  }
}

}  // namespace dflash
