// Host-side declarations shared by the translation units of libdflash.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <string>

#include "../../include/dflash.h"

namespace dflash {

// --- errors ----------------------------------------------------------------
void set_error(const std::string& msg);
dflash_status fail(dflash_status code, const std::string& msg);
dflash_status cuda_fail(cudaError_t err, const char* what);

// --- device facts, cached per device --------------------------------------
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  size_t max_smem_optin = 0;
  unsigned* status = nullptr;  // address of the library's device status word
};
dflash_status device_info(DeviceInfo* out);

// --- kernel attributes ---------------------------------------------------------
constexpr int kAttrMaxDevices = 64;

// Raises Kernel's dynamic shared-memory limit to at least `bytes` on `device`
// (the current device), once per kernel, device and process.  Safe to call
// from several host threads: each device has its own atomic record, and two
// threads racing on a first call both set the same (idempotent) attribute.
template <auto Kernel>
dflash_status smem_limit_once(int device, int bytes, const char* what) {
  static std::atomic<int> done[kAttrMaxDevices];
  if (device < 0 || device >= kAttrMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device index out of range");
  if (done[device].load(std::memory_order_acquire) >= bytes) return DFLASH_OK;
  const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, what);
  int cur = done[device].load(std::memory_order_relaxed);
  while (cur < bytes && !done[device].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
  }
  return DFLASH_OK;
}

// --- TMA descriptors --------------------------------------------------------
// 2D row-major bf16 tensor [rows][cols] with a (box_cols x box_rows) box and
// the 128-byte swizzle (box_cols * 2 must be 128).  Out-of-range rows read 0.
dflash_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_cols);
dflash_status make_tmap_bf16_4d(CUtensorMap* map, const void* base, uint64_t d1, uint64_t d2, uint64_t d3,
                                uint32_t b1, uint32_t b3);

// Workspace carving: 256-byte aligned sub-buffers.
struct WsCarver {
  uintptr_t base;
  size_t used = 0;
  explicit WsCarver(void* p) : base(reinterpret_cast<uintptr_t>(p)) {}
  template <typename T>
  T* take(size_t count) {
    used = (used + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base + used);
    used += count * sizeof(T);
    return p;
  }
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// --- verify ------------------------------------------------------------------
size_t verify_ws_bytes(int B, int bs, int V);
dflash_status launch_verify(const void* lt, const void* ld, dflash_dtype dt, const int32_t* x, int B,
                            int bs, int V, float T, uint64_t seed, uint64_t cycle, int32_t* acc,
                            int32_t* out, void* ws, cudaStream_t st, const DeviceInfo& dev);

// --- block attention ---------------------------------------------------------
size_t attn_ws_bytes(int B, int bs, int Hq, int Hkv, int cap, int window, dflash_dtype dt);
dflash_status launch_block_attn(int layer, int B, int bs, int Hq, const void* q, const void* kb,
                                const void* vb, const void* qg, const void* kg, float theta,
                                float eps, const dflash_kv_cache& c, int window, void* out, void* ws,
                                cudaStream_t st, const DeviceInfo& dev);

dflash_status launch_attn_wait_timeout_probe(int B, int bs, int Hq, const dflash_kv_cache& c, void* out, void* ws,
                                             unsigned long long limit_ns, cudaStream_t st, const DeviceInfo& dev);

// --- drafter head ------------------------------------------------------------
size_t head_ws_bytes(int M, int D, int V);
dflash_status launch_draft_head(const void* x, int B, int rows_per_seq, int D, const void* g_final, float eps,
                                const void* w_head, int V, float T, uint64_t seed, uint64_t cycle, void* logits,
                                int32_t* tokens, void* ws, cudaStream_t st, const DeviceInfo& dev);

// --- draft layer remainder ---------------------------------------------------
size_t tail_ws_bytes(int M, int D, int Hq, int I);
dflash_status launch_layer_tail(void* x, const void* attn_out, int B, int bs, int Hq, int D, int I, const void* w_o,
                                const void* g_post, const void* w_gate_up, const void* w_down, float eps, void* ws,
                                cudaStream_t st, const DeviceInfo& dev);

size_t qkv_ws_bytes(int M, int D, int Hq, int Hkv);
dflash_status launch_layer_qkv(const void* x, int B, int bs, int D, int Hq, int Hkv, const void* g_in, float eps,
                               const void* w_qkv, void* q, void* kb, void* vb, void* ws, cudaStream_t st,
                               const DeviceInfo& dev);

// --- DFlash2 variants ----------------------------------------------------------
dflash_status launch_block_conv(const void* h, int B, int bs, int D, int k, const void* w, const void* bias,
                                int residual, void* out, cudaStream_t st);
size_t topm_ws_bytes(int B, int R, int V, int m);
int topm_max_m();
dflash_status launch_draft_topm(const void* logits, int B, int R, int V, int m, float T, float lambda,
                                int32_t* idx, float* logp, float* ent, float* score, void* ws, cudaStream_t st);

// --- context fusion ----------------------------------------------------------
size_t fuse_ws_bytes(int M, int J, int dt_width, int D, int L, int Hkv, dflash_dtype dt);
dflash_status launch_fuse_context(int J, const void* const* taps, int dt_width, const int32_t* cu_new,
                                  int B, int M, const void* w_fuse, const void* g_fuse, int D,
                                  const void* w_kv, const void* k_gain, float theta, float eps,
                                  const dflash_kv_cache& c, void* h_t_out, void* ws,
                                  cudaStream_t st, const DeviceInfo& dev);

// --- diagnostics --------------------------------------------------------------
dflash_status launch_philox(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out, int n,
                            cudaStream_t st);

}  // namespace dflash
