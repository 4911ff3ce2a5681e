// C ABI entry points of libdflash: host-side validation, workspace sizing,
// device facts, TMA descriptor encoding and the library's device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>

#include "dflash_device.cuh"
#include "dflash_internal.h"

namespace dflash {

// The library's device status word (DFLASH_DEV_* bits).  Kernels receive its
// address; dflash_read_device_status() reads and clears it.
__device__ unsigned g_device_status;

static thread_local std::string t_last_error;

void set_error(const std::string& msg) { t_last_error = msg; }

dflash_status fail(dflash_status code, const std::string& msg) {
  t_last_error = msg;
  return code;
}

dflash_status cuda_fail(cudaError_t err, const char* what) {
  t_last_error = std::string(what) + ": " + cudaGetErrorName(err) + " (" + cudaGetErrorString(err) + ")";
  return DFLASH_ERR_CUDA;
}

static constexpr int kMaxDevices = 64;
static DeviceInfo g_dev[kMaxDevices];
static std::mutex g_dev_mu;

dflash_status device_info(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device != dev) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (major != 10 || minor != 3)
      return fail(DFLASH_ERR_UNSUPPORTED, "libdflash is built for sm_103a (GB300); device " +
                                              std::to_string(dev) + " is sm_" +
                                              std::to_string(major) + std::to_string(minor));
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    d.num_sms = sms;
    d.max_smem_optin = static_cast<size_t>(smem);
    d.status = static_cast<unsigned*>(p);
    d.device = dev;
  }
  *out = d;
  return DFLASH_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

dflash_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (box_cols * 2 != 128) return fail(DFLASH_ERR_UNSUPPORTED, "TMA box must be 128 bytes wide");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((cols * 2) & 15))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "TMA tensor base and row pitch must be 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return DFLASH_OK;
}

// A [d3][d2][d1][128] bf16 tensor (d0 = 128 elements innermost) read in boxes of
// 64 x b1 x 1 x b3 elements, 128-byte swizzle: the rows of a box are (d3, d1)
// pairs of 128 bytes, as a 2D box of b1 * b3 rows.
dflash_status make_tmap_bf16_4d(CUtensorMap* map, const void* base, uint64_t d1, uint64_t d2, uint64_t d3,
                                uint32_t b1, uint32_t b3) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (reinterpret_cast<uintptr_t>(base) & 15) return fail(DFLASH_ERR_INVALID_ARGUMENT, "TMA tensor base must be 16-byte aligned");
  cuuint64_t dims[4] = {128, d1, d2, d3};
  cuuint64_t strides[3] = {128 * 2, d1 * 128 * 2, d2 * d1 * 128 * 2};
  cuuint32_t box[4] = {64, b1, 1, b3};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled (4D) failed with CUresult " + std::to_string(r));
  return DFLASH_OK;
}

// --- philox diagnostic kernel -------------------------------------------------

__global__ void philox_kernel(const uint4* ctr, uint32_t k0, uint32_t k1, uint4* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = philox4x32_10(ctr[i], k0, k1);
}

dflash_status launch_philox(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out, int n,
                            cudaStream_t st) {
  if (n == 0) return DFLASH_OK;
  philox_kernel<<<(n + 255) / 256, 256, 0, st>>>(reinterpret_cast<const uint4*>(ctr), k0, k1,
                                                  reinterpret_cast<uint4*>(out), n);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH_OK : cuda_fail(e, "philox_kernel launch");
}

}  // namespace dflash

using namespace dflash;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
static bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255) == 0; }

static dflash_status check_cache(const dflash_kv_cache* c) {
  if (!c) return fail(DFLASH_ERR_INVALID_ARGUMENT, "cache descriptor is NULL");
  if (!c->k || !c->v || !c->seq_len) return fail(DFLASH_ERR_INVALID_ARGUMENT, "cache k/v/seq_len is NULL");
  if (c->num_layers < 1 || c->batch < 1 || c->num_kv_heads < 1 || c->capacity < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "cache sizes must be positive");
  if (c->head_dim != 128) return fail(DFLASH_ERR_UNSUPPORTED, "head_dim must be 128");
  if (c->dtype != DFLASH_F32 && c->dtype != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "cache dtype");
  if (!aligned16(c->k) || !aligned16(c->v)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "cache k/v must be 16-byte aligned");
  if (c->ring != 0 && c->ring != 1) return fail(DFLASH_ERR_INVALID_ARGUMENT, "cache ring must be 0 or 1");
  if (c->block_table) {  // paged layout
    if (c->dtype != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "a paged cache must be bf16");
    if (c->ring) return fail(DFLASH_ERR_UNSUPPORTED, "a paged cache cannot be a ring");
    if (c->page_size < 128 || c->page_size % 128 != 0)
      return fail(DFLASH_ERR_UNSUPPORTED, "page_size must be a positive multiple of 128");
    if (c->num_pages < 1 || c->max_pages < 1)
      return fail(DFLASH_ERR_INVALID_ARGUMENT, "num_pages and max_pages must be positive");
    if (static_cast<long long>(c->max_pages) * c->page_size != c->capacity)
      return fail(DFLASH_ERR_INVALID_ARGUMENT, "capacity must equal max_pages * page_size");
    const double prow = double(c->num_layers) * c->num_pages * c->num_kv_heads * c->page_size;
    if (prow >= 2147483647.0) return fail(DFLASH_ERR_UNSUPPORTED, "cache has 2^31 or more rows");
    return DFLASH_OK;
  }
  const double rows = double(c->num_layers) * c->batch * c->num_kv_heads * c->capacity;
  if (rows >= 2147483647.0) return fail(DFLASH_ERR_UNSUPPORTED, "cache has 2^31 or more rows");
  return DFLASH_OK;
}

static dflash_status check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return DFLASH_OK;
  if (!ws) return fail(DFLASH_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned256(ws)) return fail(DFLASH_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (have < need)
    return fail(DFLASH_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) +
                                          " bytes, have " + std::to_string(have));
  return DFLASH_OK;
}

extern "C" {

int dflash_version(void) { return (1 << 16) | 3; }

const char* dflash_last_error_string(void) { return t_last_error.c_str(); }

dflash_status dflash_read_device_status(uint32_t* flags, void* stream) {
  if (!flags) return fail(DFLASH_ERR_INVALID_ARGUMENT, "flags is NULL");
  DeviceInfo dev;
  dflash_status s = device_info(&dev);
  if (s) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0, zero = 0;
  e = cudaMemcpy(&v, dev.status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  e = cudaMemcpy(dev.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear status word");
  *flags = v;
  return DFLASH_OK;
}

dflash_status dflash_philox4x32_10(const uint32_t* ctr, uint32_t key0, uint32_t key1, uint32_t* out,
                                   int n, void* stream) {
  if (n < 0) return fail(DFLASH_ERR_INVALID_ARGUMENT, "n < 0");
  if (n > 0 && (!ctr || !out)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL buffer");
  if (!aligned16(ctr) || !aligned16(out)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "buffers must be 16-byte aligned");
  DeviceInfo dev;
  dflash_status s = device_info(&dev);
  if (s) return s;
  return launch_philox(ctr, key0, key1, out, n, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- verify ----

size_t dflash_verify_workspace_size(int batch, int block_size, int vocab, dflash_dtype dtype) {
  (void)dtype;
  if (batch < 1 || block_size < 1 || vocab < 1) return 0;
  return verify_ws_bytes(batch, block_size, vocab);
}

dflash_status dflash_verify(const void* target_logits, const void* draft_logits, dflash_dtype dtype,
                            const int32_t* draft_tokens, int batch, int block_size, int vocab,
                            float temperature, uint64_t seed, uint64_t cycle, int32_t* accepted_len,
                            int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (dtype != DFLASH_F32 && dtype != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "dtype");
  if (batch < 0 || block_size < 1 || block_size > 16 || vocab < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0, 1 <= block_size <= 16, vocab >= 1");
  if (!(temperature >= 0.0f) || std::isinf(temperature))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "temperature must be finite and >= 0");
  if (batch == 0) return DFLASH_OK;
  if (!target_logits || !accepted_len || !out_tokens)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL target_logits / accepted_len / out_tokens");
  if (block_size > 1 && !draft_tokens) return fail(DFLASH_ERR_INVALID_ARGUMENT, "draft_tokens is NULL");
  if (temperature > 0.0f && block_size > 1 && !draft_logits)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "draft_logits is NULL with temperature > 0");
  if (double(batch) * block_size * vocab >= 9.0e15) return fail(DFLASH_ERR_UNSUPPORTED, "logits too large");
  const size_t need = verify_ws_bytes(batch, block_size, vocab);
  dflash_status s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_verify(target_logits, draft_logits, dtype, draft_tokens, batch, block_size, vocab,
                       temperature, seed, cycle, accepted_len, out_tokens, workspace,
                       static_cast<cudaStream_t>(stream), dev);
}

// ----------------------------------------------------------- block attn ----

size_t dflash_block_attn_workspace_size(int batch, int block_size, int num_q_heads, int num_kv_heads,
                                        int capacity, int window, dflash_dtype dtype) {
  if (batch < 1 || block_size < 1 || num_q_heads < 1 || num_kv_heads < 1 || capacity < 1) return 0;
  return attn_ws_bytes(batch, block_size, num_q_heads, num_kv_heads, capacity, window, dtype);
}

dflash_status dflash_block_attn(int layer, int batch, int block_size, int num_q_heads, const void* q,
                                const void* kb, const void* vb, const void* q_gain,
                                const void* k_gain, float rope_theta, float eps,
                                const dflash_kv_cache* cache, int window, void* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  dflash_status s = check_cache(cache);
  if (s) return s;
  if (batch != cache->batch) return fail(DFLASH_ERR_INVALID_ARGUMENT, "batch must equal cache->batch");
  if (layer < 0 || layer >= cache->num_layers) return fail(DFLASH_ERR_INVALID_ARGUMENT, "layer out of range");
  if (block_size < 1 || block_size > 16) return fail(DFLASH_ERR_UNSUPPORTED, "block_size must be 1..16");
  const int hkv = cache->num_kv_heads;
  if (num_q_heads < 1 || num_q_heads % hkv) return fail(DFLASH_ERR_INVALID_ARGUMENT, "num_q_heads % num_kv_heads != 0");
  if ((num_q_heads / hkv) * block_size > 64)
    return fail(DFLASH_ERR_UNSUPPORTED, "(num_q_heads/num_kv_heads) * block_size must be <= 64");
  if (window < 0) return fail(DFLASH_ERR_INVALID_ARGUMENT, "window < 0");
  if (cache->ring && window != 0)
    return fail(DFLASH_ERR_UNSUPPORTED, "a ring cache is its own window: window must be 0");
  if (cache->block_table && window != 0)
    return fail(DFLASH_ERR_UNSUPPORTED, "a paged cache takes window 0 (key tiles start on page boundaries)");
  if (!q || !kb || !vb || !out) return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL q/kb/vb/out");
  if (!aligned16(q) || !aligned16(kb) || !aligned16(vb) || !aligned16(out))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "q/kb/vb/out must be 16-byte aligned");
  if (!(rope_theta > 1.0f) || !(eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "rope_theta > 1, eps >= 0");
  const size_t need = attn_ws_bytes(batch, block_size, num_q_heads, hkv, cache->capacity, window, cache->dtype);
  s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_block_attn(layer, batch, block_size, num_q_heads, q, kb, vb, q_gain, k_gain,
                           rope_theta, eps, *cache, window, out, workspace,
                           static_cast<cudaStream_t>(stream), dev);
}

dflash_status dflash_debug_block_attn_wait_timeout(int batch, int block_size, int num_q_heads,
                                                  const dflash_kv_cache* cache, void* out, void* workspace,
                                                  size_t workspace_bytes, unsigned limit_us, void* stream) {
  dflash_status s = check_cache(cache);
  if (s) return s;
  if (cache->dtype != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "the wait probe runs the bf16 path");
  if (batch != cache->batch) return fail(DFLASH_ERR_INVALID_ARGUMENT, "batch must equal cache->batch");
  if (block_size < 1 || block_size > 16) return fail(DFLASH_ERR_UNSUPPORTED, "block_size must be 1..16");
  const int hkv = cache->num_kv_heads;
  if (num_q_heads < 1 || num_q_heads % hkv) return fail(DFLASH_ERR_INVALID_ARGUMENT, "num_q_heads % num_kv_heads != 0");
  if ((num_q_heads / hkv) * block_size > 64)
    return fail(DFLASH_ERR_UNSUPPORTED, "(num_q_heads/num_kv_heads) * block_size must be <= 64");
  if (!out || !aligned16(out)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "out must be 16-byte aligned");
  if (limit_us < 1 || limit_us > 100000) return fail(DFLASH_ERR_INVALID_ARGUMENT, "limit_us must be 1..100000");
  const size_t need = attn_ws_bytes(batch, block_size, num_q_heads, hkv, cache->capacity, 0, DFLASH_BF16);
  s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_attn_wait_timeout_probe(batch, block_size, num_q_heads, *cache, out, workspace,
                                        static_cast<unsigned long long>(limit_us) * 1000ull,
                                        static_cast<cudaStream_t>(stream), dev);
}

// ------------------------------------------------------- draft layer qkv ----

size_t dflash_draft_layer_qkv_workspace_size(int batch, int block_size, int num_q_heads, int num_kv_heads,
                                             int d_model) {
  if (batch < 1 || block_size < 1 || num_q_heads < 1 || num_kv_heads < 1 || d_model < 1) return 0;
  return qkv_ws_bytes(batch * block_size, d_model, num_q_heads, num_kv_heads);
}

dflash_status dflash_draft_layer_qkv(const void* x, int batch, int block_size, int num_q_heads, int num_kv_heads,
                                     int d_model, const void* g_in, float eps, const void* w_qkv, void* q, void* kb,
                                     void* vb, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || block_size < 1 || num_q_heads < 1 || num_kv_heads < 1 || d_model < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0 and positive sizes");
  if (batch == 0) return DFLASH_OK;
  if (d_model % 128 || d_model > 4096)
    return fail(DFLASH_ERR_UNSUPPORTED, "layer q/k/v needs d_model % 128 == 0 and d_model <= 4096");
  if (!(eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  if (!x || !w_qkv || !q || !kb || !vb) return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL x/w_qkv/q/kb/vb");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(kb) || !aligned16(vb) ||
      (g_in && !aligned16(g_in)))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "pointers must be 16-byte aligned");
  const size_t need = qkv_ws_bytes(batch * block_size, d_model, num_q_heads, num_kv_heads);
  dflash_status s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_layer_qkv(x, batch, block_size, d_model, num_q_heads, num_kv_heads, g_in, eps, w_qkv, q, kb, vb,
                          workspace, static_cast<cudaStream_t>(stream), dev);
}

// ------------------------------------------------------ draft layer tail ----

size_t dflash_draft_layer_tail_workspace_size(int batch, int block_size, int num_q_heads, int d_model,
                                              int mlp_dim) {
  if (batch < 1 || block_size < 1 || num_q_heads < 1 || d_model < 1 || mlp_dim < 1) return 0;
  return tail_ws_bytes(batch * block_size, d_model, num_q_heads, mlp_dim);
}

dflash_status dflash_draft_layer_tail(void* x, const void* attn_out, int batch, int block_size, int num_q_heads,
                                      int d_model, int mlp_dim, const void* w_o, const void* g_post,
                                      const void* w_gate_up, const void* w_down, float eps, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (batch < 0 || block_size < 1 || num_q_heads < 1 || d_model < 1 || mlp_dim < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0 and positive sizes");
  if (batch == 0) return DFLASH_OK;
  if (d_model % 128 || d_model > 4096 || mlp_dim % 64 || 128 % block_size)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "layer tail needs d_model % 128 == 0 (<= 4096), mlp_dim % 64 == 0, 128 % block_size == 0");
  if (!(eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  if (!x || !attn_out || !w_o || !w_gate_up || !w_down)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL x/attn_out/w_o/w_gate_up/w_down");
  if (!aligned16(x) || !aligned16(attn_out) || !aligned16(w_o) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      (g_post && !aligned16(g_post)))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "pointers must be 16-byte aligned");
  const size_t need = tail_ws_bytes(batch * block_size, d_model, num_q_heads, mlp_dim);
  dflash_status s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_layer_tail(x, attn_out, batch, block_size, num_q_heads, d_model, mlp_dim, w_o, g_post, w_gate_up,
                           w_down, eps, workspace, static_cast<cudaStream_t>(stream), dev);
}

// ----------------------------------------------------------- draft head ----

size_t dflash_draft_head_workspace_size(int batch, int rows_per_seq, int d_model, int vocab) {
  if (batch < 1 || rows_per_seq < 1 || d_model < 1 || vocab < 1) return 0;
  return head_ws_bytes(batch * rows_per_seq, d_model, vocab);
}

dflash_status dflash_draft_head(const void* x, int batch, int rows_per_seq, int d_model, const void* g_final,
                                float eps, const void* w_head, int vocab, float temperature, uint64_t seed,
                                uint64_t cycle, void* logits_out, int32_t* tokens_out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (batch < 0 || rows_per_seq < 1 || rows_per_seq > 31 || d_model < 1 || vocab < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0, 1 <= rows_per_seq <= 31, d_model, vocab >= 1");
  if (batch == 0) return DFLASH_OK;
  if (d_model % 64 || vocab % 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "draft head needs d_model % 64 == 0 and vocab % 128 == 0");
  if (double(batch) * rows_per_seq >= 65536.0 * 1024.0)
    return fail(DFLASH_ERR_UNSUPPORTED, "draft head: too many rows");
  if (!(temperature >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "temperature must be >= 0");
  if (!(eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  if (!x || !w_head || !logits_out || !tokens_out)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL x/w_head/logits_out/tokens_out");
  if (!aligned16(x) || !aligned16(w_head) || !aligned16(logits_out) || (g_final && !aligned16(g_final)))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "x, w_head, g_final and logits_out must be 16-byte aligned");
  const size_t need = head_ws_bytes(batch * rows_per_seq, d_model, vocab);
  dflash_status s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_draft_head(x, batch, rows_per_seq, d_model, g_final, eps, w_head, vocab, temperature, seed, cycle,
                           logits_out, tokens_out, workspace, static_cast<cudaStream_t>(stream), dev);
}

// ------------------------------------------------------- DFlash2 variants ----

dflash_status dflash_block_conv(const void* h, int batch, int block_size, int d_model, int kernel, const void* w,
                                const void* bias, int residual, void* out, void* stream) {
  if (batch < 0 || block_size < 1 || block_size > 16 || d_model < 1 || kernel < 1 || kernel > 8)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0, 1 <= block_size <= 16, d_model >= 1, 1 <= kernel <= 8");
  if (residual != 0 && residual != 1) return fail(DFLASH_ERR_INVALID_ARGUMENT, "residual must be 0 or 1");
  if (batch == 0) return DFLASH_OK;
  if (d_model % 4) return fail(DFLASH_ERR_UNSUPPORTED, "block_conv needs d_model % 4 == 0");
  if (!h || !w || !out) return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL h/w/out");
  auto a8 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7) == 0; };
  if (!a8(h) || !a8(w) || !a8(out) || (bias && !a8(bias)))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "h, w, bias and out must be 8-byte aligned");
  if (double(batch) * (d_model / 4) >= 2147483647.0) return fail(DFLASH_ERR_UNSUPPORTED, "block_conv: too large");
  DeviceInfo dev;
  dflash_status s = device_info(&dev);
  if (s) return s;
  return launch_block_conv(h, batch, block_size, d_model, kernel, w, bias, residual, out,
                           static_cast<cudaStream_t>(stream));
}

size_t dflash_draft_topm_workspace_size(int batch, int rows_per_seq, int vocab, int m) {
  if (batch < 1 || rows_per_seq < 1 || vocab < 1 || m < 1) return 0;
  return topm_ws_bytes(batch, rows_per_seq, vocab, m);
}

dflash_status dflash_draft_topm(const void* logits, int batch, int rows_per_seq, int vocab, int m, float temperature,
                                float lambda, int32_t* idx_out, float* logp_out, float* entropy_out,
                                float* path_score_out, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || rows_per_seq < 1 || rows_per_seq > 16 || vocab < 1 || m < 1)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "need batch >= 0, 1 <= rows_per_seq <= 16, vocab >= 1, m >= 1");
  if (m > topm_max_m() || m > vocab) return fail(DFLASH_ERR_UNSUPPORTED, "draft_topm: m <= 8 and m <= vocab");
  if (!(temperature > 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "draft_topm: temperature must be > 0");
  if (batch == 0) return DFLASH_OK;
  if (vocab % 8 || vocab > 32 * 16384)
    return fail(DFLASH_ERR_UNSUPPORTED, "draft_topm needs vocab % 8 == 0 and vocab <= 524288");
  if (double(batch) * rows_per_seq * ((vocab + 16383) / 16384) >= 2147483647.0)
    return fail(DFLASH_ERR_UNSUPPORTED, "draft_topm: too many rows");
  if (!logits || !idx_out || !logp_out || !entropy_out || !path_score_out)
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL logits or output");
  if (!aligned16(logits)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "logits must be 16-byte aligned");
  dflash_status s = check_ws(workspace, workspace_bytes, topm_ws_bytes(batch, rows_per_seq, vocab, m));
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_draft_topm(logits, batch, rows_per_seq, vocab, m, temperature, lambda, idx_out, logp_out,
                           entropy_out, path_score_out, workspace, static_cast<cudaStream_t>(stream));
}

// --------------------------------------------------------- fuse context ----

size_t dflash_fuse_context_workspace_size(int total_new, int num_taps, int d_target, int d_model,
                                          int num_layers, int num_kv_heads, dflash_dtype dtype) {
  if (total_new < 0 || num_taps < 1 || d_target < 1 || d_model < 1 || num_layers < 1 || num_kv_heads < 1)
    return 0;
  return fuse_ws_bytes(total_new, num_taps, d_target, d_model, num_layers, num_kv_heads, dtype);
}

dflash_status dflash_fuse_context(int num_taps, const void* const* taps, int d_target,
                                  const int32_t* cu_new, int batch, int total_new,
                                  const void* w_fuse, const void* g_fuse, int d_model,
                                  const void* w_kv, const void* k_gain, float rope_theta, float eps,
                                  const dflash_kv_cache* cache, void* h_t_out, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  dflash_status s = check_cache(cache);
  if (s) return s;
  if (num_taps < 1 || num_taps > 8) return fail(DFLASH_ERR_UNSUPPORTED, "num_taps must be 1..8");
  if (!taps) return fail(DFLASH_ERR_INVALID_ARGUMENT, "taps is NULL");
  if (batch != cache->batch) return fail(DFLASH_ERR_INVALID_ARGUMENT, "batch must equal cache->batch");
  if (total_new < 0) return fail(DFLASH_ERR_INVALID_ARGUMENT, "total_new < 0");
  if (total_new > 0 && total_new > cache->capacity * batch)
    return fail(DFLASH_ERR_CAPACITY, "total_new exceeds batch * capacity");
  if (total_new == 0) return DFLASH_OK;
  if (!cu_new || !w_fuse || !w_kv) return fail(DFLASH_ERR_INVALID_ARGUMENT, "NULL cu_new / w_fuse / w_kv");
  for (int j = 0; j < num_taps; ++j) {
    if (!taps[j]) return fail(DFLASH_ERR_INVALID_ARGUMENT, "taps[" + std::to_string(j) + "] is NULL");
    if (!aligned16(taps[j])) return fail(DFLASH_ERR_INVALID_ARGUMENT, "taps must be 16-byte aligned");
  }
  if (!aligned16(w_fuse) || !aligned16(w_kv) || (h_t_out && !aligned16(h_t_out)))
    return fail(DFLASH_ERR_INVALID_ARGUMENT, "weights and h_t_out must be 16-byte aligned");
  if (cache->dtype == DFLASH_BF16) {
    if (d_target % 64 || d_model % 256)
      return fail(DFLASH_ERR_UNSUPPORTED, "bf16 fusion needs d_target % 64 == 0 and d_model % 256 == 0");
  } else {
    if (d_target % 4 || d_model % 4) return fail(DFLASH_ERR_UNSUPPORTED, "fp32 fusion needs widths % 4 == 0");
  }
  if (!(rope_theta > 1.0f) || !(eps >= 0.0f)) return fail(DFLASH_ERR_INVALID_ARGUMENT, "rope_theta > 1, eps >= 0");
  const size_t need = fuse_ws_bytes(total_new, num_taps, d_target, d_model, cache->num_layers,
                                    cache->num_kv_heads, cache->dtype);
  s = check_ws(workspace, workspace_bytes, need);
  if (s) return s;
  DeviceInfo dev;
  s = device_info(&dev);
  if (s) return s;
  return launch_fuse_context(num_taps, taps, d_target, cu_new, batch, total_new, w_fuse, g_fuse,
                             d_model, w_kv, k_gain, rope_theta, eps, *cache, h_t_out, workspace,
                             static_cast<cudaStream_t>(stream), dev);
}

}  // extern "C"
