// dflash_verify_noalloc: speculative verification without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they verify:
// code running inside a CUDA graph that is being captured (cudaMalloc is not
// a stream operation and breaks the capture), allocators that forbid
// allocation after start-up, or plain C hosts with no allocator of their own.
// For them this entry point takes its scratch from a file-scope device array
// that the library reserves when it is loaded; every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  The verification kernels write every scratch entry before
// they read it, so nothing needs clearing between calls.  Calls that overlap
// on the GPU (different streams, no ordering between them) race on the array:
// order them on one stream, or use dflash_verify with separate workspaces.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "dflash_internal.h"

namespace dflash {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// `g_noalloc_scratch` names a host-side stand-in, not device memory, so the
// address is looked up once per device with that device current.
dflash_status scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" {

size_t dflash_verify_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

dflash_status dflash_verify_noalloc(const void* target_logits, const void* draft_logits, dflash_dtype dtype,
                                    const int32_t* draft_tokens, int batch, int block_size, int vocab,
                                    float temperature, uint64_t seed, uint64_t cycle, int32_t* accepted_len,
                                    int32_t* out_tokens, void* stream) {
  if (batch > 0 && block_size >= 1 && vocab >= 1) {
    const size_t need = verify_ws_bytes(batch, block_size, vocab);
    if (need > kNoAllocScratchBytes)
      return fail(DFLASH_ERR_UNSUPPORTED,
                  "dflash_verify_noalloc: batch/block_size/vocab need " + std::to_string(need) +
                      " bytes of scratch, more than the " + std::to_string(kNoAllocScratchBytes) +
                      " bytes it reserves; use dflash_verify with a workspace");
  }
  DeviceInfo dev;
  dflash_status s = device_info(&dev);
  if (s) return s;
  void* scratch = nullptr;
  s = scratch_address(dev.device, &scratch);
  if (s) return s;
  return dflash_verify(target_logits, draft_logits, dtype, draft_tokens, batch, block_size, vocab, temperature,
                       seed, cycle, accepted_len, out_tokens, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
