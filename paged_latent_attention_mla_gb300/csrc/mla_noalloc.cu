// mla_decode_noalloc: the decode for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code hosted by a runtime that owns
// every byte of device memory and forbids allocation once it is serving, plugins
// that get no allocator from their host, and latency-critical paths where an
// allocation's implicit device synchronization is not acceptable.  For them the
// decode's scratch lives in a fixed array that is part of this library's device
// image: every GPU that loads the library holds it until the process exits.
//
// The array's address is looked up once per device (cudaGetSymbolAddress, with
// that device current) on the first call made on it; that first call should come
// before any stream capture.  The cached address belongs to the device context it
// was looked up in: after cudaDeviceReset (or any teardown of the primary
// context) the library must be reloaded before these calls are used again.
// Every call shares the array, so calls that overlap on the GPU race; the array
// keeps the last call's contents.  A call that completes without a device-side
// error writes every slot the reduction reads before reading it, so nothing
// needs clearing; when the kernel reports an error (mla_noalloc_status) the
// output of that call is incomplete and may mix in an earlier call's partials.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/mla.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// device address of the scratch array on the current device (nullptr on error)
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" mla_status_t mla_decode_noalloc(const void* q_latent, const void* q_rope, const void* ckv_cache,
                                           const void* kpe_cache, const int32_t* page_table, const int32_t* seq_lens,
                                           float scale, int window_left, void* out, float* lse, cudaStream_t stream,
                                           int B, int H, int page_size, const mla_config_t* cfg) {
  void* ws = scratch_address();
  if (!ws) return MLA_ERR_CUDA;
  // mla_decode checks the batch's workspace need against the array's size and
  // returns MLA_ERR_WORKSPACE_TOO_SMALL, launching nothing, when it does not fit.
  return mla_decode(q_latent, q_rope, ckv_cache, kpe_cache, page_table, seq_lens, scale, window_left, out, lse, ws,
                    kNoAllocScratchBytes, stream, B, H, page_size, cfg);
}

// The device-side status of the last mla_decode_noalloc on the current device: the
// same read mla_workspace_status does, on the library's own array.
extern "C" mla_status_t mla_noalloc_status(cudaStream_t stream) {
  void* ws = scratch_address();
  if (!ws) return MLA_ERR_CUDA;
  return mla_workspace_status(ws, kNoAllocScratchBytes, stream);
}
