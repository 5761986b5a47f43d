// splitkv_noalloc.cu - split-KV attention forward for callers that must not
// allocate device memory.
//
// osattn_fwd_splitkv needs a workspace for its per-range partial results,
// and its caller has to obtain that memory (usually with cudaMalloc).  Some
// callers cannot: code embedded in an application whose memory manager owns
// the whole device budget and forbids allocations behind its back, and code
// on a latency-critical path where cudaMalloc's implicit synchronisation and
// unpredictable cost are not acceptable.  This file gives them one entry
// point whose workspace is a fixed array compiled into the library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its 32 MiB until the process exits.  In host code its name
// is only a host-side stand-in; the device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "osattn.h"
#include "osattn_internal.h"

namespace {

constexpr size_t kScratchBytes = OSATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_splitkv_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (looked up on
// the first call for the device, in the runtime's primary context; a device
// reset makes a new context whose copy may sit elsewhere, which the cache
// does not notice).  Returns OSATTN_OK or OSATTN_ERR_CUDA.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OSATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || !ptr)
      return OSATTN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return OSATTN_OK;
}

}  // namespace

extern "C" int osattn_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O,
                                          float* LSE, int B, int H, int Nq, int Nkv, int d,
                                          float scale, int causal, const int32_t* key_len,
                                          int dtype, int num_splits, void* stream) {
  // The arguments first (the same checks and statuses as
  // osattn_fwd_splitkv), then whether the partials of every (split, row)
  // fit the array.
  int rc = osattn::validate_splitkv(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, key_len, dtype,
                                    num_splits);
  if (rc != OSATTN_OK) return rc;
  const size_t need = osattn_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (need > kScratchBytes) return OSATTN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != OSATTN_OK) return rc;
  // Nothing in the scratch has to start at zero: the split kernel writes
  // every partial that the combine reads, in every call.
  return osattn_fwd_splitkv(Q, K, V, O, LSE, B, H, Nq, Nkv, d, scale, causal, key_len, dtype,
                            num_splits, scratch, kScratchBytes, stream);
}
