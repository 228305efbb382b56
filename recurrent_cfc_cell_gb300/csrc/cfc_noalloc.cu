// cfc_noalloc.cu -- cfc_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// cfc_backward needs a device workspace (the pre-activation gradients and the split partial
// sums of the two contractions) that the caller allocates.  Some callers cannot do that: a
// plugin or callback hosted by a framework that owns the GPU's memory (the framework's pool
// holds it and the plugin has no allocator of its own), or a program that fixes its device
// memory footprint when it starts and may not grow it afterwards.  This entry point takes the
// same inputs and outputs but uses a workspace that is part of the library itself: a
// file-scope device array, created when the library's device code is loaded on a GPU and kept
// until the process exits.  It allocates nothing at call time.
#include <cstdint>
#include <mutex>

#include "cfc.h"

namespace {

// Every GPU that loads this library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = CFC_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.  In
// host code the array's name is only a host-side stand-in, never a device address.  The
// device is checked first, so a device of another compute capability gets the same
// CFC_ERR_UNSUPPORTED_DEVICE as from cfc_backward.  The address is cached for the life of the
// process: it does not survive cudaDeviceReset.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return CFC_ERR_UNSUPPORTED_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_UNSUPPORTED_DEVICE;
  }
  if (major != 10 || minor != 3) return CFC_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return CFC_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return CFC_OK;
}

}  // namespace

extern "C" int cfc_backward_noalloc(const float* dH, const float* u, const float* h0,
                                    const float* W, const float* ts, const float* H,
                                    const float* cache, int B, int K, int C, int n_x, float* dW,
                                    float* db, float* du, float* dh0, int dw_mode,
                                    cfc_stream_t stream) {
  size_t need = 0;
  int rc = cfc_workspace_bytes(B, K, C, n_x, dw_mode, &need);
  if (rc != CFC_OK) return rc;
  if (need > kNoAllocScratchBytes) return CFC_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  rc = noalloc_scratch(&ws);
  if (rc != CFC_OK) return rc;
  // Every workspace entry the backward pass reads is written earlier in the same call, so
  // nothing in the shared array has to start at zero or be cleared between calls.
  return cfc_backward(dH, u, h0, W, ts, H, cache, B, K, C, n_x, dW, db, du, dh0, ws,
                      kNoAllocScratchBytes, dw_mode, stream);
}
