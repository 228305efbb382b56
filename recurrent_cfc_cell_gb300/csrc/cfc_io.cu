// cfc_io.cu -- a copy done by the SMs instead of a copy engine, for moving a training step's
// inputs in from pinned host memory and its gradients back out.  Those buffers are a few MB; on
// GB300 the CPU's memory is reached over the chip-to-chip link, and many CTAs with several
// 16-byte loads in flight each move such a buffer in less time than one copy-engine transfer
// takes to get going.  Either side may be device memory or host memory that is mapped into the
// device's address space (pinned or registered).
#include <cstdint>

#include "cfc.h"
#include "cfc_launch.cuh"

namespace cfc {
namespace {

constexpr int kCopyThreads = 256;
// One 16-byte load per thread and pass, on as many CTAs as the buffer fills: for a step's
// few MB the link's round trip, not the issue rate, sets the time, so the widest grid wins
// (on GB300 the end-to-end step with 1 load per thread ran 0.7% faster than with 4, and 1.5%
// faster than with 8).
constexpr int kCopyUnroll = 1;
constexpr int kCopyMaxBlocks = 152 * 8;

// dst[i] = src[i] for i < n (16-byte words), grid-stride: each thread issues kCopyUnroll loads,
// then the stores.
__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(const uint4* __restrict__ src,
                                                              uint4* __restrict__ dst, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < n; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

// The device address of `p`, or nullptr when the device cannot reach it (pageable host memory
// that was never registered, or memory of no known kind).
const void* device_view(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return a.devicePointer;
    default:
      return nullptr;
  }
}

}  // namespace
}  // namespace cfc

extern "C" {

int cfc_copy(const void* src, void* dst, size_t bytes, cfc_stream_t stream) {
  if (!src || !dst) return CFC_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u) ||
      (bytes & 15u))
    return CFC_ERR_MISALIGNED;
  if (bytes == 0) return CFC_OK;
  const void* s = cfc::device_view(src);
  void* d = const_cast<void*>(cfc::device_view(dst));
  if (!s || !d) return CFC_ERR_INVALID_ARG;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(s), d0 = reinterpret_cast<uintptr_t>(d);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return CFC_ERR_INVALID_ARG;  // overlapping ranges
  const size_t n = bytes / 16;
  const size_t per_block = static_cast<size_t>(cfc::kCopyThreads) * cfc::kCopyUnroll;
  size_t blocks = (n + per_block - 1) / per_block;
  if (blocks > static_cast<size_t>(cfc::kCopyMaxBlocks)) blocks = cfc::kCopyMaxBlocks;
  cfc::LaunchCfg c;
  c.grid = dim3(static_cast<unsigned>(blocks), 1, 1);
  c.block = dim3(cfc::kCopyThreads, 1, 1);
  c.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cfc::launch(c, cfc::copy16_kernel, static_cast<const uint4*>(s),
                                    static_cast<uint4*>(d), n);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_LAUNCH_FAILED;
  }
  return CFC_OK;
}

}  // extern "C"
