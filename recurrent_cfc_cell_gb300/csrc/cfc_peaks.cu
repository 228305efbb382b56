// cfc_peaks.cu -- two throughput probes that measure the denominators of the CUDA-core
// rooflines on the device they run on: the fp32 FMA rate and the L2 read bandwidth.  They are
// timed by the caller (CUDA events around the call) and compute nothing of the cell.
#include "cfc.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kFmaThreads = 256;
constexpr int kFmaChains = 8;  // independent packed-FMA chains per thread (covers the latency)

// Each thread runs kFmaChains chains of `iters` packed fp32 FMAs (two lanes each); every chain
// depends on the thread's inputs, so nothing folds away, and one sum per thread is stored.
__global__ void __launch_bounds__(kFmaThreads) fma_probe_kernel(float* out, int iters, float a,
                                                                float b) {
  float2 acc[kFmaChains];
  const float x = static_cast<float>(threadIdx.x) * 1e-7f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) acc[c] = make_float2(x + c, x - c);
  const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) acc[c] = fma2(acc[c], a2, b2);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) s += acc[c].x + acc[c].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Reads `n` float4s `passes` times (grid-stride, 16-byte loads through L2 only) and stores one
// sum per thread.  With the buffer smaller than L2, after the first pass this is L2 bandwidth.
__global__ void __launch_bounds__(256) l2_probe_kernel(const float4* __restrict__ buf, size_t n,
                                                        int passes, float* out) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (int p = 0; p < passes; ++p) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
      const float4 v = __ldcg(buf + i);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y + acc.z + acc.w;
}

}  // namespace
}  // namespace cfc

extern "C" {

int cfc_probe_fma(float* out, int blocks, int iters, double* flop, cfc_stream_t stream) {
  if (!out || !flop) return CFC_ERR_NULL_PTR;
  if (blocks <= 0 || iters <= 0) return CFC_ERR_INVALID_DIM;
  cfc::LaunchCfg c;
  c.grid = dim3(static_cast<unsigned>(blocks), 1, 1);
  c.block = dim3(cfc::kFmaThreads, 1, 1);
  c.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cfc::launch(c, cfc::fma_probe_kernel, out, iters, 0.999999f, 1e-6f);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_LAUNCH_FAILED;
  }
  // two lanes x (multiply + add) per packed FMA
  *flop = 4.0 * blocks * cfc::kFmaThreads * static_cast<double>(iters) * cfc::kFmaChains;
  return CFC_OK;
}

int cfc_probe_l2_read(const float* buf, size_t n_floats, int passes, float* out, int blocks,
                      double* bytes, cfc_stream_t stream) {
  if (!buf || !out || !bytes) return CFC_ERR_NULL_PTR;
  if (n_floats < 4 || passes <= 0 || blocks <= 0) return CFC_ERR_INVALID_DIM;
  if (reinterpret_cast<uintptr_t>(buf) & 15u) return CFC_ERR_MISALIGNED;
  cfc::LaunchCfg c;
  c.grid = dim3(static_cast<unsigned>(blocks), 1, 1);
  c.block = dim3(256, 1, 1);
  c.stream = static_cast<cudaStream_t>(stream);
  const size_t n = n_floats / 4;
  const cudaError_t e = cfc::launch(c, cfc::l2_probe_kernel, reinterpret_cast<const float4*>(buf),
                                    n, passes, out);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return CFC_ERR_LAUNCH_FAILED;
  }
  *bytes = 16.0 * static_cast<double>(n) * passes;
  return CFC_OK;
}

}  // extern "C"
