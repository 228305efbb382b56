// cfc_inproj.cu -- input projection of the forward pass, hoisted out of the recurrence:
//
//   X[t][b][g][i] = sum_{k < n_x} W[g][i][k] u[t][b][k] + b[g][i]      for every t at once.
//
// It does not depend on h, so it is one parallel contraction over all B*K rows instead of a
// term on the serial K-loop.  The 4C values of a row are written into the forward's own
// outputs -- gate ff1 into H[t][b][:], gates ff2 / ta / tb into cache[t][b][0..2][:] -- which
// have exactly that size; the recurrence reads each value (before the step that needs it)
// and overwrites it with h, ff1, ff2, gate.  No extra memory is needed.
//
// CUDA-core fp32: a 64 x 64 output tile per CTA (256 threads, 4 rows x 4 consecutive gate
// rows each), k in chunks of 64 through shared memory.  A chunk's global loads are all issued
// before any is stored (one memory round trip per chunk; n_x <= 64 is one chunk), and each
// thread writes its four consecutive outputs of a row as one 16-byte store when C % 4 == 0.
#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kTR = 64, kTM = 64, kTK = 64;
constexpr int kLoads = kTK * kTR / 256;  // elements of each operand tile per thread

__global__ void __launch_bounds__(256) inproj_kernel(const float* __restrict__ u,
                                                      const float* __restrict__ W,
                                                      const float* __restrict__ bias, int BK,
                                                      int C, int n_x, float* __restrict__ H,
                                                      float* __restrict__ cache) {
  __shared__ __align__(16) float Us[kTK][kTR + 4];  // [k][row]
  __shared__ __align__(16) float Ws[kTK][kTM + 4];  // [k][m]
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int M = 4 * C, n_in = n_x + C;
  const int r0 = blockIdx.y * kTR, m0 = blockIdx.x * kTM;
  const int tid = threadIdx.x;
  const int tr = tid >> 4, tm = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < n_x; k0 += kTK) {
    // Element e of a tile: row e / kTK, column e % kTK (consecutive threads walk k).
    float ur[kLoads], wr[kLoads];
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int e = tid + q * 256;
      const int rr = e / kTK, kk = e % kTK;
      const int r = r0 + rr, m = m0 + rr, k = k0 + kk;
      ur[q] = (r < BK && k < n_x) ? __ldg(u + static_cast<size_t>(r) * n_x + k) : 0.f;
      wr[q] = (m < M && k < n_x) ? __ldg(W + static_cast<size_t>(m) * n_in + k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int e = tid + q * 256;
      Us[e % kTK][e / kTK] = ur[q];
      Ws[e % kTK][e / kTK] = wr[q];
    }
    __syncthreads();
    const int kn = min(kTK, n_x - k0);
    for (int kk = 0; kk < kn; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&Us[kk][tr * 4]);
      const float4 w = *reinterpret_cast<const float4*>(&Ws[kk][tm * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
  // Outputs m .. m + 3 of rows r: gate g = m / C goes to H (g = 0) or cache[.][g - 1].
  const int mq = m0 + tm * 4;
  if (mq >= M) return;
  if ((C & 3) == 0) {  // the four outputs share a gate and a 16-byte aligned slot
    const int g = mq / C, ch = mq - g * C;
    const float4 bm = *reinterpret_cast<const float4*>(bias + mq);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + tr * 4 + i;
      if (r >= BK) continue;
      const float4 v = make_float4(acc[i][0] + bm.x, acc[i][1] + bm.y, acc[i][2] + bm.z,
                                   acc[i][3] + bm.w);
      float* dst = (g == 0) ? H + static_cast<size_t>(r) * C + ch
                            : cache + (static_cast<size_t>(r) * 3 + (g - 1)) * C + ch;
      *reinterpret_cast<float4*>(dst) = v;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int m = mq + j;
    if (m >= M) continue;
    const int g = m / C, ch = m - g * C;
    const float bm = bias[m];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + tr * 4 + i;
      if (r >= BK) continue;
      const float v = acc[i][j] + bm;
      if (g == 0) H[static_cast<size_t>(r) * C + ch] = v;
      else cache[(static_cast<size_t>(r) * 3 + (g - 1)) * C + ch] = v;
    }
  }
}

}  // namespace

cudaError_t inproj_launch(const float* u, const float* W, const float* bias, int BK, int C,
                          int n_x, float* H, float* cache, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3((4 * C + kTM - 1) / kTM, (BK + kTR - 1) / kTR, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return launch(c, inproj_kernel, u, W, bias, BK, C, n_x, H, cache);
}

}  // namespace cfc
