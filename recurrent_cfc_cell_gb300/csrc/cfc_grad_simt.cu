// cfc_grad_simt.cu -- CUDA-core fp32 contractions after the BPTT recurrence:
//
//   dW[m][n] = sum_{r<BK} d_pre[r][m] * z[r][n]      (m < 4C, n < n_in, r = t*B + b)
//   du[r][k] = sum_{m<4C} d_pre[r][m] * W[m][k]       (k < n_x)
//
// The weight gradient is the batch-and-time sum that the DQN plan (page "H100 Epoch
// Optimization Phase 2", Task 2) turns into one GEMM "dW = dY^T X" instead of per-sample
// atomic accumulation; here it is split over the reduction (B*K rows) into S partial tiles
// whose deterministic sum is taken by reduce_axis0.  z is never materialised: row r of z is
// [u[t][b] ; h_{t-1}[b]] with h_{-1} = h0, read straight from u, H and h0.
//
// These kernels are the fp32 reference path (exact fp32 FMA, no operand rounding); the
// tensor-core contraction is the fast path.
#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;

__device__ __forceinline__ float z_at(const float* __restrict__ u, const float* __restrict__ H,
                                      const float* __restrict__ h0, int B, int C, int n_x, int r,
                                      int n) {
  if (n < n_x) return u[static_cast<size_t>(r) * n_x + n];
  const int j = n - n_x;
  if (j >= C) return 0.f;
  if (r >= B) return H[static_cast<size_t>(r - B) * C + j];
  return h0[static_cast<size_t>(r) * C + j];  // t = 0: row r is batch row b = r
}

// grid (ceil(n_in/64), ceil(4C/64), S); 256 threads, 4x4 outputs each.
__global__ void __launch_bounds__(256) dw_simt_kernel(const float* __restrict__ d_pre,
                                                       const float* __restrict__ u,
                                                       const float* __restrict__ H,
                                                       const float* __restrict__ h0, int B, int K,
                                                       int C, int n_x, int S,
                                                       float* __restrict__ partial) {
  __shared__ __align__(16) float As[kTK][kTM];
  __shared__ __align__(16) float Zs[kTK][kTN];
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int M = 4 * C, N = n_x + C, BK = B * K;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  const int s = blockIdx.z;
  const int chunk = (BK + S - 1) / S;
  const int r_lo = s * chunk;
  const int r_hi = min(BK, r_lo + chunk);
  const int tid = threadIdx.x;
  const int tm = tid >> 4, tn = tid & 15;
  float acc[4][4] = {};
  for (int r0 = r_lo; r0 < r_hi; r0 += kTK) {
#pragma unroll
    for (int q = 0; q < (kTK * kTM) / 256; ++q) {
      const int e = tid + q * 256;
      const int rr = e / kTM, mm = e % kTM;
      const int r = r0 + rr, m = m0 + mm;
      As[rr][mm] = (r < r_hi && m < M) ? d_pre[static_cast<size_t>(r) * M + m] : 0.f;
      const int n = n0 + mm;
      Zs[rr][mm] = (r < r_hi && n < N) ? z_at(u, H, h0, B, C, n_x, r, n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < kTK; ++rr) {
      const float4 a = *reinterpret_cast<const float4*>(&As[rr][tm * 4]);
      const float4 zz = *reinterpret_cast<const float4*>(&Zs[rr][tn * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float zv[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(av[i], zv[q], acc[i][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tn * 4 + q;
      if (n < N) partial[(static_cast<size_t>(s) * M + m) * N + n] = acc[i][q];
    }
  }
}

// du: grid (ceil(n_x/64), ceil(BK/64)); 256 threads, 4x4 outputs each.
__global__ void __launch_bounds__(256) du_simt_kernel(const float* __restrict__ d_pre,
                                                       const float* __restrict__ W, int BK, int C,
                                                       int n_x, float* __restrict__ du) {
  __shared__ __align__(16) float As[kTK][kTM + 4];  // [m][r]
  __shared__ __align__(16) float Ws[kTK][kTN];      // [m][k]
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int M = 4 * C, n_in = n_x + C;
  const int r0 = blockIdx.y * kTM, k0 = blockIdx.x * kTN;
  const int tid = threadIdx.x;
  const int tr = tid >> 4, tk = tid & 15;
  float acc[4][4] = {};
  for (int mb = 0; mb < M; mb += kTK) {
#pragma unroll
    for (int q = 0; q < (kTK * kTM) / 256; ++q) {
      const int e = tid + q * 256;
      const int rr = e / kTK, mm = e % kTK;  // consecutive threads walk m (coalesced rows)
      const int r = r0 + rr, m = mb + mm;
      As[mm][rr] = (r < BK && m < M) ? d_pre[static_cast<size_t>(r) * M + m] : 0.f;
      const int mw = e / kTN, kk = e % kTN;
      const int m2 = mb + mw, k = k0 + kk;
      Ws[mw][kk] = (m2 < M && k < n_x) ? W[static_cast<size_t>(m2) * n_in + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int mm = 0; mm < kTK; ++mm) {
      const float4 a = *reinterpret_cast<const float4*>(&As[mm][tr * 4]);
      const float4 ww = *reinterpret_cast<const float4*>(&Ws[mm][tk * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float wv[4] = {ww.x, ww.y, ww.z, ww.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(av[i], wv[q], acc[i][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + tr * 4 + i;
    if (r >= BK) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = k0 + tk * 4 + q;
      if (k < n_x) du[static_cast<size_t>(r) * n_x + k] = acc[i][q];
    }
  }
}

}  // namespace

int dw_simt_splits(int BK) {
  int S = (BK + 255) / 256;
  if (S < 1) S = 1;
  if (S > 32) S = 32;
  return S;
}

cudaError_t dw_simt_launch(const float* d_pre, const float* u, const float* H, const float* h0,
                           int B, int K, int C, int n_x, int S, float* partial, cudaStream_t s,
                           bool pdl) {
  const int M = 4 * C, N = n_x + C;
  LaunchCfg c;
  c.grid = dim3((N + kTN - 1) / kTN, (M + kTM - 1) / kTM, S);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return launch(c, dw_simt_kernel, d_pre, u, H, h0, B, K, C, n_x, S, partial);
}

cudaError_t du_simt_launch(const float* d_pre, const float* W, int BK, int C, int n_x,
                           float* du, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3((n_x + kTN - 1) / kTN, (BK + kTM - 1) / kTM, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return launch(c, du_simt_kernel, d_pre, W, BK, C, n_x, du);
}

}  // namespace cfc
