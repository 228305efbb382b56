// cfc_decay.cu -- the pages' own leaky (tau-decay) cell on the CUDA cores: the input
// projection, the forward recurrence over K steps and the reverse-time BPTT with dtau.
//
// Page "K-loop Parallelization -- Block-per-Batch Kernel Refactor" names the backward kernel's
// gradients grad_w_in, grad_w_rec, grad_b and grad_tau (section "Per-Kernel Breakdown") and a
// per-block decay vector sdecay[n_hid] (section "Large shared-mem note"), without equations.
// The cell computed here (a reading of those names):
//
//     a_t = W [x_t ; h_{t-1}] + b,   e_t = tanh(a_t),   d_t = exp(-ts[t,b] / tau),
//     h_t = d_t h_{t-1} + (1 - d_t) e_t
//
// and its exact gradients.  One pre-activation per hidden unit (instead of four gates), so each
// step is one [C x C] mat-vec per batch row.  The weight and input gradients are dense sums over
// the B*K rows and run afterwards on the tensor-core contraction (cfc_contract.cu), as for the
// four-gate cell; this file holds the recurrences.
//
// Layout of a recurrence CTA (CP = C rounded up to 32, at most 128; 2 CP threads; R batch rows):
// thread 2 i + hf owns hidden unit i and half hf of the mat-vec's reduction: in the forward, the
// row W_rec[i][hf CP/2 ..] in registers; in the BPTT, the column W_rec[hf CP/2 .. ][i] (for
// W_rec^T da).  The vector of the step (h_{t-1}, or da_t) sits in shared memory, double
// buffered, so each step needs one CTA barrier.  The pair's partial sums meet by one shuffle.
// Per-row inputs of the next step are loaded one step ahead.  The rows of a CTA run in phases
// (all mat-vecs, then all updates) so their latency chains overlap.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kProjRows = 8;  // rows per projection CTA (one warp each)

// X[r][c] = b[c] + sum_k x[r][k] W[c][k] (k < n_x) for the B*K rows r, written into E (the
// recurrence reads X there and overwrites it with tanh(a)).  W_in^T is staged through shared
// memory 32 inputs at a time; lane l of warp w computes channels l, l + 32, ... of row w.
__global__ void __launch_bounds__(256) decay_proj_kernel(const float* __restrict__ x,
                                                         const float* __restrict__ W,
                                                         const float* __restrict__ bias, int BK,
                                                         int C, int n_x, float* __restrict__ E) {
  __shared__ float wt[32][129];          // [k][c] chunk of W_in^T
  __shared__ float xs[kProjRows][32];    // [row][k] chunk of x
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kProjRows + warp;
  const int n_in = n_x + C;
  float acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    acc[j] = c < C ? __ldg(bias + c) : 0.f;
  }
  for (int k0 = 0; k0 < n_x; k0 += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * 128; e += 256) {
      const int c = e >> 5, k = e & 31;
      wt[k][c] = (c < C && k0 + k < n_x) ? __ldg(W + static_cast<size_t>(c) * n_in + k0 + k) : 0.f;
    }
    xs[warp][lane] = (r < BK && k0 + lane < n_x) ? __ldg(x + static_cast<size_t>(r) * n_x + k0 + lane) : 0.f;
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float xv = xs[warp][k];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(wt[k][lane + 32 * j], xv, acc[j]);
    }
  }
  if (r < BK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = lane + 32 * j;
      if (c < C) E[static_cast<size_t>(r) * C + c] = acc[j];
    }
  }
}

struct DecayFwdParams {
  const float* h0;     // [B][C]
  const float* W;      // [C][n_x + C]
  const float* tau;    // [C]
  const float* ts;     // [K][B]
  float* H;            // [K][B][C]  OUTPUT
  float* E;            // [K][B][C]  in: X = W_in x + b;  OUTPUT: tanh(a)
  int B, K, C, n_x;
};

// Forward recurrence, one CTA per R batch rows, all K steps.
template <int CP, int R>
__global__ void __launch_bounds__(2 * CP) decay_fwd_kernel(const DecayFwdParams p) {
  constexpr int HALF = CP / 2;
  __shared__ __align__(16) float hs[2][R][CP];  // h_{t-1} of the rows, double buffered
  const int tid = threadIdx.x, i = tid >> 1, hf = tid & 1;
  const int B = p.B, K = p.K, C = p.C, n_in = p.n_x + C;
  const int row0 = blockIdx.x * R;
  const bool ok_i = i < C;
  // W_rec[i][HALF hf + j], paired for the packed FMA.
  float2 w[HALF / 2];
#pragma unroll
  for (int j = 0; j < HALF / 2; ++j) {
    const int c0 = HALF * hf + 2 * j;
    const float* wr = p.W + static_cast<size_t>(ok_i ? i : 0) * n_in + p.n_x;
    w[j] = make_float2(ok_i && c0 < C ? __ldg(wr + c0) : 0.f,
                       ok_i && c0 + 1 < C ? __ldg(wr + c0 + 1) : 0.f);
  }
  const float inv_tau = ok_i ? 1.f / __ldg(p.tau + i) : 0.f;
  bool rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rok[r] = row0 + r < B;
    // The pair's first lane writes each slot once (zero where no channel or row lives).
    if (hf == 0)
      hs[0][r][i] = (ok_i && rok[r]) ? __ldg(p.h0 + static_cast<size_t>(row0 + r) * C + i) : 0.f;
  }
  float xn[R], tn[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const size_t o = static_cast<size_t>(row0 + r) * C + i;
    xn[r] = (ok_i && rok[r]) ? __ldcg(p.E + o) : 0.f;
    tn[r] = rok[r] ? __ldg(p.ts + row0 + r) : 0.f;
  }
  __syncthreads();
  for (int t = 0; t < K; ++t) {
    const int cur = t & 1;
    float xc[R], tc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xc[r] = xn[r];
      tc[r] = tn[r];
    }
    if (t + 1 < K) {  // the next step's X and ts, one step ahead
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const size_t tb = static_cast<size_t>(t + 1) * B + row0 + r;
        xn[r] = (ok_i && rok[r]) ? __ldcg(p.E + tb * C + i) : 0.f;
        tn[r] = rok[r] ? __ldg(p.ts + tb) : 0.f;
      }
    }
    float a[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4* hv = reinterpret_cast<const float4*>(&hs[cur][r][HALF * hf]);
      float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < HALF / 4; ++q) {
        const float4 v = hv[q];
        s0 = fma2(w[2 * q], make_float2(v.x, v.y), s0);
        s1 = fma2(w[2 * q + 1], make_float2(v.z, v.w), s1);
      }
      a[r] = (s0.x + s0.y) + (s1.x + s1.y);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float at = a[r] + __shfl_xor_sync(0xffffffffu, a[r], 1) + xc[r];
      const float e = tanhf(at);
      const float d = __expf(-tc[r] * inv_tau);
      const float hp = hs[cur][r][ok_i ? i : 0];
      const float h = d * hp + (1.f - d) * e;
      if (hf == 0) {
        hs[cur ^ 1][r][i] = ok_i ? h : 0.f;
        if (ok_i && rok[r]) {
          const size_t o = (static_cast<size_t>(t) * B + row0 + r) * C + i;
          p.H[o] = h;
          p.E[o] = e;
        }
      }
    }
    __syncthreads();
  }
}

struct DecayBwdParams {
  const float* dH;     // [K][B][C]
  const float* h0;     // [B][C]
  const float* W;      // [C][n_x + C]
  const float* tau;    // [C]
  const float* ts;     // [K][B]
  const float* H;      // [K][B][C]
  const float* E;      // [K][B][C]  tanh(a)
  __nv_bfloat16* da;   // OUTPUT: operand rows of da, 2 mp bf16 per (t, b) row (hi, then lo)
  float* dh0;          // OUTPUT [B][C]
  float* dtau_part;    // OUTPUT [B][C]: dtau summed over the steps of each row
  int B, K, C, n_x, mp;
};

// BPTT, one CTA per R batch rows, steps K-1 .. 0.  With G the gradient reaching h_t:
//   da = G (1 - d) (1 - e^2),  dtau_row += G (h_{t-1} - e) d ts / tau^2,
//   G_{t-1} = dH[t-1] + G d + W_rec^T da.
template <int CP, int R>
__global__ void __launch_bounds__(2 * CP) decay_bwd_kernel(const DecayBwdParams p) {
  constexpr int HALF = CP / 2;
  __shared__ __align__(16) float das[2][R][CP];  // da of the step, double buffered
  const int tid = threadIdx.x, j = tid >> 1, hf = tid & 1;
  const int B = p.B, K = p.K, C = p.C, n_in = p.n_x + C;
  const int row0 = blockIdx.x * R;
  const bool ok_j = j < C;
  // Column j of W_rec over the rows i = HALF hf + 2 q (+1), paired for the packed FMA.
  float2 wc[HALF / 2];
#pragma unroll
  for (int q = 0; q < HALF / 2; ++q) {
    const int i0 = HALF * hf + 2 * q;
    const float* col = p.W + p.n_x + (ok_j ? j : 0);
    wc[q] = make_float2(ok_j && i0 < C ? __ldg(col + static_cast<size_t>(i0) * n_in) : 0.f,
                        ok_j && i0 + 1 < C ? __ldg(col + static_cast<size_t>(i0 + 1) * n_in) : 0.f);
  }
  const float inv_tau = ok_j ? 1.f / __ldg(p.tau + j) : 0.f;
  bool rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rok[r] = row0 + r < B;
  // Inputs of step t for the rows: dH, e = tanh(a), h_{t-1}, ts.
  auto load = [&](int t, float (&dh)[R], float (&e)[R], float (&hp)[R], float (&tv)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool v = ok_j && rok[r];
      const size_t tb = static_cast<size_t>(t) * B + row0 + r;
      dh[r] = v ? __ldcg(p.dH + tb * C + j) : 0.f;
      e[r] = v ? __ldcg(p.E + tb * C + j) : 0.f;
      hp[r] = !v ? 0.f
            : t > 0 ? __ldcg(p.H + (tb - B) * C + j)
                    : __ldg(p.h0 + static_cast<size_t>(row0 + r) * C + j);
      tv[r] = rok[r] ? __ldg(p.ts + tb) : 0.f;
    }
  };
  float G[R], acc[R], dHn[R], en[R], hpn[R], tsn[R];
#pragma unroll
  for (int r = 0; r < R; ++r) G[r] = acc[r] = 0.f;
  load(K - 1, dHn, en, hpn, tsn);
  for (int t = K - 1; t >= 0; --t) {
    const int cur = t & 1;
    float dHc[R], ec[R], hpc[R], tsc[R], dv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      dHc[r] = dHn[r]; ec[r] = en[r]; hpc[r] = hpn[r]; tsc[r] = tsn[r];
    }
    if (t >= 1) load(t - 1, dHn, en, hpn, tsn);  // one step ahead
#pragma unroll
    for (int r = 0; r < R; ++r) {
      G[r] += dHc[r];
      const float d = __expf(-tsc[r] * inv_tau);
      dv[r] = d;
      const float da = G[r] * (1.f - d) * (1.f - ec[r] * ec[r]);
      acc[r] += G[r] * (hpc[r] - ec[r]) * d * tsc[r] * inv_tau * inv_tau;
      if (hf == 0) {
        das[cur][r][j] = ok_j ? da : 0.f;
        if (ok_j && rok[r]) {
          __nv_bfloat16* q = p.da + (static_cast<size_t>(t) * B + row0 + r) * 2 * p.mp + j;
          const __nv_bfloat16 hi = __float2bfloat16_rn(da);
          q[0] = hi;
          q[p.mp] = __float2bfloat16_rn(da - __bfloat162float(hi));
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4* dv4 = reinterpret_cast<const float4*>(&das[cur][r][HALF * hf]);
      float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < HALF / 4; ++q) {
        const float4 v = dv4[q];
        s0 = fma2(wc[2 * q], make_float2(v.x, v.y), s0);
        s1 = fma2(wc[2 * q + 1], make_float2(v.z, v.w), s1);
      }
      const float part = (s0.x + s0.y) + (s1.x + s1.y);
      const float delta = part + __shfl_xor_sync(0xffffffffu, part, 1);
      G[r] = G[r] * dv[r] + delta;
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (hf == 0 && ok_j && rok[r]) {
      const size_t o = static_cast<size_t>(row0 + r) * C + j;
      p.dh0[o] = G[r];
      p.dtau_part[o] = acc[r];
    }
}

// Rows per CTA: as few as keep the CTAs within about two waves of 148 SMs.
int decay_rows(int B) { return B <= 296 ? 1 : (B <= 592 ? 2 : 4); }

template <int CP, int R>
cudaError_t fwd_k(const DecayFwdParams& p, cudaStream_t s) {
  LaunchCfg c;
  c.grid = dim3((p.B + R - 1) / R, 1, 1);
  c.block = dim3(2 * CP, 1, 1);
  c.stream = s;
  return launch(c, decay_fwd_kernel<CP, R>, p);
}

template <int CP, int R>
cudaError_t bwd_k(const DecayBwdParams& p, cudaStream_t s) {
  LaunchCfg c;
  c.grid = dim3((p.B + R - 1) / R, 1, 1);
  c.block = dim3(2 * CP, 1, 1);
  c.stream = s;
  return launch(c, decay_bwd_kernel<CP, R>, p);
}

template <int CP>
cudaError_t fwd_cp(const DecayFwdParams& p, int R, cudaStream_t s) {
  return R == 1 ? fwd_k<CP, 1>(p, s) : R == 2 ? fwd_k<CP, 2>(p, s) : fwd_k<CP, 4>(p, s);
}
template <int CP>
cudaError_t bwd_cp(const DecayBwdParams& p, int R, cudaStream_t s) {
  return R == 1 ? bwd_k<CP, 1>(p, s) : R == 2 ? bwd_k<CP, 2>(p, s) : bwd_k<CP, 4>(p, s);
}

}  // namespace

bool decay_supported(int C, int n_x) { return C >= 1 && C <= kDecayMaxC && n_x >= 1; }

cudaError_t decay_proj_launch(const float* x, const float* W, const float* b, int BK, int C,
                              int n_x, float* E, cudaStream_t s) {
  if (C > kDecayMaxC) return cudaErrorInvalidValue;
  LaunchCfg c;
  c.grid = dim3((BK + kProjRows - 1) / kProjRows, 1, 1);
  c.block = dim3(32 * kProjRows, 1, 1);
  c.stream = s;
  return launch(c, decay_proj_kernel, x, W, b, BK, C, n_x, E);
}

cudaError_t decay_fwd_launch(const float* h0, const float* W, const float* tau, const float* ts,
                             int B, int K, int C, int n_x, float* H, float* E, cudaStream_t s) {
  DecayFwdParams p{h0, W, tau, ts, H, E, B, K, C, n_x};
  const int R = decay_rows(B);
  if (C <= 32) return fwd_cp<32>(p, R, s);
  if (C <= 64) return fwd_cp<64>(p, R, s);
  if (C <= 128) return fwd_cp<128>(p, R, s);
  return cudaErrorInvalidValue;
}

cudaError_t decay_bwd_launch(const float* dH, const float* h0, const float* W, const float* tau,
                             const float* ts, const float* H, const float* E, int B, int K,
                             int C, int n_x, void* da_rows, int mp, float* dh0, float* dtau_part,
                             cudaStream_t s) {
  DecayBwdParams p{dH, h0, W, tau, ts, H, E, static_cast<__nv_bfloat16*>(da_rows), dh0,
                   dtau_part, B, K, C, n_x, mp};
  const int R = decay_rows(B);
  if (C <= 32) return bwd_cp<32>(p, R, s);
  if (C <= 64) return bwd_cp<64>(p, R, s);
  if (C <= 128) return bwd_cp<128>(p, R, s);
  return cudaErrorInvalidValue;
}

}  // namespace cfc
