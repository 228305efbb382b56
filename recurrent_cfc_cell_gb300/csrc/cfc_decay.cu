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
// eight lanes serve a quad of four hidden units.  Lane sl of the eight holds, for each of the
// quad's units, the weights of the reduction entries in chunks 8 q + sl (4 entries a chunk):
// in the forward the rows W_rec[unit][..], in the BPTT the columns W_rec[..][unit] (for
// W_rec^T da).  Every vector value a lane loads from shared memory feeds four FMAs (one per
// unit), and the eight lanes of a warp quarter read eight consecutive 16-byte chunks (no bank
// conflicts; the four quads of a warp read the same chunks, a broadcast).  A reduce-scatter of
// three shuffle levels leaves unit (lane >> 1) & 3 of the quad in each lane pair; the even
// lane of the pair writes it.  The vector of the step (h_{t-1}, or da_t) sits in shared
// memory, double buffered, so each step needs one CTA barrier.  Per-row inputs of the next
// step are loaded one step ahead.  The rows of a CTA run in phases (all mat-vecs, then all
// updates) so their latency chains overlap.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

// Projection tiles: 64 rows x 64 hidden units per CTA of 256 threads, each thread 4 rows x 4
// consecutive units, k in chunks of 64 through shared memory.
constexpr int kPR = 64, kPC = 64, kPK = 64;
constexpr int kPLoads = kPK * kPR / 256;  // elements of each operand tile per thread

// X[r][c] = b[c] + sum_{k < n_x} x[r][k] W[c][k] for the B*K rows r, written into E (the
// recurrence reads X there and overwrites it with tanh(a)).  A chunk's global loads (x and W_in
// rows, consecutive threads walking k) are all issued before any is stored.
__global__ void __launch_bounds__(256) decay_proj_kernel(const float* __restrict__ x,
                                                         const float* __restrict__ W,
                                                         const float* __restrict__ bias, int BK,
                                                         int C, int n_x, float* __restrict__ E) {
  __shared__ __align__(16) float xs[kPK][kPR + 4];  // [k][row]
  __shared__ __align__(16) float ws[kPK][kPC + 4];  // [k][unit]
  const int n_in = n_x + C;
  const int r0 = blockIdx.y * kPR, c0 = blockIdx.x * kPC;
  const int tid = threadIdx.x;
  const int tr = tid >> 4, tc = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < n_x; k0 += kPK) {
    float xr[kPLoads], wr[kPLoads];
#pragma unroll
    for (int q = 0; q < kPLoads; ++q) {
      const int e = tid + q * 256;
      const int rr = e / kPK, kk = e % kPK;
      const int r = r0 + rr, c = c0 + rr, k = k0 + kk;
      xr[q] = (r < BK && k < n_x) ? __ldg(x + static_cast<size_t>(r) * n_x + k) : 0.f;
      wr[q] = (c < C && k < n_x) ? __ldg(W + static_cast<size_t>(c) * n_in + k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kPLoads; ++q) {
      const int e = tid + q * 256;
      xs[e % kPK][e / kPK] = xr[q];
      ws[e % kPK][e / kPK] = wr[q];
    }
    __syncthreads();
    const int kn = min(kPK, n_x - k0);
    for (int kk = 0; kk < kn; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][tr * 4]);
      const float4 w = *reinterpret_cast<const float4*>(&ws[kk][tc * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + tc * 4 + j;
    if (c >= C) continue;
    const float bc = __ldg(bias + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + tr * 4 + i;
      if (r < BK) E[static_cast<size_t>(r) * C + c] = acc[i][j] + bc;
    }
  }
}

// Slots of the BPTT's input ring (copies run two steps ahead of their use).
constexpr int kDecayRing = 3;

// Chunks of four reduction entries a lane holds (chunks 8 q + sl, q < kQ) and the reduction
// over the eight lanes of a unit quad: a[u] is the lane's partial sum of unit u; the result,
// the full sum of unit (lane >> 1) & 3, is in both lanes of each pair.
template <int CP>
struct Quad {
  static constexpr int kQ = CP / 32;
};
__device__ __forceinline__ float quad_reduce_scatter(const float (&a)[4], int lane) {
  const bool b2 = lane & 4, b1 = lane & 2;
  const float k0 = b2 ? a[2] : a[0], k1 = b2 ? a[3] : a[1];
  const float s0 = k0 + __shfl_xor_sync(0xffffffffu, b2 ? a[0] : a[2], 4);
  const float s1 = k1 + __shfl_xor_sync(0xffffffffu, b2 ? a[1] : a[3], 4);
  float acc = (b1 ? s1 : s0) + __shfl_xor_sync(0xffffffffu, b1 ? s0 : s1, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  return acc;
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
  constexpr int kQ = Quad<CP>::kQ;
  __shared__ __align__(16) float hs[2][R][CP];  // h_{t-1} of the rows, double buffered
  const int tid = threadIdx.x, lane = tid & 31, sl = lane & 7;
  const int B = p.B, K = p.K, C = p.C, n_in = p.n_x + C;
  const int row0 = blockIdx.x * R;
  const int ubase = 4 * (tid >> 3);            // the quad's first unit
  const int i = ubase + ((lane >> 1) & 3);     // this lane pair's unit after the reduction
  const bool writer = (lane & 1) == 0;
  const bool ok_i = i < C;
  // W_rec[ubase + u][4 (8 q + sl) + e], paired for the packed FMA.
  float2 w[4][kQ][2];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int unit = ubase + u;
    const float* wr = p.W + static_cast<size_t>(unit < C ? unit : 0) * n_in + p.n_x;
#pragma unroll
    for (int q = 0; q < kQ; ++q)
#pragma unroll
      for (int ep = 0; ep < 2; ++ep) {
        const int k = 4 * (8 * q + sl) + 2 * ep;
        w[u][q][ep] = make_float2(unit < C && k < C ? __ldg(wr + k) : 0.f,
                                  unit < C && k + 1 < C ? __ldg(wr + k + 1) : 0.f);
      }
  }
  const float inv_tau = ok_i ? 1.f / __ldg(p.tau + i) : 0.f;
  bool rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rok[r] = row0 + r < B;
    // The pair's even lane writes each slot once (zero where no unit or row lives).
    if (writer)
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
      const float4* hv = reinterpret_cast<const float4*>(&hs[cur][r][0]);
      float2 acc2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) acc2[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const float4 v = hv[8 * q + sl];
        const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc2[u] = fma2(w[u][q][0], v01, acc2[u]);
          acc2[u] = fma2(w[u][q][1], v23, acc2[u]);
        }
      }
      float au[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) au[u] = acc2[u].x + acc2[u].y;
      a[r] = quad_reduce_scatter(au, lane);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float at = a[r] + xc[r];
      const float e = tanhf(at);
      const float d = __expf(-tc[r] * inv_tau);
      const float hp = hs[cur][r][ok_i ? i : 0];
      const float h = d * hp + (1.f - d) * e;
      if (writer) {
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
  constexpr int kQ = Quad<CP>::kQ;
  __shared__ __align__(16) float das[2][R][CP];  // da of the step, double buffered
  __shared__ __align__(16) float ring[kDecayRing][R][4][CP];  // dH, e, h_{t-1}, ts by step
  // The first kernel of its call (an ordinary launch): its dependents -- the operand build,
  // which reads only the forward's outputs and the inputs -- may start beside it at once.
  grid_dep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, sl = lane & 7;
  const int B = p.B, K = p.K, C = p.C, n_in = p.n_x + C;
  const int row0 = blockIdx.x * R;
  const int ubase = 4 * (tid >> 3);            // the quad's first unit
  const int j = ubase + ((lane >> 1) & 3);     // this lane pair's unit after the reduction
  const bool writer = (lane & 1) == 0;
  const bool ok_j = j < C;
  // Column ubase + u of W_rec over the rows 4 (8 q + sl) + e, paired for the packed FMA.
  float2 wc[4][kQ][2];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int unit = ubase + u;
    const float* col = p.W + p.n_x + (unit < C ? unit : 0);
#pragma unroll
    for (int q = 0; q < kQ; ++q)
#pragma unroll
      for (int ep = 0; ep < 2; ++ep) {
        const int k = 4 * (8 * q + sl) + 2 * ep;
        wc[u][q][ep] =
            make_float2(unit < C && k < C ? __ldg(col + static_cast<size_t>(k) * n_in) : 0.f,
                        unit < C && k + 1 < C ? __ldg(col + static_cast<size_t>(k + 1) * n_in) : 0.f);
      }
  }
  const float inv_tau = ok_j ? 1.f / __ldg(p.tau + j) : 0.f;
  bool rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rok[r] = row0 + r < B;
  // The inputs of each step -- dH, e = tanh(a), h_{t-1} (units along the row) and ts -- arrive
  // in a ring of kDecayRing shared-memory slots by cp.async, two steps ahead of their use:
  // thread u < C copies unit u of the three vectors, thread C copies ts.  Slots of units and
  // rows that do not exist stay zero.
  for (int e = tid; e < kDecayRing * R * 4 * CP; e += 2 * CP) (&ring[0][0][0][0])[e] = 0.f;
  __syncthreads();
  auto issue = [&](int t) {
    const int sl3 = t % kDecayRing;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (!rok[r]) continue;
      const size_t tb = static_cast<size_t>(t) * B + row0 + r;
      if (tid < C) {
        cp_async_4(smem_addr(&ring[sl3][r][0][tid]), p.dH + tb * C + tid);
        cp_async_4(smem_addr(&ring[sl3][r][1][tid]), p.E + tb * C + tid);
        cp_async_4(smem_addr(&ring[sl3][r][2][tid]),
                   t > 0 ? p.H + (tb - B) * C + tid
                         : p.h0 + static_cast<size_t>(row0 + r) * C + tid);
      } else if (tid == C) {
        cp_async_4(smem_addr(&ring[sl3][r][3][0]), p.ts + tb);
      }
    }
  };
  float G[R], acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) G[r] = acc[r] = 0.f;
  issue(K - 1);
  cp_async_commit();
  if (K >= 2) issue(K - 2);
  cp_async_commit();
  cp_async_wait<1>();  // step K - 1's copies (K - 2's may be pending)
  __syncthreads();
  for (int t = K - 1; t >= 0; --t) {
    const int cur = t & 1, sl3 = t % kDecayRing;
    // Step t - 2 goes into the slot step t + 1 used (every thread is past it: the barrier of
    // step t + 1); one group per step, empty at the end, keeps the wait count uniform.
    if (t >= 2) issue(t - 2);
    cp_async_commit();
    float dv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int jj = ok_j ? j : 0;
      const float dHc = ring[sl3][r][0][jj], ec = ring[sl3][r][1][jj];
      const float hpc = ring[sl3][r][2][jj], tsc = ring[sl3][r][3][0];
      G[r] += ok_j ? dHc : 0.f;
      const float d = __expf(-tsc * inv_tau);
      dv[r] = d;
      const float da = G[r] * (1.f - d) * (1.f - ec * ec);
      acc[r] += G[r] * (hpc - ec) * d * tsc * inv_tau * inv_tau;
      if (writer) {
        das[cur][r][j] = ok_j ? da : 0.f;
        if (ok_j && rok[r]) {
          __nv_bfloat16* q = p.da + (static_cast<size_t>(t) * B + row0 + r) * 2 * p.mp + j;
          const __nv_bfloat16 hi = __float2bfloat16_rn(da);
          q[0] = hi;
          q[p.mp] = __float2bfloat16_rn(da - __bfloat162float(hi));
        }
      }
    }
    cp_async_wait<1>();  // step t - 1's copies are in (step t - 2's may be pending)
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4* dv4 = reinterpret_cast<const float4*>(&das[cur][r][0]);
      float2 acc2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) acc2[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const float4 v = dv4[8 * q + sl];
        const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc2[u] = fma2(wc[u][q][0], v01, acc2[u]);
          acc2[u] = fma2(wc[u][q][1], v23, acc2[u]);
        }
      }
      float au[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) au[u] = acc2[u].x + acc2[u].y;
      G[r] = G[r] * dv[r] + quad_reduce_scatter(au, lane);
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (writer && ok_j && rok[r]) {
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

int decay_bwd_ctas(int B) { return (B + decay_rows(B) - 1) / decay_rows(B); }

cudaError_t decay_proj_launch(const float* x, const float* W, const float* b, int BK, int C,
                              int n_x, float* E, cudaStream_t s) {
  if (C > kDecayMaxC) return cudaErrorInvalidValue;
  LaunchCfg c;
  c.grid = dim3((C + kPC - 1) / kPC, (BK + kPR - 1) / kPR, 1);
  c.block = dim3(256, 1, 1);
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
