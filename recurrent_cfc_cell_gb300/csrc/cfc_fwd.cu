// cfc_fwd.cu -- forward recurrence of the CfC cell over all K steps in one persistent launch.
//
// Successor of cfc_step_batched (page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor", sections "Problem" and "Architecture Choice"): that kernel ran one CfC step per
// launch, first as a single block looping over the batch, then as one block per batch row,
// 64 launches per training step.  Here one launch runs the whole K-loop:
//
//   * a thread-block cluster of CS CTAs serves R batch rows; CTA `rank` owns hidden channels
//     [16*rank, 16*rank+16) and keeps the 64 matching rows of W (4 gates x 16 channels, over the
//     padded z = [u_t ; h_{t-1}]) in REGISTERS for the whole launch: 256 threads = 4 K-slices x
//     64 rows, KW weights each;
//   * per step every CTA computes its 64 pre-activations for its R rows (z read from shared
//     memory by warp-uniform broadcast loads), applies tanh / sigmoid, writes H and the cache,
//     and pushes its 16 new h values to every CTA of the cluster with st.async into their
//     shared z buffer; the remote mbarrier counts the bytes, so the next step waits on one
//     local mbarrier instead of a cluster-wide barrier;
//   * z, the K-slice partial sums and the mbarriers are double-buffered by step parity.
//
// The cell (the pages name the kernels but print no equations):
//   P_g = W_g [u_t ; h_{t-1}] + b_g,  ff1 = tanh(P_ff1), ff2 = tanh(P_ff2),
//   gate = sigmoid(P_ta * ts[t,b] + P_tb),  h_t = ff1 * (1 - gate) + gate * ff2.
#include "cfc_kernels.h"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kKS = 4;  // K-slices of the z vector (one per 64-thread group)

template <int KW>
__global__ void __launch_bounds__(kRecThreads, 1) cfc_fwd_kernel(const FwdParams p) {
  extern __shared__ __align__(16) float smem[];
  const int R = p.R;
  const int NZp = p.NZp;
  float* zbuf = smem;                         // [2][R][NZp]
  float* red = zbuf + 2 * R * NZp;            // [2][R][4][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + 2 * R * kKS * kRowsPerCta);  // [2]
  int* abort_flag = reinterpret_cast<int*>(bars + 2);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * R;  // first batch row of this cluster
  const int CS = p.CS;
  const int B = p.B, K = p.K, C = p.C, n_x = p.n_x, n_in = p.n_in, nxp = p.nxp;

  // ---- weights of this thread: row `lr` (channel-major, gate-minor), slice `ks` ----
  const int ks = tid >> 6;
  const int lr = tid & 63;
  const int ch = kChanPerCta * rank + (lr >> 2);
  const int gt_idx = lr & 3;
  float w[KW];
#pragma unroll
  for (int c = 0; c < KW; ++c) {
    const int zc = ks * KW + c;
    float v = 0.f;
    if (ch < C) {
      int col = -1;
      if (zc < n_x) col = zc;
      else if (zc >= nxp && zc - nxp < C) col = n_x + (zc - nxp);
      if (col >= 0) v = p.W[(static_cast<size_t>(gt_idx) * C + ch) * n_in + col];
    }
    w[c] = v;
  }
  const float bias = (ch < C) ? p.bias[gt_idx * C + ch] : 0.f;

  // ---- prologue: barriers, z_0 = [u_0 ; h0] ----
  const uint32_t bar0 = smem_addr(&bars[0]);  // bars[s] lives at bar0 + 8 s
  const uint32_t tx_bytes = static_cast<uint32_t>(CS * R * kChanPerCta * 4);
  if (tid == 0) {
    mbar_init((bar0 + 0u), 1);
    mbar_init((bar0 + 8u), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  for (int e = tid; e < 2 * R * NZp; e += kRecThreads) zbuf[e] = 0.f;
  __syncthreads();
  for (int e = tid; e < R * n_x; e += kRecThreads) {
    const int r = e / n_x, k = e - (e / n_x) * n_x;
    const int b = row0 + r;
    if (b < B) zbuf[r * NZp + k] = p.u[static_cast<size_t>(b) * n_x + k];
  }
  for (int e = tid; e < R * C; e += kRecThreads) {
    const int r = e / C, j = e - (e / C) * C;
    const int b = row0 + r;
    if (b < B) zbuf[r * NZp + nxp + j] = p.h0[static_cast<size_t>(b) * C + j];
  }
  // Step t consumes h_{t-1} through bars[t & 1]; arm the first two consumers (t = 1, 2).
  if (tid == 0) {
    if (K >= 2) mbar_arrive_expect_tx((bar0 + 8u), tx_bytes);
    if (K >= 3) mbar_arrive_expect_tx((bar0 + 0u), tx_bytes);
  }
  cluster_sync_all();

  uint32_t phase = 0;  // bit s: parity of the next phase of bars[s] to wait for
  for (int t = 0; t < K; ++t) {
    const int s = t & 1;
    const float* z = zbuf + s * R * NZp;
    float* rd = red + s * R * kKS * kRowsPerCta;

    // Prefetch u_{t+1} into the other z buffer (last read two steps ago).
    if (t + 1 < K) {
      float* zn = zbuf + (s ^ 1) * R * NZp;
      const float* un = p.u + (static_cast<size_t>(t + 1) * B) * n_x;
      for (int e = tid; e < R * n_x; e += kRecThreads) {
        const int r = e / n_x, k = e - (e / n_x) * n_x;
        const int b = row0 + r;
        zn[r * NZp + k] = (b < B) ? un[static_cast<size_t>(b) * n_x + k] : 0.f;
      }
    }

    // Wait for every CTA's slice of h_{t-1}.
    if (t > 0) {
      const bool ok = mbar_wait_bounded_cluster((bar0 + 8u * (s)), (phase >> s) & 1u, p.status);
      phase ^= (1u << s);
      if (!ok) *abort_flag = 1;
      if (tid == 0 && t + 2 <= K - 1) mbar_arrive_expect_tx((bar0 + 8u * (s)), tx_bytes);
    }

    // Pre-activation partial sums over this thread's K-slice for every row of the group.
    for (int r = 0; r < R; ++r) {
      const float4* zr = reinterpret_cast<const float4*>(z + r * NZp + ks * KW);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int c = 0; c < KW / 4; ++c) {
        const float4 v = zr[c];
        a0 = fmaf(w[4 * c + 0], v.x, a0);
        a1 = fmaf(w[4 * c + 1], v.y, a1);
        a2 = fmaf(w[4 * c + 2], v.z, a2);
        a3 = fmaf(w[4 * c + 3], v.w, a3);
      }
      rd[(r * kKS + ks) * kRowsPerCta + lr] = (a0 + a1) + (a2 + a3);
    }
    __syncthreads();
    if (*abort_flag) break;

    // Gate phase: one thread per (row, W row); the four gates of a channel sit in a lane quad.
    for (int idx = tid; idx < R * kRowsPerCta; idx += kRecThreads) {
      const int r = idx >> 6;
      const float* q = rd + r * kKS * kRowsPerCta + lr;
      const float P = (((q[0] + q[kRowsPerCta]) + q[2 * kRowsPerCta]) + q[3 * kRowsPerCta]) + bias;
      const int base = lane & ~3;
      const float P_ff1 = __shfl_sync(0xffffffffu, P, base + 0);
      const float P_ff2 = __shfl_sync(0xffffffffu, P, base + 1);
      const float P_ta = __shfl_sync(0xffffffffu, P, base + 2);
      const float P_tb = __shfl_sync(0xffffffffu, P, base + 3);
      const int b = row0 + r;
      const float tsv = (b < B) ? p.ts[static_cast<size_t>(t) * B + b] : 1.f;
      const float f1 = tanhf(P_ff1);
      const float f2 = tanhf(P_ff2);
      const float g = sigmoid_acc(fmaf(P_ta, tsv, P_tb));
      const float h = f1 * (1.f - g) + g * f2;
      if (b < B && ch < C) {
        const size_t tb = static_cast<size_t>(t) * B + b;
        if (gt_idx == 0) {
          p.H[tb * C + ch] = h;
        } else {
          const float cv = (gt_idx == 1) ? f1 : (gt_idx == 2 ? f2 : g);
          p.cache[(tb * 3 + (gt_idx - 1)) * C + ch] = cv;
        }
      }
      if (t + 1 < K) {
        float* zn = zbuf + (s ^ 1) * R * NZp;
        const uint32_t dst = smem_addr(zn + r * NZp + nxp + ch);
        for (int qr = gt_idx; qr < CS; qr += 4) {
          st_async_b32(map_to_rank(dst, qr), h, map_to_rank((bar0 + 8u * (s ^ 1)), qr));
        }
      }
    }
  }
  // No CTA leaves while a peer may still address its shared memory.
  cluster_sync_all();
}

template <int KW>
cudaError_t set_attrs(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(cfc_fwd_kernel<KW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(cfc_fwd_kernel<KW>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                              1);
}

template <int KW>
cudaError_t prepare_kw(int CS, size_t smem, int* max_active) {
  cudaError_t e = set_attrs<KW>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, 1, 1);
  cfg.blockDim = dim3(kRecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_active, cfc_fwd_kernel<KW>, &cfg);
}

template <int KW>
cudaError_t launch_kw(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * p.CS, 1, 1);
  cfg.blockDim = dim3(kRecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cfc_fwd_kernel<KW>, p);
}

constexpr int kKWs[] = {8, 12, 16, 24, 32, 44, 48, 64, 80};

}  // namespace

int fwd_kw_for(int nxp, int CS) {
  const int nz = nxp + kChanPerCta * CS;
  if (nz > kMaxZ) return -1;
  const int need = (nz + kKS - 1) / kKS;
  for (int kw : kKWs)
    if (kw >= need) return kw;
  return -1;
}

size_t fwd_smem_bytes(int R, int NZp) {
  return sizeof(float) * (2ull * R * NZp + 2ull * R * kKS * kRowsPerCta) + 2 * sizeof(uint64_t) +
         16;
}

cudaError_t fwd_prepare(int KW, int CS, size_t smem, int* max_active) {
  switch (KW) {
    case 8: return prepare_kw<8>(CS, smem, max_active);
    case 12: return prepare_kw<12>(CS, smem, max_active);
    case 16: return prepare_kw<16>(CS, smem, max_active);
    case 24: return prepare_kw<24>(CS, smem, max_active);
    case 32: return prepare_kw<32>(CS, smem, max_active);
    case 44: return prepare_kw<44>(CS, smem, max_active);
    case 48: return prepare_kw<48>(CS, smem, max_active);
    case 64: return prepare_kw<64>(CS, smem, max_active);
    case 80: return prepare_kw<80>(CS, smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t fwd_launch(int KW, const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
  switch (KW) {
    case 8: return launch_kw<8>(p, n_clusters, smem, s);
    case 12: return launch_kw<12>(p, n_clusters, smem, s);
    case 16: return launch_kw<16>(p, n_clusters, smem, s);
    case 24: return launch_kw<24>(p, n_clusters, smem, s);
    case 32: return launch_kw<32>(p, n_clusters, smem, s);
    case 44: return launch_kw<44>(p, n_clusters, smem, s);
    case 48: return launch_kw<48>(p, n_clusters, smem, s);
    case 64: return launch_kw<64>(p, n_clusters, smem, s);
    case 80: return launch_kw<80>(p, n_clusters, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cfc
