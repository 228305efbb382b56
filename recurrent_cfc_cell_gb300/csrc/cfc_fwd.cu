// cfc_fwd.cu -- forward recurrence of the CfC cell over all K steps in one persistent launch.
//
// Successor of cfc_step_batched (page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor", sections "Problem" and "Architecture Choice"): that kernel ran one CfC step per
// launch, first as a single block looping over the batch, then as one block per batch row,
// 64 launches per training step.  Here one launch runs the whole K-loop.
//
// The cell (the pages name the kernels but print no equations):
//   P_g = W_g [u_t ; h_{t-1}] + b_g,  ff1 = tanh(P_ff1), ff2 = tanh(P_ff2),
//   gate = sigmoid(P_ta * ts[t,b] + P_tb),  h_t = ff1 * (1 - gate) + gate * ff2.
// The input part X = W_u u_t + b is computed beforehand for all steps (cfc_inproj.cu) and
// handed over in place in H / cache; this kernel adds the recurrent part W_h h_{t-1}.
//
// Layout and schedule (every step is warp-local; no CTA-wide barrier inside the K-loop):
//   * a thread-block cluster of CS CTAs serves R batch rows; CTA `rank` owns hidden channels
//     [16*rank, 16*rank+16), and warp w of it owns channels 16*rank + 2w + {0, 1}: 8 W rows
//     (2 channels x 4 gates);
//   * lanes 16ci + sl keep the four gate rows of channel ci over the sl-th sixteenth of the
//     recurrent columns (CS columns) in REGISTERS, so every h value loaded from shared memory
//     feeds four FMAs; a 5-shuffle reduce-scatter over the 16 lanes leaves gate g of channel ci
//     in lanes 16ci + 4g + (0..3), so activations, H / cache stores and the st.async pushes of
//     the new h to all CS CTAs happen in the same warp;
//   * h rows in shared memory are split into sixteen slices padded to an odd number of 16-byte
//     chunks, so the vector loads of a quarter-warp hit distinct banks;
//   * X and ts of step t+1 are loaded into registers during step t (X with an L2 load, since
//     this kernel later overwrites that location with H / cache), so no global-memory latency
//     sits on the serial chain; the number of batch rows per cluster (R) is a compile-time
//     parameter so these per-row values stay in registers;
//   * the destination mbarrier counts the pushed bytes, so a step waits on one local mbarrier.
//     h buffers and mbarriers alternate with the step parity.
#include "cfc_kernels.h"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

template <int CS>
struct FwdShape {
  static constexpr int CHP = kChanPerCta * CS;  // padded channel count
  static constexpr int HS = CHP / 16;           // h columns per lane (= CS)
  // Slice pitch: vector loads of 8 consecutive lanes must cover distinct banks.
  static constexpr int HSP = (HS >= 4 && (HS / 4) % 2 == 0) ? HS + 4 : HS;
  static constexpr int HROW = 16 * HSP;         // h row in shared memory
};

// Load n consecutive floats (n = 1, 2 or a multiple of 4) from shared memory.
template <int N>
__device__ __forceinline__ void lds_vec(const float* src, float (&dst)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + c);
      dst[c] = v.x; dst[c + 1] = v.y; dst[c + 2] = v.z; dst[c + 3] = v.w;
    }
  } else if constexpr (N == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    dst[0] = v.x; dst[1] = v.y;
  } else {
    dst[0] = src[0];
  }
}

template <int CS>
__device__ __forceinline__ int hpos(int j) {
  using S = FwdShape<CS>;
  return (j / S::HS) * S::HSP + (j % S::HS);
}

template <int CS, int R>
__global__ void __launch_bounds__(kRecThreads, 2) cfc_fwd_kernel(const FwdParams p) {
  using S = FwdShape<CS>;
  extern __shared__ __align__(16) float smem[];
  float* hbuf = smem;  // [2][R][HROW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(hbuf + 2 * R * S::HROW);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * R;  // first batch row of this cluster
  const int B = p.B, K = p.K, C = p.C, n_x = p.n_x, n_in = p.n_in;

  // This lane: channel ci, column slice sl; after the reduce-scatter it holds gate g.
  const int ci = lane >> 4;
  const int sl = lane & 15;
  const int g = (lane >> 2) & 3;
  const int ch = kChanPerCta * rank + 2 * warp + ci;
  float wh[4][S::HS];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg)
#pragma unroll
    for (int c = 0; c < S::HS; ++c) {
      const int j = sl * S::HS + c;
      wh[gg][c] = (ch < C && j < C)
                      ? p.W[(static_cast<size_t>(gg) * C + ch) * n_in + n_x + j] : 0.f;
    }
  // Per-lane addresses, computed once: the K-loop only advances pointers by a fixed stride
  // per step and issues predicated loads and stores (no index arithmetic or divergent
  // branches on the serial chain).
  //   X of this lane's (channel, gate g) -- written in place into H / cache by the
  //   projection -- for row row0 + r of step t: xp + t * xstep + r * xrow;
  //   the value this lane stores (lane q < 4: H, ff1, ff2, gate) likewise with q for g.
  const int q = lane & 15;
  const int chc = ch < C ? ch : 0;  // padded channels read a valid location
  const size_t xrow = (g == 0) ? static_cast<size_t>(C) : 3ull * C;
  const size_t srow = (q == 0) ? static_cast<size_t>(C) : 3ull * C;
  const float* xp = ((g == 0) ? p.H : p.cache + static_cast<size_t>(g - 1) * C) + chc +
                    static_cast<size_t>(row0 < B ? row0 : 0) * xrow;
  float* sp = ((q == 0) ? p.H : p.cache + static_cast<size_t>(q > 0 && q < 4 ? q - 1 : 0) * C) +
              chc + static_cast<size_t>(row0 < B ? row0 : 0) * srow;
  const float* tsp = p.ts + (row0 < B ? row0 : 0);
  const size_t xstep = static_cast<size_t>(B) * xrow, sstep = static_cast<size_t>(B) * srow;
  bool xok[R], sok[R], rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rok[r] = row0 + r < B;
    xok[r] = rok[r] && ch < C;
    sok[r] = xok[r] && q < 4;
  }

  // X and ts of the step whose X row starts at xs (ts at tss), for every row of the group.
  auto load_step = [&](const float* xs, const float* tss, float (&xv)[R], float (&tv)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xv[r] = xok[r] ? __ldcg(xs + r * xrow) : 0.f;
      tv[r] = rok[r] ? __ldg(tss + r) : 0.f;
    }
  };

  // ---- prologue ----
  const uint32_t bar0 = smem_addr(&bars[0]);  // bars[s] lives at bar0 + 8 s
  const uint32_t tx_bytes = static_cast<uint32_t>(CS * R * kChanPerCta * 4);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    fence_mbar_init_cluster();
  }
  for (int e = tid; e < 2 * R * S::HROW; e += kRecThreads) smem[e] = 0.f;
  __syncthreads();
  for (int e = tid; e < R * C; e += kRecThreads) {
    const int r = e / C, j = e - (e / C) * C;
    if (row0 + r < B)
      hbuf[r * S::HROW + hpos<CS>(j)] = p.h0[static_cast<size_t>(row0 + r) * C + j];
  }
  float xc[R], tc[R];  // X and ts of the current step
  load_step(xp, tsp, xc, tc);
  // Step t consumes h_{t-1} through bars[t & 1]; arm the first two consumers (t = 1, 2).
  if (tid == 0) {
    if (K >= 2) mbar_arrive_expect_tx(bar0 + 8u, tx_bytes);
    if (K >= 3) mbar_arrive_expect_tx(bar0, tx_bytes);
  }
  __syncthreads();     // h0 visible to every warp
  cluster_sync_all();  // barrier inits and buffers ready cluster-wide

  // Pushes of the new h: lane q < CS writes this lane's channel into CTA q's buffer.  Remote
  // addresses of buffer 0 / row 0; buffer d, row r is (d * R + r) * HROW floats further on.
  const bool pushes = q < CS;
  // (ch, not the clamped chc: a padded channel has its own slot in the padded h row.)
  const uint32_t push0 = pushes ? map_to_rank(smem_addr(hbuf + hpos<CS>(ch)), q) : 0u;
  const uint32_t rbar0 = pushes ? map_to_rank(bar0, q) : 0u;

  const float* xnext = xp + xstep;  // X and ts of step t + 1
  const float* tsnext = tsp + B;
  uint32_t phase = 0;  // bit s: parity of the next phase of bars[s] to wait for
  for (int t = 0; t < K; ++t) {
    const int s = t & 1;
    // X and ts of the next step; consumed one step later, so their latency is hidden.
    float xn[R], tn[R];
    if (t + 1 < K) {
      load_step(xnext, tsnext, xn, tn);
      xnext += xstep;
      tsnext += B;
    }

    // h_{t-1} from every CTA of the cluster.
    if (t > 0) {
      const bool ok = __all_sync(
          0xffffffffu, mbar_wait_bounded_cluster(bar0 + 8u * s, (phase >> s) & 1u, p.status));
      phase ^= (1u << s);
      if (!ok) break;
      if (tid == 0 && t + 2 <= K - 1) mbar_arrive_expect_tx(bar0 + 8u * s, tx_bytes);
    }

    const float* hb = hbuf + s * R * S::HROW + sl * S::HSP;
    const uint32_t pdst = push0 + static_cast<uint32_t>((s ^ 1) * R * S::HROW * 4);
    const uint32_t pbar = rbar0 + 8u * (s ^ 1);
    const bool b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float hv[S::HS];
      lds_vec<S::HS>(hb + r * S::HROW, hv);
      float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < S::HS; ++c)
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) a[gg] = fmaf(wh[gg][c], hv[c], a[gg]);
      // Reduce-scatter over the 16 lanes of the channel: lane keeps gate (lane >> 2) & 3.
      const float k0 = b3 ? a[2] : a[0], k1 = b3 ? a[3] : a[1];
      const float s0 = k0 + __shfl_xor_sync(0xffffffffu, b3 ? a[0] : a[2], 8);
      const float s1 = k1 + __shfl_xor_sync(0xffffffffu, b3 ? a[1] : a[3], 8);
      float acc = (b2 ? s1 : s0) + __shfl_xor_sync(0xffffffffu, b2 ? s0 : s1, 4);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      const float P = acc + xc[r];

      // Activations: lanes of gate 0 / 1 evaluate tanh(P) = 2 sigmoid(2P) - 1, lanes of gate
      // 2 the time gate sigmoid(P_ta ts + P_tb) (P_tb from the gate-3 lane four lanes up).
      const float P_tb = __shfl_sync(0xffffffffu, P, (lane + 4) & 31);
      const float x =
          (g < 2) ? 2.f * P : fmaf(P, tc[r], P_tb);
      const float sg = sigmoid_acc(x);
      const float y = (g < 2) ? fmaf(2.f, sg, -1.f) : sg;
      const int half = lane & 16;
      const float f1 = __shfl_sync(0xffffffffu, y, half + 0);
      const float f2 = __shfl_sync(0xffffffffu, y, half + 4);
      const float gt = __shfl_sync(0xffffffffu, y, half + 8);
      const float h = f1 * (1.f - gt) + gt * f2;
      st_async_b32_if(pushes && t + 1 < K, pdst + static_cast<uint32_t>(r * S::HROW * 4), h,
                      pbar);
      const float sv = (q == 0) ? h : (q == 1) ? f1 : (q == 2 ? f2 : gt);
      if (sok[r]) sp[r * srow] = sv;
    }
    sp += sstep;
    if (t + 1 < K) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        xc[r] = xn[r];
        tc[r] = tn[r];
      }
    }
  }
  // No CTA leaves while a peer may still address its shared memory.
  cluster_sync_all();
}

template <int CS, int R>
cudaError_t prepare_k(size_t smem, int* max_active) {
  // The attribute is a per-function maximum: set it to the device's opt-in limit once.
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(optin)) {
    *max_active = 0;
    return cudaSuccess;
  }
  auto* kern = cfc_fwd_kernel<CS, R>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  return cudaOccupancyMaxActiveClusters(max_active, kern, &cfg);
}

template <int CS, int R>
cudaError_t launch_k(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * CS, 1, 1);
  cfg.blockDim = dim3(kRecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cfc_fwd_kernel<CS, R>, p);
}

template <int CS>
cudaError_t prepare_cs(int R, size_t smem, int* max_active) {
  switch (R) {
    case 1: return prepare_k<CS, 1>(smem, max_active);
    case 2: return prepare_k<CS, 2>(smem, max_active);
    case 4: return prepare_k<CS, 4>(smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

template <int CS>
cudaError_t launch_cs(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
  switch (p.R) {
    case 1: return launch_k<CS, 1>(p, n_clusters, smem, s);
    case 2: return launch_k<CS, 2>(p, n_clusters, smem, s);
    case 4: return launch_k<CS, 4>(p, n_clusters, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t fwd_smem_bytes(int R, int CS) {
  const size_t hs = CS;
  const size_t hsp = (hs >= 4 && (hs / 4) % 2 == 0) ? hs + 4 : hs;
  return sizeof(float) * 2ull * R * 16 * hsp + 2 * sizeof(uint64_t) + 16;
}

cudaError_t fwd_prepare(int CS, int R, size_t smem, int* max_active) {
  switch (CS) {
    case 1: return prepare_cs<1>(R, smem, max_active);
    case 2: return prepare_cs<2>(R, smem, max_active);
    case 4: return prepare_cs<4>(R, smem, max_active);
    case 8: return prepare_cs<8>(R, smem, max_active);
    case 16: return prepare_cs<16>(R, smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t fwd_launch(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
  switch (p.CS) {
    case 1: return launch_cs<1>(p, n_clusters, smem, s);
    case 2: return launch_cs<2>(p, n_clusters, smem, s);
    case 4: return launch_cs<4>(p, n_clusters, smem, s);
    case 8: return launch_cs<8>(p, n_clusters, smem, s);
    case 16: return launch_cs<16>(p, n_clusters, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cfc
