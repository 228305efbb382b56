// cfc_bwd.cu -- reverse-time BPTT recurrence of the CfC cell over all K steps in one launch.
//
// Successor of cfc_step_backward_batched (page "K-loop Parallelization -- Block-per-Batch
// Kernel Refactor", sections "Problem", "Architecture Choice" item 3 and "Per-Kernel
// Breakdown"): that kernel ran one reverse step per launch and accumulated weight gradients
// with `+=` into a per-(batch row, channel) scratch, reduced after the K-loop.  Here the
// recurrence only produces the pre-activation gradients d_pre[t][b][gate][i] (each written
// once, no atomics, no `+=`); the weight and bias gradients are one dense contraction and one
// axis-0 sum afterwards.
//
// Per step (t = K-1 .. 0), with gate, ff1, ff2 from the forward cache:
//   dh      = dH[t] + delta                        (delta = 0 at t = K-1)
//   dP_ff1  = dh (1 - gate)(1 - ff1^2),  dP_ff2 = dh gate (1 - ff2^2)
//   ds      = dh (ff2 - ff1) gate (1 - gate),  dP_ta = ds ts[t,b],  dP_tb = ds
//   delta  <- W_h^T d_pre[t]      (W_h = the C recurrent columns of W);   dh0 = final delta.
//
// Layout: a cluster of CS CTAs serves R batch rows; CTA `rank` owns channels
// [16*rank, 16*rank+16) and its 64 W rows.  Thread (j, rg) keeps W_h[rows of group rg][j] in
// registers (4*CS values), computes the partial delta[j] over its rows and pushes it with
// st.async to the CTA that owns channel j, into slot (rank, rg).  The owner adds its 16 slots
// in a fixed order, so the result is bitwise reproducible.
#include "cfc_kernels.h"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kSlots = 16;  // partial-delta contributions each channel receives (CS * RG)

template <int CS>
__global__ void __launch_bounds__(kRecThreads, 1) cfc_bwd_kernel(const BwdParams p) {
  constexpr int RG = 16 / CS;          // row groups per CTA
  constexpr int RPT = kRowsPerCta / RG;  // W rows per thread (= 4 * CS)
  constexpr int CHP = kChanPerCta * CS;  // padded channel count

  extern __shared__ __align__(16) float smem[];
  const int R = p.R;
  float* dbuf = smem;                                  // [2][R][16 slots][16]
  float* dps = dbuf + 2 * R * kSlots * kChanPerCta;    // [2][R][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(dps + 2 * R * kRowsPerCta);
  int* abort_flag = reinterpret_cast<int*>(bars + 2);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * R;
  const int B = p.B, K = p.K, C = p.C, n_x = p.n_x, n_in = p.n_in;

  // ---- W_h^T block of this thread: column j, rows [rg*RPT, rg*RPT + RPT) ----
  const int j = tid % CHP;
  const int rg = tid / CHP;
  float w[RPT];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int lrow = rg * RPT + k;
    const int ch = kChanPerCta * rank + (lrow >> 2);
    const int g = lrow & 3;
    w[k] = (ch < C && j < C) ? p.W[(static_cast<size_t>(g) * C + ch) * n_in + n_x + j] : 0.f;
  }
  // Destination of this thread's partial: owner CTA of channel j, slot (rank, rg).
  const int owner = j / kChanPerCta;
  const int slot = rank * RG + rg;

  // Gate-phase identity: row lr = 4 i + g of this CTA.
  const int lr = tid & 63;
  const int gi = lr & 3;
  const int ch = kChanPerCta * rank + (lr >> 2);

  const uint32_t bar0 = smem_addr(&bars[0]);  // bars[s] lives at bar0 + 8 s
  const uint32_t tx_bytes = static_cast<uint32_t>(R * kSlots * kChanPerCta * 4);
  if (tid == 0) {
    mbar_init((bar0 + 0u), 1);
    mbar_init((bar0 + 8u), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  // Consumer c (= the step that reads delta; -1 is the dh0 epilogue) uses bars[c & 1].
  // Consumers run c = K-2 .. -1; arm the first two.
  if (tid == 0) {
    mbar_arrive_expect_tx((bar0 + 8u * ((K - 2) & 1)), tx_bytes);
    if (K >= 2) mbar_arrive_expect_tx((bar0 + 8u * ((K - 3) & 1)), tx_bytes);
  }
  cluster_sync_all();

  uint32_t phase = 0;
  for (int t = K - 1; t >= 0; --t) {
    const int s = t & 1;
    const float* din = dbuf + s * R * kSlots * kChanPerCta;
    float* dp_s = dps + s * R * kRowsPerCta;

    if (t < K - 1) {
      const bool ok = mbar_wait_bounded_cluster((bar0 + 8u * (s)), (phase >> s) & 1u, p.status);
      phase ^= (1u << s);
      if (!ok) *abort_flag = 1;
      if (tid == 0 && t - 2 >= -1) mbar_arrive_expect_tx((bar0 + 8u * (s)), tx_bytes);
    }

    // d_pre for (row r, channel ch, gate gi); delta summed over the 16 slots in fixed order.
    for (int idx = tid; idx < R * kRowsPerCta; idx += kRecThreads) {
      const int r = idx >> 6;
      const int b = row0 + r;
      float dsum = 0.f;
      if (t < K - 1) {
        const float* sl = din + r * kSlots * kChanPerCta + (lr >> 2);
        dsum = ((sl[(4 * gi + 0) * kChanPerCta] + sl[(4 * gi + 1) * kChanPerCta]) +
                sl[(4 * gi + 2) * kChanPerCta]) + sl[(4 * gi + 3) * kChanPerCta];
      }
      dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
      dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
      float dpv = 0.f;
      if (b < B && ch < C) {
        const size_t tb = static_cast<size_t>(t) * B + b;
        const float dh = p.dH[tb * C + ch] + dsum;
        const float f1 = p.cache[(tb * 3 + 0) * C + ch];
        const float f2 = p.cache[(tb * 3 + 1) * C + ch];
        const float g = p.cache[(tb * 3 + 2) * C + ch];
        const float ds = dh * (f2 - f1) * g * (1.f - g);
        if (gi == 0) dpv = dh * (1.f - g) * (1.f - f1 * f1);
        else if (gi == 1) dpv = dh * g * (1.f - f2 * f2);
        else if (gi == 2) dpv = ds * p.ts[tb];
        else dpv = ds;
        p.d_pre[(tb * 4 + gi) * C + ch] = dpv;
      }
      dp_s[r * kRowsPerCta + lr] = dpv;
    }
    __syncthreads();
    if (*abort_flag) break;

    // Partial delta[j] over this thread's rows, for every batch row; push to the owner.
    const int sn = s ^ 1;  // buffer of consumer t-1
    float* dst_base = dbuf + sn * R * kSlots * kChanPerCta;
    for (int r = 0; r < R; ++r) {
      const float4* d4 = reinterpret_cast<const float4*>(dp_s + r * kRowsPerCta + rg * RPT);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int k = 0; k < RPT / 4; ++k) {
        const float4 v = d4[k];
        a0 = fmaf(w[4 * k + 0], v.x, a0);
        a1 = fmaf(w[4 * k + 1], v.y, a1);
        a2 = fmaf(w[4 * k + 2], v.z, a2);
        a3 = fmaf(w[4 * k + 3], v.w, a3);
      }
      const float acc = (a0 + a1) + (a2 + a3);
      // Gather four consecutive channels into the lane whose j is a multiple of 4.
      const float v1 = __shfl_down_sync(0xffffffffu, acc, 1);
      const float v2 = __shfl_down_sync(0xffffffffu, acc, 2);
      const float v3 = __shfl_down_sync(0xffffffffu, acc, 3);
      if ((lane & 3) == 0) {
        const uint32_t dst =
            smem_addr(dst_base + (r * kSlots + slot) * kChanPerCta + (j % kChanPerCta));
        st_async_v4(map_to_rank(dst, owner), acc, v1, v2, v3, map_to_rank((bar0 + 8u * (sn)), owner));
      }
    }
  }

  // Epilogue: dh0 = delta after step 0 (consumer -1 reads bars[1]).
  if (!*abort_flag) {
    const bool ok = mbar_wait_bounded_cluster((bar0 + 8u), (phase >> 1) & 1u, p.status);
    if (!__syncthreads_or(ok ? 0 : 1)) {
      const float* din = dbuf + 1 * R * kSlots * kChanPerCta;
      for (int idx = tid; idx < R * kRowsPerCta; idx += kRecThreads) {
        const int r = idx >> 6;
        const int b = row0 + r;
        const float* sl = din + r * kSlots * kChanPerCta + (lr >> 2);
        float dsum = ((sl[(4 * gi + 0) * kChanPerCta] + sl[(4 * gi + 1) * kChanPerCta]) +
                      sl[(4 * gi + 2) * kChanPerCta]) + sl[(4 * gi + 3) * kChanPerCta];
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
        if (gi == 0 && b < B && ch < C) p.dh0[static_cast<size_t>(b) * C + ch] = dsum;
      }
    }
  }
  cluster_sync_all();
}

template <int CS>
cudaError_t prepare_cs(size_t smem, int* max_active) {
  cudaError_t e = cudaFuncSetAttribute(cfc_bwd_kernel<CS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cfc_bwd_kernel<CS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  return cudaOccupancyMaxActiveClusters(max_active, cfc_bwd_kernel<CS>, &cfg);
}

template <int CS>
cudaError_t launch_cs(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, cfc_bwd_kernel<CS>, p);
}

}  // namespace

size_t bwd_smem_bytes(int R) {
  return sizeof(float) * (2ull * R * kSlots * kChanPerCta + 2ull * R * kRowsPerCta) +
         2 * sizeof(uint64_t) + 16;
}

cudaError_t bwd_prepare(int CS, size_t smem, int* max_active) {
  switch (CS) {
    case 1: return prepare_cs<1>(smem, max_active);
    case 2: return prepare_cs<2>(smem, max_active);
    case 4: return prepare_cs<4>(smem, max_active);
    case 8: return prepare_cs<8>(smem, max_active);
    case 16: return prepare_cs<16>(smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t bwd_launch(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s) {
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
