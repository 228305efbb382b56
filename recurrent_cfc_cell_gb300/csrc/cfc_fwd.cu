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
//     [32*rank, 32*rank+32), and warp w of it owns channels 32*rank + 4w + {0..3}: 16 W rows
//     (4 channels x 4 gates);
//   * lanes 8cj + sl keep the four gate rows of channel cj over the sl-th eighth of the
//     recurrent columns (4*CS columns) in REGISTERS, so every h value loaded from shared memory
//     feeds four FMAs; a 4-shuffle reduce-scatter over the 8 lanes leaves gate g of channel cj
//     in lanes 8cj + 2g + (0, 1), and the activations and H / cache stores happen in the same
//     warp;
//   * the warp's four new h values are contiguous in the h row, so they travel as ONE 16-byte
//     st.async per destination CTA: a cluster moves 8*CS 16-byte pushes per CTA and step
//     (measured on GB300: few wide pushes per step exchange markedly faster than many 4-byte
//     ones once two clusters share an SM, and 32 channels per CTA halve the CTA count);
//   * h rows in shared memory are split into eight slices padded to an odd number of 16-byte
//     chunks, so the vector loads of the eight lanes of a channel hit distinct banks;
//   * X and ts of step t+1 are loaded into registers during step t (X with an L2 load, since
//     this kernel later overwrites that location with H / cache), so no global-memory latency
//     sits on the serial chain; the number of batch rows per cluster (R) is a compile-time
//     parameter so these per-row values stay in registers;
//   * the destination mbarrier counts the pushed bytes, so a step waits on one local mbarrier.
//     h buffers and mbarriers alternate with the step parity;
//   * per-lane addresses are computed once; the K-loop advances pointers by a fixed stride and
//     uses predicated loads, stores and st.async (no index arithmetic or divergent branches on
//     the serial chain);
//   * the W_h block of the CTA is read coalesced into shared memory in the prologue and from
//     there into registers.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

template <int CS>
struct FwdShape {
  static constexpr int CHP = kFwdChanPerCta * CS;  // padded channel count
  static constexpr int HS = CHP / 8;               // h columns per lane (= 4 CS)
  // Slice pitch: the vector loads of the 8 lanes of a channel must cover distinct banks.
  static constexpr int HSP = ((HS / 4) % 2 == 0) ? HS + 4 : HS;
  static constexpr int HROW = 8 * HSP;             // h row in shared memory
  static constexpr int WP = CHP + 4;               // row pitch of the staged W_h block
};

// Load N consecutive floats (N a multiple of 4) from shared memory as N / 2 pairs.
template <int N>
__device__ __forceinline__ void lds_pairs(const float* src, float2 (&dst)[N / 2]) {
  static_assert(N % 4 == 0, "h slices are whole float4s");
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + c);
    dst[c / 2] = make_float2(v.x, v.y);
    dst[c / 2 + 1] = make_float2(v.z, v.w);
  }
}

template <int CS>
__device__ __forceinline__ int hpos(int j) {
  using S = FwdShape<CS>;
  return (j / S::HS) * S::HSP + (j % S::HS);
}

// BF: H and the cache are stored as bf16 (FwdParams::out_bf16), X read from xH / xcache.
template <int CS, int R, bool BF>
__global__ void __launch_bounds__(kRecThreads, (CS >= 8 || R >= 8) ? 1 : 2) cfc_fwd_kernel(const FwdParams p) {
  using S = FwdShape<CS>;
  extern __shared__ __align__(16) float smem[];
  float* hbuf = smem;  // [2][R][HROW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(hbuf + 2 * R * S::HROW);

  grid_dep_launch_dependents();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * R;  // first batch row of this cluster
  const int B = p.B, K = p.K, C = p.C, n_x = p.n_x, n_in = p.n_in;

  // This lane: channel cj, column slice sl; after the reduce-scatter it holds gate g.
  const int cj = lane >> 3;
  const int sl = lane & 7;
  const int g = (lane >> 1) & 3;
  const int ch = kFwdChanPerCta * rank + 4 * warp + cj;

  // Per-lane addresses, computed once.
  //   X of this lane's (channel, gate g) -- written in place into H / cache by the
  //   projection -- for row row0 + r of step t: xp + t * xstep + r * xrow;
  //   the value this lane stores (lanes sl < 4: H, ff1, ff2, gate) likewise with sl for g.
  const int chc = ch < C ? ch : 0;  // padded channels read a valid location
  const size_t xrow = (g == 0) ? static_cast<size_t>(C) : 3ull * C;
  const size_t srow = (sl == 0) ? static_cast<size_t>(C) : 3ull * C;
  const float* xp = ((g == 0) ? p.xH : p.xcache + static_cast<size_t>(g - 1) * C) + chc +
                    static_cast<size_t>(row0) * xrow;
  // Output of this lane: element offset `so` in H (sl == 0) or in the cache (ff1, ff2, gate),
  // fp32 or bf16.
  const bool to_h = sl == 0;
  size_t so = static_cast<size_t>(to_h ? 0 : sl > 0 && sl < 4 ? sl - 1 : 0) * C + chc +
              static_cast<size_t>(row0) * srow;
  constexpr bool obf = BF;
  const float* tsp = p.ts + row0;
  const size_t xstep = static_cast<size_t>(B) * xrow, sstep = static_cast<size_t>(B) * srow;
  bool xok[R], sok[R], rok[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rok[r] = row0 + r < B;
    xok[r] = rok[r] && ch < C;
    sok[r] = xok[r] && sl < 4;
  }

  // X and ts of the step whose X row starts at xs (ts at tss), for every row of the group.
  auto load_step = [&](const float* xs, const float* tss, float (&xv)[R], float (&tv)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xv[r] = xok[r] ? __ldcg(xs + r * xrow) : 0.f;
      tv[r] = rok[r] ? __ldg(tss + r) : 0.f;
    }
  };

  // h0 of this CTA's rows (element e = tid + 256 i of the R x C block), loaded now and written
  // into the h buffer once the W staging area is free again.
  constexpr int kH0 = (R * S::CHP + kRecThreads - 1) / kRecThreads;
  float h0v[kH0];
#pragma unroll
  for (int i = 0; i < kH0; ++i) {
    const int e = tid + i * kRecThreads, r = e / S::CHP, j = e % S::CHP;
    h0v[i] = (e < R * S::CHP && row0 + r < B && j < C)
                 ? __ldg(p.h0 + static_cast<size_t>(row0 + r) * C + j) : 0.f;
  }

  // W_h rows of the CTA's channels, staged coalesced as [4 gates x 32 channels][WP] (the whole
  // shared-memory area is free before the K-loop), then this lane's 4 x HS block to registers.
  // The loads of a chunk are all issued before its stores, and the first chunk is in flight
  // together with h0 and the step-0 loads below.
  float2 wh[4][S::HS / 2];  // consecutive h inputs paired for the packed FMA
  float xc[R], tc[R];  // X and ts of the current step
  {
    float* wst = smem;
    constexpr int kPerThread = 4 * kFwdChanPerCta * S::CHP / kRecThreads;
    constexpr int kChunk = kPerThread < 64 ? kPerThread : 64;
    for (int i0 = 0; i0 < kPerThread; i0 += kChunk) {
      float v[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const int e = (i0 + i) * kRecThreads + tid;
        const int lrow = e / S::CHP, col = e % S::CHP;
        const int gg = lrow / kFwdChanPerCta, c = kFwdChanPerCta * rank + lrow % kFwdChanPerCta;
        v[i] = (c < C && col < C) ? __ldg(p.W + (static_cast<size_t>(gg) * C + c) * n_in + n_x + col)
                                  : 0.f;
      }
      if (i0 == 0) {
        // X comes from the projection kernel: wait for it (a no-op unless this launch is a
        // dependent one), then start the step-0 loads.
        grid_dep_wait();
        load_step(xp, tsp, xc, tc);
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const int e = (i0 + i) * kRecThreads + tid;
        wst[(e / S::CHP) * S::WP + e % S::CHP] = v[i];
      }
    }
    __syncthreads();
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
      const float* src = wst + (gg * kFwdChanPerCta + 4 * warp + cj) * S::WP + sl * S::HS;
#pragma unroll
      for (int c = 0; c < S::HS; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + c);
        wh[gg][c / 2] = make_float2(v.x, v.y);
        wh[gg][c / 2 + 1] = make_float2(v.z, v.w);
      }
    }
    __syncthreads();
  }

  // ---- prologue ----
  const uint32_t bar0 = smem_addr(&bars[0]);  // bars[s] lives at bar0 + 8 s
  const uint32_t tx_bytes = static_cast<uint32_t>(CS * R * kFwdChanPerCta * 4);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    fence_mbar_init_cluster();
  }
  for (int e = tid; e < 2 * R * S::HROW; e += kRecThreads) smem[e] = 0.f;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kH0; ++i) {
    const int e = tid + i * kRecThreads;
    if (e < R * S::CHP) hbuf[(e / S::CHP) * S::HROW + hpos<CS>(e % S::CHP)] = h0v[i];
  }
  // Step t consumes h_{t-1} through bars[t & 1]; arm the first two consumers (t = 1, 2).
  if (tid == 0) {
    if (K >= 2) mbar_arrive_expect_tx(bar0 + 8u, tx_bytes);
    if (K >= 3) mbar_arrive_expect_tx(bar0, tx_bytes);
  }
  __syncthreads();     // h0 visible to every warp
  cluster_sync_all();  // barrier inits and buffers ready cluster-wide

  // Pushes of the new h: lane q < CS writes the warp's four channels into CTA q's buffer.
  // Remote addresses of buffer 0 / row 0; buffer d, row r is (d * R + r) * HROW floats on.
  const bool pushes = lane < CS;
  const uint32_t push0 =
      pushes ? map_to_rank(smem_addr(hbuf + hpos<CS>(kFwdChanPerCta * rank + 4 * warp)), lane)
             : 0u;
  const uint32_t rbar0 = pushes ? map_to_rank(bar0, lane) : 0u;

  const float* xnext = xp + xstep;  // X and ts of step t + 1
  const float* tsnext = tsp + B;
  uint32_t phase = 0;  // bit s: parity of the next phase of bars[s] to wait for
  // One step: X and ts of step t in (xcur, tcur), those of step t + 1 loaded into (xn, tn).
  // Two calls per loop iteration with the arrays swapped: no register copies of pending loads.
  auto body = [&](int t, float (&xcur)[R], float (&tcur)[R], float (&xn)[R],
                  float (&tn)[R]) -> bool {
    const int s = t & 1;
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
      if (!ok) return false;
      if (tid == 0 && t + 2 <= K - 1) mbar_arrive_expect_tx(bar0 + 8u * s, tx_bytes);
    }

    const float* hb = hbuf + s * R * S::HROW + sl * S::HSP;
    const uint32_t pdst = push0 + static_cast<uint32_t>((s ^ 1) * R * S::HROW * 4);
    const uint32_t pbar = rbar0 + 8u * (s ^ 1);
    const bool b2 = lane & 4, b1 = lane & 2;
    const int base = lane & 24;
    // The rows are independent within a step, so the step runs in phases over all R rows
    // (products, then activations, then pushes and stores): the rows' latency chains overlap,
    // and no asynchronous push sits between one row's shared loads and the next row's.
    float P[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float2 hv[S::HS / 2];
      lds_pairs<S::HS>(hb + r * S::HROW, hv);
      float2 a2[4];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) a2[gg] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < S::HS / 2; ++c)
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) a2[gg] = fma2(wh[gg][c], hv[c], a2[gg]);
      float a[4];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) a[gg] = a2[gg].x + a2[gg].y;
      // Reduce-scatter over the 8 lanes of the channel: lane keeps gate (lane >> 1) & 3.
      const float k0 = b2 ? a[2] : a[0], k1 = b2 ? a[3] : a[1];
      const float s0 = k0 + __shfl_xor_sync(0xffffffffu, b2 ? a[0] : a[2], 4);
      const float s1 = k1 + __shfl_xor_sync(0xffffffffu, b2 ? a[1] : a[3], 4);
      float acc = (b1 ? s1 : s0) + __shfl_xor_sync(0xffffffffu, b1 ? s0 : s1, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      P[r] = acc + xcur[r];
    }
    float hn[R], sv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      // Activations: lanes of gate 0 / 1 evaluate tanh(P) = 2 sigmoid(2P) - 1, lanes of gate
      // 2 the time gate sigmoid(P_ta ts + P_tb) (P_tb from the gate-3 lane two lanes up).
      const float P_tb = __shfl_sync(0xffffffffu, P[r], (lane + 2) & 31);
      const float x = (g < 2) ? 2.f * P[r] : fmaf(P[r], tcur[r], P_tb);
      const float sg = sigmoid_fast(x);
      const float y = (g < 2) ? fmaf(2.f, sg, -1.f) : sg;
      const float f1 = __shfl_sync(0xffffffffu, y, base + 0);
      const float f2 = __shfl_sync(0xffffffffu, y, base + 2);
      const float gt = __shfl_sync(0xffffffffu, y, base + 4);
      hn[r] = f1 * (1.f - gt) + gt * f2;
      sv[r] = (sl == 0) ? hn[r] : (sl == 1) ? f1 : (sl == 2 ? f2 : gt);
    }
    // The warp's four channels of each row, gathered for one 16-byte push per destination CTA.
    float4 hq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      hq[r].x = __shfl_sync(0xffffffffu, hn[r], 0);
      hq[r].y = __shfl_sync(0xffffffffu, hn[r], 8);
      hq[r].z = __shfl_sync(0xffffffffu, hn[r], 16);
      hq[r].w = __shfl_sync(0xffffffffu, hn[r], 24);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      st_async_v4_if(pushes && t + 1 < K, pdst + static_cast<uint32_t>(r * S::HROW * 4), hq[r].x,
                     hq[r].y, hq[r].z, hq[r].w, pbar);
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (sok[r]) {
        const size_t o = so + r * srow;
        if constexpr (obf)
          reinterpret_cast<__nv_bfloat16*>(to_h ? p.H : p.cache)[o] = __float2bfloat16_rn(sv[r]);
        else
          (to_h ? p.H : p.cache)[o] = sv[r];
      }
    so += sstep;
    return true;
  };
  float xb[R], tb[R];
  for (int t = 0; t < K; t += 2) {
    if (!body(t, xc, tc, xb, tb)) break;
    if (t + 1 < K && !body(t + 1, xb, tb, xc, tc)) break;
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
  // The bf16-output variant has the same launch bounds and shared memory, hence the same
  // occupancy: both get the attributes, the fp32 one is measured.
  auto* kern = cfc_fwd_kernel<CS, R, false>;
  for (auto* k : {cfc_fwd_kernel<CS, R, false>, cfc_fwd_kernel<CS, R, true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
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
cudaError_t launch_k(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3(n_clusters * CS, 1, 1);
  c.block = dim3(kRecThreads, 1, 1);
  c.smem = smem;
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(CS, 1, 1);
  return p.out_bf16 ? launch(c, cfc_fwd_kernel<CS, R, true>, p)
                    : launch(c, cfc_fwd_kernel<CS, R, false>, p);
}

template <int CS>
cudaError_t prepare_cs(int R, size_t smem, int* max_active) {
  switch (R) {
    case 1: return prepare_k<CS, 1>(smem, max_active);
    case 2: return prepare_k<CS, 2>(smem, max_active);
    case 4: return prepare_k<CS, 4>(smem, max_active);
    case 8: return prepare_k<CS, 8>(smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

template <int CS>
cudaError_t launch_cs(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
                      bool pdl) {
  switch (p.R) {
    case 1: return launch_k<CS, 1>(p, n_clusters, smem, s, pdl);
    case 2: return launch_k<CS, 2>(p, n_clusters, smem, s, pdl);
    case 4: return launch_k<CS, 4>(p, n_clusters, smem, s, pdl);
    case 8: return launch_k<CS, 8>(p, n_clusters, smem, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t fwd_smem_bytes(int R, int CS) {
  const size_t hs = 4ull * CS;
  const size_t hsp = ((hs / 4) % 2 == 0) ? hs + 4 : hs;
  const size_t loop = sizeof(float) * 2ull * R * 8 * hsp + 2 * sizeof(uint64_t) + 16;
  // The prologue stages the CTA's W_h block ([4 x 32][32 CS + 4] floats) in the same area.
  const size_t stage = sizeof(float) * 4ull * kFwdChanPerCta * (kFwdChanPerCta * CS + 4);
  return loop > stage ? loop : stage;
}

cudaError_t fwd_prepare(int CS, int R, size_t smem, int* max_active) {
  switch (CS) {
    case 1: return prepare_cs<1>(R, smem, max_active);
    case 2: return prepare_cs<2>(R, smem, max_active);
    case 4: return prepare_cs<4>(R, smem, max_active);
    case 8: return prepare_cs<8>(R, smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t fwd_launch(const FwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
                       bool pdl) {
  switch (p.CS) {
    case 1: return launch_cs<1>(p, n_clusters, smem, s, pdl);
    case 2: return launch_cs<2>(p, n_clusters, smem, s, pdl);
    case 4: return launch_cs<4>(p, n_clusters, smem, s, pdl);
    case 8: return launch_cs<8>(p, n_clusters, smem, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cfc
