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
// Layout and schedule (every step is warp-local; no CTA-wide barrier inside the K-loop):
//   * a cluster of CS CTAs serves R batch rows; CTA `rank` owns channels [32*rank, 32*rank+32)
//     and warp w owns channels 32*rank + 4w + {0..3};
//   * every CTA pushes its 128 new d_pre values (32 channels x 4 gates) to every CTA with
//     st.async (one 16-byte push per channel and destination), so each CTA holds the whole
//     d_pre[t] vector (4C values) after one mbarrier wait;
//   * warp w keeps the four W_h^T columns of its channels in REGISTERS, lane l holding them
//     over the l-th thirty-second of the 4C gathered rows (4*CS rows), so every d_pre value
//     loaded from shared memory feeds four FMAs; a 6-shuffle reduce-scatter leaves delta of
//     channel cj in lanes 8cj .. 8cj+7, and the same warp forms dh, the four d_pre values of
//     each channel and the pushes.  The gathered vector is stored in thirty-two slices padded
//     to an odd number of 16-byte chunks, so the vector loads of a quarter-warp hit distinct
//     banks.  The summation order is fixed: bitwise reproducible;
//   * with 32 channels per CTA a cluster has C/32 CTAs: the 32x64x128 workload runs one CTA
//     per SM (measured on GB300, CTAs that share an SM slow every step of the chain);
//   * dH, ff1, ff2, gate and ts of step t-1 are loaded into registers during step t when the
//     cluster serves at most four rows (the row count is then a compile-time parameter); for
//     larger row groups they arrive two steps ahead through a cp.async ring (5 lanes per
//     channel copy, the warp reads after __syncwarp).  Either way no global-memory latency
//     sits on the serial chain;
//   * per-lane addresses are computed once; the K-loop advances pointers by a fixed stride and
//     uses predicated loads, stores and st.async;
//   * the W_h^T columns are read once, coalesced, into shared memory and from there into
//     registers (a direct load would fetch one 32-byte sector per 4-byte value).
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kWarps = kRecThreads / 32;
constexpr int kPre = 3;      // prefetch ring depth (copies run two steps ahead)
constexpr int kRowBlock = 4; // rows per phase block of the ring path (its row counts are multiples)
constexpr int kPreComp = 5;  // dH, ff1, ff2, gate, ts

// Lanes 8*cj + c (c < 5) copy component c of this warp's channel cj for step t.  A bf16 cache
// component is copied as the 4-byte pair of channels (ch & ~1, ch | 1) that holds it (C is even
// then), and the consumer takes its half (ring_value).
template <bool BF>
__device__ __forceinline__ void issue_pre(const BwdParams& p, float* pre, int t, int row0,
                                          int rank, int warp, int lane) {
  if (t < 0) return;
  const int cj = lane >> 3, c = lane & 7;
  if (c >= kPreComp) return;
  const int ch = kBwdChanPerCta * rank + 4 * warp + cj;
  if (ch >= p.C) return;
  for (int r = 0; r < p.R; ++r) {
    const int b = row0 + r;
    if (b >= p.B) break;
    const size_t tb = static_cast<size_t>(t) * p.B + b;
    const void* src =
        (c == 0)       ? static_cast<const void*>(p.dH + tb * p.C + ch)
        : (c == 4)     ? static_cast<const void*>(p.ts + tb)
        : BF           ? static_cast<const void*>(reinterpret_cast<const __nv_bfloat16*>(p.cache) +
                                                  (tb * 3 + (c - 1)) * p.C + (ch & ~1))
                       : static_cast<const void*>(p.cache + (tb * 3 + (c - 1)) * p.C + ch);
    float* dst = pre + ((((t % kPre) * p.R + r) * kWarps + warp) * 4 + cj) * kPreComp + c;
    cp_async_4(smem_addr(dst), src);
  }
}

template <int CS>
struct BwdShape {
  static constexpr int CHP = kBwdChanPerCta * CS;  // padded channel count
  static constexpr int NG = 4 * CHP;               // gathered d_pre values per row
  static constexpr int RS = NG / 32;               // rows per lane (= 4 * CS)
  // Slice pitch: vector loads of 8 consecutive lanes must cover distinct banks.
  static constexpr int RSP = (RS >= 4 && (RS / 4) % 2 == 0) ? RS + 4 : RS;
  static constexpr int GROW = 32 * RSP;         // gathered row in shared memory
};

template <int CS>
__device__ __forceinline__ int gpos(int gidx) {
  using S = BwdShape<CS>;
  return (gidx / S::RS) * S::RSP + (gidx % S::RS);
}

// delta for the four channels of this warp from this lane's slice of the gathered d_pre
// vector; lanes 8cj .. 8cj+7 return channel cj.
template <int RS>
__device__ __forceinline__ float gathered_delta(const float2 (&wt)[4][RS / 2], const float* dvp,
                                                int lane) {
  float2 a2[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) a2[c] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < RS; k += 4) {
    const float4 v = *reinterpret_cast<const float4*>(dvp + k);
    const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
#pragma unroll
    for (int c = 0; c < 4; ++c) a2[c] = fma2(wt[c][k / 2], lo, a2[c]);
#pragma unroll
    for (int c = 0; c < 4; ++c) a2[c] = fma2(wt[c][k / 2 + 1], hi, a2[c]);
  }
  float a[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) a[c] = a2[c].x + a2[c].y;
  // Reduce-scatter over the 32 lanes: xor 16 keeps channels {0,1} / {2,3}, xor 8 one channel,
  // then the eight lanes of a channel sum.
  const bool b16 = lane & 16, b8 = lane & 8;
  const float k0 = b16 ? a[2] : a[0], k1 = b16 ? a[3] : a[1];
  const float s0 = k0 + __shfl_xor_sync(0xffffffffu, b16 ? a[0] : a[2], 16);
  const float s1 = k1 + __shfl_xor_sync(0xffffffffu, b16 ? a[1] : a[3], 16);
  float d = (b8 ? s1 : s0) + __shfl_xor_sync(0xffffffffu, b8 ? s0 : s1, 8);
  d += __shfl_xor_sync(0xffffffffu, d, 4);
  d += __shfl_xor_sync(0xffffffffu, d, 2);
  d += __shfl_xor_sync(0xffffffffu, d, 1);
  return d;
}

// Prefetched inputs of one step for RT rows (register path): dH, ff1, ff2, gate, ts.  dHp,
// cp (cpb: the same element of a bf16 cache, read when BF) and tsp address row row0 of the
// step; row r is C, 3C and 1 elements further on.
template <int RT, bool BF>
__device__ __forceinline__ void load_step_regs(const float* dHp, const float* cp,
                                               const __nv_bfloat16* cpb, const float* tsp, int C,
                                               const bool (&rok)[RT],
                                               float (&v)[RT][kPreComp]) {
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const size_t o = static_cast<size_t>(r) * C;
    v[r][0] = rok[r] ? __ldcg(dHp + o) : 0.f;
    if constexpr (BF) {
      v[r][1] = rok[r] ? __bfloat162float(cpb[3 * o]) : 0.f;
      v[r][2] = rok[r] ? __bfloat162float(cpb[3 * o + C]) : 0.f;
      v[r][3] = rok[r] ? __bfloat162float(cpb[3 * o + 2 * C]) : 0.f;
    } else {
      v[r][1] = rok[r] ? __ldcg(cp + 3 * o) : 0.f;
      v[r][2] = rok[r] ? __ldcg(cp + 3 * o + C) : 0.f;
      v[r][3] = rok[r] ? __ldcg(cp + 3 * o + 2 * C) : 0.f;
    }
    v[r][4] = rok[r] ? __ldg(tsp + r) : 0.f;
  }
}

// A ring slot as the consumer's value: components 1-3 of a bf16 cache hold the channel pair
// (ch & ~1, ch | 1); bf16 -> fp32 puts the 16 bits in the upper half.
template <bool BF>
__device__ __forceinline__ float ring_value(float slot, int c, int ch) {
  if (!BF || c == 0 || c == 4) return slot;
  const uint32_t u = __float_as_uint(slot);
  return __uint_as_float((ch & 1) ? (u & 0xffff0000u) : (u << 16));
}

// RT = 1, 2, 4: rows per cluster fixed at compile time, inputs prefetched into registers.
// RT = 0: p.R rows (any count), inputs through the cp.async ring.
// BF: the cache holds bf16 elements (BwdParams::cache_bf16).
template <int CS, int RT, bool BF>
// Two CTAs per SM fit (128 registers) wherever the variant allows it without spilling, so a
// BPTT CTA launched as a dependent of the forward can stage its weights beside a running
// forward CTA.
__global__ void __launch_bounds__(kRecThreads, (CS >= 8 || (CS == 4 && (RT == 0 || RT == 4))) ? 1 : 2)
    cfc_bwd_kernel(const BwdParams p) {
  using S = BwdShape<CS>;
  extern __shared__ __align__(16) float smem[];
  const int R = RT > 0 ? RT : p.R;
  float* dg = smem;                      // [2][R][GROW]  d_pre[t+1] for step t in dg[t & 1]
  float* pre = dg + 2 * R * S::GROW;     // ring path: [kPre][R][8 warps][4][5]
  const int pre_floats = RT > 0 ? 0 : kPre * R * kWarps * 4 * kPreComp;
  uint64_t* bars = reinterpret_cast<uint64_t*>(pre + pre_floats);
  // Dependents are released only after this kernel's own dependency wait (below): the
  // operand build that follows reads the forward's H without waiting for this kernel.

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * R;
  const int B = p.B, K = p.K, C = p.C, n_x = p.n_x, n_in = p.n_in;

  const int cj = lane >> 3;        // channel of this 8-lane group
  const int gq = (lane >> 1) & 3;  // gate this lane's d_pre belongs to
  const int q = lane & 7;          // destination CTA of this lane's push
  const int ch = kBwdChanPerCta * rank + 4 * warp + cj;
  const int base = lane & 24;

  // Per-lane addresses, computed once: the K-loop only moves pointers by a fixed stride per
  // step and issues predicated loads and stores (no index arithmetic or divergent branches on
  // the serial chain).  Pointers address row row0 of step t.
  constexpr int RR = RT > 0 ? RT : 1;
  const int chc = ch < C ? ch : 0;  // padded channels address a valid location
  const size_t t_last = static_cast<size_t>(K - 1) * B + row0;
  const float* dHp = p.dH + t_last * C + chc;
  // The same cache element as fp32 (cp) or, BF, as bf16 (cpb); only one of them is used.
  const float* cp = BF ? nullptr : p.cache + t_last * 3 * C + chc;
  const __nv_bfloat16* cpb =
      BF ? reinterpret_cast<const __nv_bfloat16*>(p.cache) + t_last * 3 * C + chc : nullptr;
  const float* tsp = p.ts + t_last;
  float* dpp = p.d_pre + (t_last * 4 + gq) * C + chc;  // d_pre of this lane's gate
  const size_t bc = static_cast<size_t>(B) * C;
  bool rok[RR];
#pragma unroll
  for (int r = 0; r < RR; ++r) rok[r] = row0 + r < B;
  // fp32 output: one lane of each (channel, gate) pair stores d_pre.  bf16 operand rows (2 *
  // dpitch values per row): the even lane stores the hi term, the odd lane the lo term.
  const bool planes = p.dplanes > 0;
  const bool stores = ch < C && ((lane & 1) == 0 || p.dplanes == 2);
  const size_t prow = 2 * static_cast<size_t>(p.dpitch);  // bf16 values per operand row
  __nv_bfloat16* dqp = reinterpret_cast<__nv_bfloat16*>(p.d_pre) + t_last * prow +
                       ((lane & 1) ? p.dpitch : 0) + static_cast<size_t>(gq) * C + chc;

  // W_h^T columns of this warp's four channels over gathered rows [lane*RS, lane*RS + RS).
  // Gathered row q*128 + 4i + g is W row g*C + 32q + i.  Staged through shared memory as
  // [NG][33] (the whole smem area is free before the loop): consecutive threads read
  // consecutive channels of one W row, a chunk of loads in flight before any store.
  float2 wt[4][S::RS / 2];  // consecutive gathered rows paired for the packed FMA
  float cur[RR][kPreComp];  // register path: inputs of the current step
  {
    float* wtmp = smem;
    constexpr int kPitch = kBwdChanPerCta + 1;
    constexpr int kPerThread = S::NG * kBwdChanPerCta / kRecThreads;
    constexpr int kChunk = kPerThread < 64 ? kPerThread : 64;
    for (int i0 = 0; i0 < kPerThread; i0 += kChunk) {
      float v[kChunk];
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const int e = (i0 + i) * kRecThreads + tid;
        const int gidx = e / kBwdChanPerCta, jl = e % kBwdChanPerCta;
        const int chr = kBwdChanPerCta * (gidx / 128) + (gidx % 128) / 4;
        const int j = kBwdChanPerCta * rank + jl;
        v[i] = (chr < C && j < C)
                   ? __ldg(p.W + (static_cast<size_t>(gidx & 3) * C + chr) * n_in + n_x + j)
                   : 0.f;
      }
      if constexpr (RT > 0) {
        if (i0 == 0) {
          // dH and the forward cache may come from the previous kernel: wait for it (a no-op
          // unless this launch is a dependent one), then start the step K-1 loads, in flight
          // together with the first chunk of W_h^T.
          grid_dep_wait();
          grid_dep_launch_dependents();
          load_step_regs<RR, BF>(dHp, cp, cpb, tsp, C, rok, cur);
          dHp -= bc;
          if constexpr (BF) cpb -= 3 * bc; else cp -= 3 * bc;
          tsp -= B;
        }
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        const int e = (i0 + i) * kRecThreads + tid;
        wtmp[(e / kBwdChanPerCta) * kPitch + e % kBwdChanPerCta] = v[i];
      }
    }
    __syncthreads();
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int k = 0; k < S::RS; k += 2)
        wt[cc][k / 2] = make_float2(wtmp[(lane * S::RS + k) * kPitch + 4 * warp + cc],
                                    wtmp[(lane * S::RS + k + 1) * kPitch + 4 * warp + cc]);
    __syncthreads();
  }

  const uint32_t bar0 = smem_addr(&bars[0]);  // bars[s] lives at bar0 + 8 s
  const uint32_t tx_bytes = static_cast<uint32_t>(CS * R * 4 * kBwdChanPerCta * 4);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8u, 1);
    fence_mbar_init_cluster();
  }
  for (int e = tid; e < 2 * R * S::GROW; e += kRecThreads) dg[e] = 0.f;
  // Consumer c (the step that reads d_pre[c+1]; -1 is the dh0 epilogue) uses bars[c & 1].
  // Consumers run c = K-2 .. -1; arm the first two.
  if (tid == 0) {
    mbar_arrive_expect_tx(bar0 + 8u * ((K - 2) & 1), tx_bytes);
    if (K >= 2) mbar_arrive_expect_tx(bar0 + 8u * ((K - 3) & 1), tx_bytes);
  }
  // The four d_pre of channel cj go to slot rank*128 + 4*(4w + cj) of every CTA's gathered
  // vector; remote addresses of buffer 0 / row 0 (buffer d, row r: (d R + r) GROW floats on).
  const bool pushes = q < CS;
  const uint32_t push0 =
      pushes ? map_to_rank(smem_addr(dg + gpos<CS>(rank * 4 * kBwdChanPerCta + 4 * (4 * warp + cj))), q)
             : 0u;
  const uint32_t rbar0 = pushes ? map_to_rank(bar0, q) : 0u;

  if constexpr (RT == 0) {
    // The ring lives where the W_h^T staging was: start it only now.
    grid_dep_wait();
    grid_dep_launch_dependents();
    issue_pre<BF>(p, pre, K - 1, row0, rank, warp, lane);
    cp_async_commit();
    issue_pre<BF>(p, pre, K - 2, row0, rank, warp, lane);
    cp_async_commit();
  }
  cluster_sync_all();

  uint32_t phase = 0;
  bool ok = true;
  for (int t = K - 1; t >= 0; --t) {
    const int s = t & 1;
    float nxt[RR][kPreComp];
    if constexpr (RT > 0) {
      if (t >= 1) {  // step t - 1, used one step later
        load_step_regs<RR, BF>(dHp, cp, cpb, tsp, C, rok, nxt);
        dHp -= bc;
        if constexpr (BF) cpb -= 3 * bc; else cp -= 3 * bc;
        tsp -= B;
      }
    } else {
      // Ring: step t-2 goes into the slot step t+1 used; every lane of the warp has read it.
      __syncwarp();
      issue_pre<BF>(p, pre, t - 2, row0, rank, warp, lane);
      cp_async_commit();
    }

    if (t < K - 1) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded_cluster(bar0 + 8u * s, (phase >> s) & 1u, p.status));
      phase ^= (1u << s);
      if (!ok) break;
      if (tid == 0 && t - 2 >= -1) mbar_arrive_expect_tx(bar0 + 8u * s, tx_bytes);
    }
    if constexpr (RT == 0) {
      cp_async_wait<2>();  // the warp's copies for step t (groups t-1, t-2 may be pending)
      __syncwarp();
    }

    const float* pre_t = pre + ((t % kPre) * R * kWarps + warp) * 4 * kPreComp + cj * kPreComp;
    const uint32_t pdst = push0 + static_cast<uint32_t>((s ^ 1) * R * S::GROW * 4);
    const uint32_t pbar = rbar0 + 8u * (s ^ 1);
    // Rows are independent within a step: each block of RB rows runs in phases (products,
    // then gradients, then stores and pushes) so the rows' latency chains overlap and no
    // asynchronous push sits between one row's shared loads and the next row's.
    constexpr int RB = RT > 0 ? RT : kRowBlock;
#pragma unroll 1
    for (int r0 = 0; r0 < R; r0 += RB) {
      float delta[RB];
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
        delta[rb] = (t < K - 1) ? gathered_delta<S::RS>(
                                      wt, dg + (s * R + r0 + rb) * S::GROW + lane * S::RSP, lane)
                                : 0.f;
      float dpv[RB];
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        const int r = r0 + rb;
        const bool valid = row0 + r < B && ch < C;
        float v[kPreComp];  // dH, ff1, ff2, gate, ts of (t, b, ch)
#pragma unroll
        for (int c = 0; c < kPreComp; ++c)
          v[c] = RT > 0 ? cur[RT > 0 ? rb : 0][c]
                        : ring_value<BF>(pre_t[r * kWarps * 4 * kPreComp + c], c, ch);
        const float dh = v[0] + delta[rb];
        const float f1 = v[1], f2 = v[2], g = v[3];
        const float ds = dh * (f2 - f1) * g * (1.f - g);
        // This lane's gate, by selects (neighbouring lane pairs hold different gates, so a
        // branch here would split the warp four ways).
        const float p0 = dh * (1.f - g) * (1.f - f1 * f1);
        const float p1 = dh * g * (1.f - f2 * f2);
        const float p2 = ds * v[4];
        const float sel = (gq == 0) ? p0 : (gq == 1) ? p1 : (gq == 2) ? p2 : ds;
        dpv[rb] = valid ? sel : 0.f;
      }
      // The four gates of channel cj -> one 16-byte push to every CTA of the cluster.
      float4 dq[RB];
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        dq[rb].x = __shfl_sync(0xffffffffu, dpv[rb], base + 0);
        dq[rb].y = __shfl_sync(0xffffffffu, dpv[rb], base + 2);
        dq[rb].z = __shfl_sync(0xffffffffu, dpv[rb], base + 4);
        dq[rb].w = __shfl_sync(0xffffffffu, dpv[rb], base + 6);
      }
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
        st_async_v4_if(pushes, pdst + static_cast<uint32_t>((r0 + rb) * S::GROW * 4), dq[rb].x,
                       dq[rb].y, dq[rb].z, dq[rb].w, pbar);
      if (planes) {
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(dpv[rb]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(dpv[rb] - __bfloat162float(hi));
          if (stores && row0 + r0 + rb < B) dqp[static_cast<size_t>(r0 + rb) * prow] = (lane & 1) ? lo : hi;
        }
      } else {
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
          if (stores && row0 + r0 + rb < B) dpp[static_cast<size_t>(r0 + rb) * 4 * C] = dpv[rb];
      }
    }
    dpp -= 4 * bc;
    dqp -= static_cast<size_t>(B) * prow;
    if constexpr (RT > 0) {
      if (t >= 1) {
#pragma unroll
        for (int r = 0; r < RR; ++r)
#pragma unroll
          for (int c = 0; c < kPreComp; ++c) cur[r][c] = nxt[r][c];
      }
    }
  }

  // Epilogue: dh0 = W_h^T d_pre[0] (consumer -1 reads bars[1]).
  if (ok) {
    ok = __all_sync(0xffffffffu, mbar_wait_bounded_cluster(bar0 + 8u, (phase >> 1) & 1u, p.status));
    if (ok) {
      for (int r = 0; r < R; ++r) {
        const float delta =
            gathered_delta<S::RS>(wt, dg + (1 * R + r) * S::GROW + lane * S::RSP, lane);
        const int b = row0 + r;
        if ((lane & 7) == 0 && b < B && ch < C) p.dh0[static_cast<size_t>(b) * C + ch] = delta;
      }
    }
  }
  if constexpr (RT == 0) cp_async_wait<0>();
  cluster_sync_all();
}

template <int CS, int RT>
cudaError_t prepare_k(size_t smem, int* max_active) {
  // The attribute is a per-function maximum: set it to the device's opt-in limit once, so any
  // row grouping chosen later (from cached occupancy results) can launch.
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(optin)) {
    *max_active = 0;
    return cudaSuccess;
  }
  // The bf16-cache variant has the same launch bounds and shared memory, hence the same
  // occupancy: both get the attributes, the fp32 one is measured.
  auto* kern = cfc_bwd_kernel<CS, RT, false>;
  for (auto* k : {cfc_bwd_kernel<CS, RT, false>, cfc_bwd_kernel<CS, RT, true>}) {
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

template <int CS, int RT>
cudaError_t launch_k(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3(n_clusters * CS, 1, 1);
  c.block = dim3(kRecThreads, 1, 1);
  c.smem = smem;
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(CS, 1, 1);
  return p.cache_bf16 ? launch(c, cfc_bwd_kernel<CS, RT, true>, p)
                      : launch(c, cfc_bwd_kernel<CS, RT, false>, p);
}

// Row groups of 1, 2 or 4 use the register-prefetch kernels, larger ones the ring kernel.
int bwd_variant(int R) { return (R == 1 || R == 2 || R == 4) ? R : 0; }

template <int CS>
cudaError_t prepare_cs(int R, size_t smem, int* max_active) {
  switch (bwd_variant(R)) {
    case 1: return prepare_k<CS, 1>(smem, max_active);
    case 2: return prepare_k<CS, 2>(smem, max_active);
    case 4: return prepare_k<CS, 4>(smem, max_active);
    default: return prepare_k<CS, 0>(smem, max_active);
  }
}

template <int CS>
cudaError_t launch_cs(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
                      bool pdl) {
  switch (bwd_variant(p.R)) {
    case 1: return launch_k<CS, 1>(p, n_clusters, smem, s, pdl);
    case 2: return launch_k<CS, 2>(p, n_clusters, smem, s, pdl);
    case 4: return launch_k<CS, 4>(p, n_clusters, smem, s, pdl);
    default:
      // The ring kernel walks its rows in whole blocks.
      if (p.R % kRowBlock != 0) return cudaErrorInvalidValue;
      return launch_k<CS, 0>(p, n_clusters, smem, s, pdl);
  }
}

}  // namespace

size_t bwd_smem_bytes(int R, int CS) {
  const size_t RS = 4ull * CS;
  const size_t GROW = 32 * (((RS / 4) % 2 == 0) ? RS + 4 : RS);
  const size_t ring = bwd_variant(R) > 0 ? 0 : 1ull * kPre * R * kWarps * 4 * kPreComp;
  const size_t loop = sizeof(float) * (2ull * R * GROW + ring) + 2 * sizeof(uint64_t) + 16;
  // The prologue stages the CTA's W_h^T block ([4 * 32 CS][33] floats) in the same area.
  const size_t stage = sizeof(float) * 4ull * kBwdChanPerCta * CS * (kBwdChanPerCta + 1);
  return loop > stage ? loop : stage;
}

cudaError_t bwd_prepare(int CS, int R, size_t smem, int* max_active) {
  switch (CS) {
    case 1: return prepare_cs<1>(R, smem, max_active);
    case 2: return prepare_cs<2>(R, smem, max_active);
    case 4: return prepare_cs<4>(R, smem, max_active);
    case 8: return prepare_cs<8>(R, smem, max_active);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t bwd_launch(const BwdParams& p, int n_clusters, size_t smem, cudaStream_t s,
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
