// cfc_bwd_tc.cu -- the BPTT recurrence with each step's contraction on the 5th-generation
// tensor cores, for large batches.
//
// The reverse-time recurrence of page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor" (sections "Problem" and "Per-Kernel Breakdown": dh = dH + delta, the gate
// gradients, then delta = W_h^T d_pre for the step before) is, for many batch rows at once, one
// contraction per step: [rows x 4C] d_pre times [4C x C] W_h.  Rows are independent, so a CTA
// owns 128 batch rows outright and no data crosses CTAs:
//   tensor memory  two fp32 accumulators [128 rows (lanes) x C channels]: delta[t+1], read by
//                  the epilogue, and delta[t], being accumulated (they swap every step);
//   shared memory  as many stages as fit (3 at C = 256, 4 at C = 128), each one 32-deep chunk
//                  of the reduction: the d_pre chunk [128 rows x 32 gate rows] (A) and the
//                  W_h^T chunk [C x 32 gate rows] (B), both in three bf16 terms in the
//                  non-swizzled K-major layout.
// The reduction index runs channel-major (k = 4 c + g), so a chunk is 8 channels x 4 gates.
// Eight epilogue warps turn delta[t+1] plus dH and the cache into d_pre chunk by chunk, the two
// warps of a tensor-memory lane quarter taking alternate chunks (one row and 8 channels per
// thread, so global accesses are whole 32-byte sectors), and write d_pre to global memory for
// the weight gradients; one thread streams the W_h^T chunks
// from a pre-split copy in global memory; one thread issues the MMAs of each chunk as both
// operands land.  Precision: both operands are split into three bf16 terms (x = hi + mid + lo,
// all 24 significand bits; bf16 keeps fp32's range, as d_pre has no bound), and the product
// keeps hi*hi + hi*mid + mid*hi + hi*lo + lo*hi + mid*mid with fp32 accumulation.
// Every wait is bounded; a timeout is recorded in the status word and every role stops.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kBM = 128;                          // batch rows per CTA (MMA M)
constexpr int kBK = 32;                           // reduction entries per chunk
constexpr int kBEpiWarps = 8;                     // two per tensor-memory lane quarter
constexpr int kBThreads = (kBEpiWarps + 1) * 32;  // + one control warp
constexpr int kBTerms = 3;

template <int C>
struct BtShape {
  static constexpr int NCH = 4 * C / kBK;         // chunks per step
  static constexpr int A_TERM = kBM * kBK * 2;    // bytes of one bf16 term of a d_pre chunk
  static constexpr int B_TERM = C * kBK * 2;      // bytes of one bf16 term of a W_h^T chunk
  static constexpr int STAGE = kBTerms * (A_TERM + B_TERM);
  // Stages: as many as fit beside the barriers in 227 KB, at most 4.
  static constexpr int NST_FIT = (227 * 1024 - 512) / STAGE;
  static constexpr int NST = NST_FIT < 4 ? NST_FIT : 4;
  static constexpr int USED = NST * STAGE + (3 * NST + 1) * 8 + 16 + 128;
  // At least half an SM's shared memory: each CTA takes all 512 tensor-memory columns.
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
  static constexpr size_t SPLIT = static_cast<size_t>(NCH) * kBTerms * B_TERM;
};

struct Split3 {
  __nv_bfloat16 t[3];
};
__device__ __forceinline__ Split3 split3(float x) {
  Split3 s;
  s.t[0] = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(s.t[0]);
  s.t[1] = __float2bfloat16_rn(r1);
  s.t[2] = __float2bfloat16_rn(r1 - __bfloat162float(s.t[1]));
  return s;
}
__device__ __forceinline__ uint32_t pack_bf2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// Byte offset of (row n, k) in a K-major, non-swizzled operand of `rows` rows:
// [k / 8][n / 8][n % 8][k % 8].
__device__ __forceinline__ uint32_t kmajor_offset(int n, int k, int rows) {
  return static_cast<uint32_t>(((k >> 3) * (rows >> 3) + (n >> 3)) * 128 + (n & 7) * 16 +
                               (k & 7) * 2);
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version; layout type 0 (no swizzle)
  return d;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 32-byte global accesses (whole sectors; the address must be 32-byte aligned).
__device__ __forceinline__ void ld_global_v8(const float* a, float (&v)[8]) {
  asm volatile("ld.global.cg.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(a));
}
__device__ __forceinline__ void st_global_v8(float* a, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(a), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// Bulk copy global -> this CTA's shared memory, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// W_h^T in the streamed layout: chunk kc, term tm, then [C x 32] K-major, where reduction
// entry k of chunk kc is gate row (g, c) with 4 c + g = 32 kc + k, and row n is channel n:
// the value is W[g][c][n_x + n].
template <int C>
__global__ void bwd_tc_split_kernel(const float* __restrict__ W, int n_x, int n_in,
                                    uint8_t* __restrict__ out) {
  using S = BtShape<C>;
  grid_dep_launch_dependents();
  // Completes only after the previous kernel of the stream has, so a dependent of this kernel
  // may read that kernel's outputs too.
  grid_dep_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= S::NCH * kBK * C) return;
  const int kc = idx / (kBK * C), rem = idx - kc * (kBK * C);
  const int k = rem / C, n = rem - k * C;
  const int j = kBK * kc + k, c = j >> 2, g = j & 3;
  const Split3 sp = split3(__ldg(W + (static_cast<size_t>(g) * C + c) * n_in + n_x + n));
  const uint32_t off = kmajor_offset(n, k, C);
#pragma unroll
  for (int tm = 0; tm < kBTerms; ++tm)
    *reinterpret_cast<__nv_bfloat16*>(out + (static_cast<size_t>(kc) * kBTerms + tm) *
                                                S::B_TERM + off) = sp.t[tm];
}

template <int C>
__global__ void __launch_bounds__(kBThreads, 1) cfc_bwd_tc_kernel(const BwdParams p) {
  using S = BtShape<C>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* sm = smem_raw + ((128u - (raw & 127u)) & 127u);
  constexpr int NST = S::NST;
  static_assert(NST >= 2, "two stages at least");
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + NST * S::STAGE);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * NST + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kBM;
  const int B = p.B, K = p.K;
  const uint32_t fa0 = smem_addr(&bars[0]);              // full_a[s]: d_pre chunk written
  const uint32_t fb0 = smem_addr(&bars[NST]);            // full_b[s]: W_h^T chunk landed
  const uint32_t em0 = smem_addr(&bars[2 * NST]);        // empty[s]: chunk's MMAs done
  const uint32_t done_bar = smem_addr(&bars[3 * NST]);   // a step's delta complete
  const uint32_t sm0 = smem_addr(sm);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(fa0 + 8u * s, kBEpiWarps * 32 / 2);  // a chunk is written by one warp group
      mbar_init(fb0 + 8u * s, 1);
      mbar_init(em0 + 8u * s, 1);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init_cluster();
  }
  // dH, the cache and the pre-split W_h^T come from earlier kernels; tensor memory is taken
  // only after they have finished, so this kernel never waits for columns they hold.
  // Dependents are released only after this wait: the operand build that follows reads the
  // forward's H without waiting for this kernel.
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (warp == kBEpiWarps) {
    tmem_alloc(smem_addr(tslot), 512);
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kBEpiWarps) {
    if (lane == 0) {
      // ---- MMA issuer: delta[t] (accumulator n & 1) += d_pre chunk x W_h^T chunk ----
      const uint32_t idesc = umma_idesc_bf16(kBM, C);
      constexpr uint32_t kLboA = (kBM / 8) * 128, kLboB = (C / 8) * 128;
      bool ok = true;
      int commits = 0;  // phases of done_bar this thread has committed
      for (int n = 0; n < K && ok; ++n) {
        const uint32_t dcur = tmem + static_cast<uint32_t>((n & 1) * C);
        uint32_t acc = 0;
        for (int kc = 0; kc < S::NCH; ++kc) {
          const int i = n * S::NCH + kc, s = i % NST;
          const uint32_t ph = (i / NST) & 1;
          ok = mbar_wait_bounded_cta(fa0 + 8u * s, ph, p.status) &&
               mbar_wait_bounded_cta(fb0 + 8u * s, ph, p.status);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t st = sm0 + s * S::STAGE;
          const uint64_t a0 = desc_kmajor(st, kLboA, 128);
          const uint64_t b0 = desc_kmajor(st + kBTerms * S::A_TERM, kLboB, 128);
#pragma unroll
          for (int s2 = 0; s2 < kBK / 16; ++s2) {  // 16-deep steps: k-cores 2 s2, 2 s2 + 1
            const uint64_t a = a0 + static_cast<uint64_t>((2 * s2 * kLboA) >> 4);
            const uint64_t b = b0 + static_cast<uint64_t>((2 * s2 * kLboB) >> 4);
            constexpr uint64_t ta = S::A_TERM >> 4, tb = S::B_TERM >> 4;
            // (A term, B term): hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid
            umma_bf16(dcur, a, b, idesc, acc);
            acc = 1;
            umma_bf16(dcur, a, b + tb, idesc, 1);
            umma_bf16(dcur, a + ta, b, idesc, 1);
            umma_bf16(dcur, a, b + 2 * tb, idesc, 1);
            umma_bf16(dcur, a + 2 * ta, b, idesc, 1);
            umma_bf16(dcur, a + ta, b + tb, idesc, 1);
          }
          umma_commit(em0 + 8u * s);  // the stage may be refilled once these MMAs are done
        }
        umma_commit(done_bar);
        ++commits;
      }
      // After an early stop the epilogue may leave before the last committed MMAs finish;
      // they depend on nothing outside this CTA, so wait for them before tensor memory is
      // freed.
      if (!ok && commits > 0) (void)mbar_wait_bounded_cta(done_bar, (commits - 1) & 1, p.status);
    } else if (lane == 1) {
      // ---- W_h^T chunk producer ----
      const uint8_t* wsplit = static_cast<const uint8_t*>(p.wsplit);
      bool ok = true;
      int issued = 0;  // chunks whose copies this thread has started
      for (int n = 0; n < K && ok; ++n) {
        for (int kc = 0; kc < S::NCH; ++kc) {
          const int i = n * S::NCH + kc, s = i % NST;
          if (i >= NST) ok = mbar_wait_bounded_cta(em0 + 8u * s, (i / NST - 1) & 1, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(fb0 + 8u * s, kBTerms * S::B_TERM);
          const uint32_t dst = sm0 + s * S::STAGE + kBTerms * S::A_TERM;
#pragma unroll
          for (int tm = 0; tm < kBTerms; ++tm)
            bulk_g2s(dst + tm * S::B_TERM,
                     wsplit + (static_cast<size_t>(kc) * kBTerms + tm) * S::B_TERM, S::B_TERM,
                     fb0 + 8u * s);
          ++issued;
        }
      }
      // After an early stop, no copy into this CTA's shared memory may still be in flight when
      // it exits: wait for the last chunks' copies to land (bulk copies from global memory
      // always complete).
      if (!ok)
        for (int i = issued > NST ? issued - NST : 0; i < issued; ++i)
          (void)mbar_wait_bounded_cta(fb0 + 8u * (i % NST), (i / NST) & 1, p.status);
    }
  } else {
    // ---- epilogue warps: row r = 32 q + lane.  Warp group hh (warps 4 hh .. 4 hh + 3, one per
    // lane quarter) takes the chunks kc with kc % 2 == hh and all 8 channels of each, so every
    // global access is a whole 32-byte sector. ----
    const int q = warp & 3, hh = warp >> 2;
    const int r = 32 * q + lane, b = row0 + r;
    const bool rok = b < B;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    // dH and ff1, ff2, gate of the chunk's 8 channels for this row at step t.
    auto load8 = [&](int t, int kc, float (&v)[4][8]) {
      if (rok) {
        const size_t tb = static_cast<size_t>(t) * B + b;
        const int c0 = 8 * kc;
        const float* cp = p.cache + tb * 3 * C + c0;
        ld_global_v8(p.dH + tb * C + c0, v[0]);
        ld_global_v8(cp, v[1]);
        ld_global_v8(cp + C, v[2]);
        ld_global_v8(cp + 2 * C, v[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int c = 0; c < 8; ++c) v[e][c] = 0.f;
      }
    };
    bool ok = true;
    float cur[4][8], nxt[4][8];
    load8(K - 1, hh, cur);
    for (int n = 0; n < K && ok; ++n) {
      const int t = K - 1 - n;
      if (n > 0) {
        ok = mbar_wait_bounded_cta(done_bar, (n - 1) & 1, p.status);  // delta[t+1] complete
        if (!ok) break;
        tc_fence_after_sync();
      }
      const uint32_t dprev = lane_base + static_cast<uint32_t>(((n + 1) & 1) * C);
      const float tsv = rok ? __ldg(p.ts + static_cast<size_t>(t) * B + b) : 0.f;
      float* dpp = p.d_pre + (static_cast<size_t>(t) * B + b) * 4 * C;
      for (int kc = hh; kc < S::NCH; kc += 2) {
        // This group's next chunk in flight while this one is worked on.
        if (kc + 2 < S::NCH) load8(t, kc + 2, nxt);
        else if (t > 0) load8(t - 1, hh, nxt);
        float dl[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (n > 0) tmem_ld8(dprev + 8 * kc, dl);
        float pv[4][8];  // [gate][channel]
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float dh = cur[0][c] + dl[c];
          const float f1 = cur[1][c], f2 = cur[2][c], g = cur[3][c];
          const float ds = dh * (f2 - f1) * g * (1.f - g);
          pv[0][c] = dh * (1.f - g) * (1.f - f1 * f1);
          pv[1][c] = dh * g * (1.f - f2 * f2);
          pv[2][c] = ds * tsv;
          pv[3][c] = ds;
        }
        if (rok) {
#pragma unroll
          for (int gg = 0; gg < 4; ++gg)
            st_global_v8(dpp + static_cast<size_t>(gg) * C + 8 * kc, pv[gg]);
        }
        // The chunk's operand terms, ready before the stage is free.  Entries k = 4 c + gg:
        // k-core kq holds channels 2 kq and 2 kq + 1.
        uint32_t w[4][kBTerms][4];
#pragma unroll
        for (int kq = 0; kq < 4; ++kq)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int c = 2 * kq + e2;
            const Split3 s0 = split3(pv[0][c]), s1 = split3(pv[1][c]);
            const Split3 s2 = split3(pv[2][c]), s3 = split3(pv[3][c]);
#pragma unroll
            for (int tm = 0; tm < kBTerms; ++tm) {
              w[kq][tm][2 * e2] = pack_bf2(s0.t[tm], s1.t[tm]);
              w[kq][tm][2 * e2 + 1] = pack_bf2(s2.t[tm], s3.t[tm]);
            }
          }
        const int i = n * S::NCH + kc, s = i % NST;
        if (i >= NST) {  // the stage's previous chunk consumed by its MMAs
          ok = mbar_wait_bounded_cta(em0 + 8u * s, (i / NST - 1) & 1, p.status);
          if (!ok) break;
        }
        uint8_t* ast = sm + s * S::STAGE;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const uint32_t off = kmajor_offset(r, 8 * kq, kBM);
#pragma unroll
          for (int tm = 0; tm < kBTerms; ++tm)
            *reinterpret_cast<uint4*>(ast + tm * S::A_TERM + off) =
                make_uint4(w[kq][tm][0], w[kq][tm][1], w[kq][tm][2], w[kq][tm][3]);
        }
        fence_proxy_async_smem();  // the chunk -> visible to the MMAs (async proxy)
        tc_fence_before_sync();    // this chunk's tensor-memory loads precede the arrive
        mbar_arrive(fa0 + 8u * s);
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int c = 0; c < 8; ++c) cur[e][c] = nxt[e][c];
      }
    }
    // dh0 = delta[0], in the accumulator of the last step.
    if (ok) ok = mbar_wait_bounded_cta(done_bar, (K - 1) & 1, p.status);
    tc_fence_after_sync();
    const uint32_t dlast = lane_base + static_cast<uint32_t>(((K - 1) & 1) * C);
    for (int c0 = hh * (C / 2); c0 < (hh + 1) * (C / 2); c0 += 16) {
      float v[16];
      tmem_ld16(dlast + c0, v);
      if (ok && rok) {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(p.dh0 + static_cast<size_t>(b) * C + c0 + e) =
              make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kBEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int C>
cudaError_t prepare_k(int* max_active) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const int smem = BtShape<C>::SMEM;
  if (smem > optin) {
    *max_active = 0;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(cfc_bwd_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_active, cfc_bwd_tc_kernel<C>,
                                                       kBThreads, smem);
}

template <int C>
cudaError_t split_k(const float* W, int n_x, void* wsplit, cudaStream_t s, bool pdl) {
  using S = BtShape<C>;
  const int total = S::NCH * kBK * C;
  LaunchCfg c;
  c.grid = dim3((total + 255) / 256, 1, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return launch(c, bwd_tc_split_kernel<C>, W, n_x, n_x + C, static_cast<uint8_t*>(wsplit));
}

template <int C>
cudaError_t launch_k(const BwdParams& p, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3((p.B + kBM - 1) / kBM, 1, 1);
  c.block = dim3(kBThreads, 1, 1);
  c.smem = BtShape<C>::SMEM;
  c.stream = s;
  c.pdl = pdl;
  return launch(c, cfc_bwd_tc_kernel<C>, p);
}

}  // namespace

bool bwd_tc_supported(int C) { return C == 128 || C == 256; }

size_t bwd_tc_split_bytes(int C) {
  if (C == 128) return BtShape<128>::SPLIT;
  if (C == 256) return BtShape<256>::SPLIT;
  return 0;
}

cudaError_t bwd_tc_split(const float* W, int C, int n_x, void* wsplit, cudaStream_t s,
                         bool pdl) {
  if (C == 128) return split_k<128>(W, n_x, wsplit, s, pdl);
  if (C == 256) return split_k<256>(W, n_x, wsplit, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_tc_prepare(int C, int* max_active_ctas) {
  if (C == 128) return prepare_k<128>(max_active_ctas);
  if (C == 256) return prepare_k<256>(max_active_ctas);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_tc_launch(const BwdParams& p, cudaStream_t s, bool pdl) {
  if (p.dplanes != 0) return cudaErrorInvalidValue;  // this recurrence writes fp32 d_pre only
  if (p.C == 128) return launch_k<128>(p, s, pdl);
  if (p.C == 256) return launch_k<256>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace cfc
