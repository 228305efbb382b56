// cfc_bwd_ks.cu -- the BPTT recurrence for large batches, with each step's contraction split
// along its reduction index over a thread-block cluster.
//
// The reverse-time recurrence of page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor" (sections "Problem" and "Per-Kernel Breakdown": dh = dH + delta, the gate
// gradients, then delta = W_h^T d_pre for the step before) is, for many batch rows at once, one
// contraction per step: [rows x 4C] d_pre times [4C x C] W_h.  A cluster of C / 32 CTAs serves
// 128 batch rows; CTA j owns channels 32 j .. 32 j + 31, i.e. the 128 reduction entries
// k = 4 c + g of those channels (g the gate).  Per step, CTA j:
//   1. multiplies its own d_pre slice (A: [128 rows x 128 k], three bf16 terms, kept in tensor
//      memory, where the same CTA wrote it) by its slice of W_h^T (B: [C x 128 k], streamed
//      from a pre-split copy in 32-deep chunks): a partial delta [128 rows x C] in tensor
//      memory, six MMAs per 16-deep step (hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid);
//   2. reduce-scatters the partial deltas over the cluster: the 32 columns of channel block i go
//      to CTA i (st.async into its receive slot j), and every CTA sums the C / 32 slots of its
//      own block in rank order (a fixed order: bitwise reproducible);
//   3. forms dh = dH + delta and the four gate gradients of its 32 channels for each row,
//      writes them to global memory (fp32 d_pre, for the weight gradients) and writes their
//      three bf16 terms into tensor memory as the next step's A.
// So 128 rows keep C / 32 SMs busy instead of one, each doing 1 / (C / 32) of the MMAs.  The
// last exchange gives dh0.
//
// Roles (288 threads): eight epilogue warps, two per tensor-memory lane quarter (row r = 32 q +
// lane; warp q + 4 h takes channels 16 h .. 16 h + 15 of the CTA's 32 and column half h of the
// drain); control warp lane 0 issues the MMAs, lane 1 streams the W_h^T chunks.  Every wait is
// bounded; a timeout is recorded in the status word, and all CTAs leave through one final
// cluster barrier, so none exits while another may still write into its shared memory.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kRows = 128;              // batch rows per cluster (MMA M, tensor-memory lanes)
constexpr int kChan = 32;               // channels per CTA
constexpr int kSlice = 4 * kChan;       // reduction entries per CTA
constexpr int kKc = 32;                 // reduction entries per streamed W_h^T chunk
constexpr int kChunks = kSlice / kKc;   // chunks per step
constexpr int kTerms = 3;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (kEpiWarps + 1) * 32;
constexpr int kWStages = 2;
constexpr uint32_t kACols = kSlice / 2;  // tensor-memory columns of one A term (bf16 pairs)
constexpr int kEpiBar = 1;               // named barrier of the epilogue warps

template <int C>
struct KsShape {
  static constexpr int CS = C / kChan;            // CTAs per cluster
  static constexpr int B_TERM = C * kKc * 2;      // one bf16 term of a W_h^T chunk
  static constexpr int WSTAGE = kTerms * B_TERM;
  static constexpr int SLOT = kRows * kChan * 4;  // one sender's block: 128 rows x 32 fp32
  static constexpr int RECV = CS * SLOT;
  static constexpr int NBARS = 2 * kWStages + 4;
  static constexpr int USED = kWStages * WSTAGE + RECV + NBARS * 8 + 16 + 1024;
  // More than half an SM: each CTA takes all 512 tensor-memory columns.
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
  static constexpr uint32_t ACOL0 = C;            // A terms follow the partial delta
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

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version; no swizzle
  return d;
}

// D (tensor memory) += A (tensor memory) * B (shared memory descriptor), bf16, fp32 accumulate.
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
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

__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Named barrier over `n` threads that returns the OR of `pred` over them (so the epilogue
// warps take every stop decision together and never leave one another at a barrier).
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// 16 consecutive floats at a 16-byte-aligned global address.
__device__ __forceinline__ void ld16(const float* a, float (&v)[16]) {
  const float4* p = reinterpret_cast<const float4*>(a);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 q = __ldcg(p + i);
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
}
__device__ __forceinline__ void st16(float* a, const float (&v)[16]) {
  float4* p = reinterpret_cast<float4*>(a);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int C>
__global__ void __launch_bounds__(kThreads, 1) cfc_bwd_ks_kernel(const BwdParams p) {
  using S = KsShape<C>;
  constexpr int CS = S::CS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t ws0 = smem_addr(sm);                             // W_h^T stages
  float* recv = reinterpret_cast<float*>(sm + kWStages * S::WSTAGE);  // [CS][128][32], swizzled
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kWStages * S::WSTAGE + S::RECV);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + S::NBARS);
  const uint32_t wfull0 = smem_addr(&bars[0]);              // W stage landed
  const uint32_t wempty0 = smem_addr(&bars[kWStages]);      // W stage's MMAs done
  const uint32_t a_ready = smem_addr(&bars[2 * kWStages]);  // next A written (256 arrivals)
  const uint32_t mma_done = smem_addr(&bars[2 * kWStages + 1]);
  const uint32_t recv_full = smem_addr(&bars[2 * kWStages + 2]);  // all CS blocks received
  const uint32_t free_bar = smem_addr(&bars[2 * kWStages + 3]);   // every CTA read its blocks

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int row0 = static_cast<int>(cluster_id_x()) * kRows;
  const int B = p.B, K = p.K;

  if (tid == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(wfull0 + 8u * s, 1);
      mbar_init(wempty0 + 8u * s, 1);
    }
    mbar_init(a_ready, kEpiWarps * 32);
    mbar_init(mma_done, 1);
    mbar_init(recv_full, 1);
    mbar_init(free_bar, CS);
    fence_mbar_init_cluster();
  }
  // dH, the cache and the pre-split W_h^T come from earlier kernels.  Tensor memory is taken
  // only after they have finished; dependents are released only after this wait (the operand
  // build that follows reads the forward's H without waiting for this kernel).
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (warp == kEpiWarps) {
    tmem_alloc(smem_addr(tslot), 512);
    tc_fence_before_sync();
  }
  if (tid == 0) mbar_arrive_expect_tx(recv_full, CS * S::SLOT);  // the first exchange
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  cluster_sync_all();  // every CTA's barriers initialised before any remote arrive or store

  if (warp == kEpiWarps) {
    if (lane == 0) {
      // ---- MMA issuer: step n (1 .. K) multiplies the A written in step n - 1 ----
      const uint32_t idesc = umma_idesc_bf16(kRows, C);
      constexpr uint32_t kLboB = (C / 8) * 128;
      bool ok = true;
      int commits = 0;
      for (int n = 1; n <= K && ok; ++n) {
        ok = mbar_wait_bounded_cta(a_ready, (n - 1) & 1, p.status);
        if (!ok) break;
        tc_fence_after_sync();
        for (int kc = 0; kc < kChunks; ++kc) {
          const int ci = (n - 1) * kChunks + kc, s = ci % kWStages;
          ok = mbar_wait_bounded_cta(wfull0 + 8u * s, (ci / kWStages) & 1, p.status);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t b0 = desc_kmajor(ws0 + s * S::WSTAGE, kLboB, 128);
#pragma unroll
          for (int s2 = 0; s2 < kKc / 16; ++s2) {
            const int ks = 2 * kc + s2;  // 16-deep step within the CTA's 128 entries
            const uint32_t a = tmem + S::ACOL0 + 8 * ks;
            const uint64_t b = b0 + static_cast<uint64_t>((2 * s2 * kLboB) >> 4);
            constexpr uint64_t tb = S::B_TERM >> 4;
            const uint32_t first = (kc == 0 && s2 == 0) ? 0u : 1u;
            // (A term, B term): hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid
            umma_tmem_a(tmem, a, b, idesc, first);
            umma_tmem_a(tmem, a, b + tb, idesc, 1);
            umma_tmem_a(tmem, a + kACols, b, idesc, 1);
            umma_tmem_a(tmem, a, b + 2 * tb, idesc, 1);
            umma_tmem_a(tmem, a + 2 * kACols, b, idesc, 1);
            umma_tmem_a(tmem, a + kACols, b + tb, idesc, 1);
          }
          umma_commit(wempty0 + 8u * s);
        }
        umma_commit(mma_done);
        ++commits;
      }
      // The MMAs committed here finish before tensor memory is freed, whatever else stopped.
      if (!ok && commits > 0) (void)mbar_wait_bounded_cta(mma_done, (commits - 1) & 1, p.status);
    } else if (lane == 1) {
      // ---- W_h^T chunk producer: this CTA's chunks 4 rank .. 4 rank + 3, once per step ----
      const uint8_t* wsplit = static_cast<const uint8_t*>(p.wsplit);
      bool ok = true;
      int issued = 0;
      for (int ci = 0; ci < K * kChunks && ok; ++ci) {
        const int s = ci % kWStages;
        if (ci >= kWStages)
          ok = mbar_wait_bounded_cta(wempty0 + 8u * s, (ci / kWStages - 1) & 1, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(wfull0 + 8u * s, S::WSTAGE);
        const int kc = kChunks * rank + ci % kChunks;
#pragma unroll
        for (int tm = 0; tm < kTerms; ++tm)
          bulk_g2s(ws0 + s * S::WSTAGE + tm * S::B_TERM,
                   wsplit + (static_cast<size_t>(kc) * kTerms + tm) * S::B_TERM, S::B_TERM,
                   wfull0 + 8u * s);
        ++issued;
      }
      if (!ok)
        for (int ci = issued > kWStages ? issued - kWStages : 0; ci < issued; ++ci)
          (void)mbar_wait_bounded_cta(wfull0 + 8u * (ci % kWStages), (ci / kWStages) & 1,
                                      p.status);
    }
  } else {
    // ---- epilogue warps ----
    const int q = warp & 3, h = warp >> 2;
    const int r = 32 * q + lane, b = row0 + r;
    const bool rok = b < B;
    const int ch0 = kChan * rank + 16 * h;  // this thread's 16 channels
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t recv_s = smem_addr(recv);
    // 16-byte chunk v (channels 4 v .. 4 v + 3) of this thread's row in sender block `slot` of
    // any CTA's receive buffer.  Chunk-major ([slot][v][row]): the 32 lanes of a warp (32
    // consecutive rows) store one contiguous 512-byte run per st.async and read one per load.
    auto recv_addr = [&](int slot, int v) {
      return recv_s + static_cast<uint32_t>(((slot * (kChan / 4) + v) * kRows + r) * 16);
    };
    float in[4][16];  // dH, ff1, ff2, gate of this row's 16 channels at step t
    auto load_inputs = [&](int t) {
      if (rok) {
        const size_t tb = static_cast<size_t>(t) * B + b;
        ld16(p.dH + tb * C + ch0, in[0]);
        const float* cp = p.cache + tb * 3 * C + ch0;
        ld16(cp, in[1]);
        ld16(cp + C, in[2]);
        ld16(cp + 2 * C, in[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int c = 0; c < 16; ++c) in[e][c] = 0.f;
      }
    };
    load_inputs(K - 1);  // step K-1 has no exchange before it
    bool ok = true;
    for (int n = 0; n <= K && ok; ++n) {
      const int t = K - 1 - n;
      float delta[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) delta[c] = 0.f;
      if (n > 0) {
        // ---- partial delta of this step -> the cluster; then this CTA's block summed ----
        ok = mbar_wait_bounded_cta(mma_done, (n - 1) & 1, p.status);
        if (ok && n >= 2) ok = mbar_wait_bounded_cluster(free_bar, (n - 2) & 1, p.status);
        if (bar_or(kEpiBar, kEpiWarps * 32, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int i = h * (CS / 2); i < (h + 1) * (CS / 2); ++i) {
          float v[32];
          tmem_ld32(lane_base + 32 * i, v);
          const uint32_t rbar = map_to_rank(recv_full, i);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            st_async_v4(map_to_rank(recv_addr(rank, c4), i), v[4 * c4], v[4 * c4 + 1],
                        v[4 * c4 + 2], v[4 * c4 + 3], rbar);
        }
        tc_fence_before_sync();  // the drain precedes the next step's MMAs (via a_ready)
        // This step's inputs: in flight while the other CTAs' blocks arrive (the last exchange,
        // n = K, only gives dh0 and reads no step's inputs).
        if (t >= 0) load_inputs(t);
        ok = mbar_wait_bounded_cluster(recv_full, (n - 1) & 1, p.status);
        if (bar_or(kEpiBar, kEpiWarps * 32, !ok)) {
          ok = false;
          break;
        }
#pragma unroll 1
        for (int i = 0; i < CS; ++i) {  // rank order: a fixed summation order
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const float4 x = *reinterpret_cast<const float4*>(
                recv + (recv_addr(i, 4 * h + v4) - recv_s) / 4);
            delta[4 * v4] += x.x; delta[4 * v4 + 1] += x.y;
            delta[4 * v4 + 2] += x.z; delta[4 * v4 + 3] += x.w;
          }
        }
        // Every epilogue thread has read this step's blocks: re-arm for the next exchange and
        // tell every CTA (itself included) that its block slots here are free again.
        asm volatile("bar.sync %0, %1;" ::"n"(kEpiBar), "n"(kEpiWarps * 32) : "memory");
        if (tid == 0) {
          if (n < K) mbar_arrive_expect_tx(recv_full, CS * S::SLOT);
          for (int i = 0; i < CS; ++i) mbar_arrive_remote(map_to_rank(free_bar, i));
        }
      }
      if (n == K) {  // the last exchange: delta = W_h^T d_pre[0] = dh0
        if (rok) {
          st16(p.dh0 + static_cast<size_t>(b) * C + ch0, delta);
        }
        break;
      }
      // ---- d_pre of step t for this row's 16 channels ----
      const float tsv = rok ? __ldg(p.ts + static_cast<size_t>(t) * B + b) : 0.f;
      float pv[4][16];  // [gate][channel]
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float dh = in[0][c] + delta[c];
        const float f1 = in[1][c], f2 = in[2][c], g = in[3][c];
        const float ds = dh * (f2 - f1) * g * (1.f - g);
        pv[0][c] = dh * (1.f - g) * (1.f - f1 * f1);
        pv[1][c] = dh * g * (1.f - f2 * f2);
        pv[2][c] = ds * tsv;
        pv[3][c] = ds;
      }
      if (rok) {
        float* dpp = p.d_pre + (static_cast<size_t>(t) * B + b) * 4 * C + ch0;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) st16(dpp + static_cast<size_t>(gg) * C, pv[gg]);
      }
      // The next A: entries k = 4 c + g of this row.  Tensor-memory column j of a term holds
      // entries 2 j and 2 j + 1, so local channel c' packs gates (0, 1) in column 2 c' and
      // (2, 3) in column 2 c' + 1.  Eight channels (16 columns) per store.
      if (n + 1 <= K) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[kTerms][16];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int cc = 8 * half + c;
            const Split3 s0 = split3(pv[0][cc]), s1 = split3(pv[1][cc]);
            const Split3 s2 = split3(pv[2][cc]), s3 = split3(pv[3][cc]);
#pragma unroll
            for (int tm = 0; tm < kTerms; ++tm) {
              w[tm][2 * c] = pack_bf2(s0.t[tm], s1.t[tm]);
              w[tm][2 * c + 1] = pack_bf2(s2.t[tm], s3.t[tm]);
            }
          }
#pragma unroll
          for (int tm = 0; tm < kTerms; ++tm)
            tmem_st16(lane_base + S::ACOL0 + tm * kACols + 32 * h + 16 * half, w[tm]);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before_sync();
        mbar_arrive(a_ready);
      }
    }
  }

  // Leave together: no CTA exits while another may still write into its shared memory.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == kEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int C>
cudaError_t prepare_k(int* max_active_clusters) {
  using S = KsShape<C>;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (S::SMEM > optin) {
    *max_active_clusters = 0;
    return cudaSuccess;
  }
  auto* kern = cfc_bwd_ks_kernel<C>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S::CS, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = S::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S::CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_active_clusters, kern, &cfg);
}

template <int C>
cudaError_t launch_k(const BwdParams& p, cudaStream_t s, bool pdl) {
  using S = KsShape<C>;
  LaunchCfg c;
  c.grid = dim3(((p.B + kRows - 1) / kRows) * S::CS, 1, 1);
  c.block = dim3(kThreads, 1, 1);
  c.smem = S::SMEM;
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(S::CS, 1, 1);
  return launch(c, cfc_bwd_ks_kernel<C>, p);
}

}  // namespace

cudaError_t bwd_ks_prepare(int C, int* max_active_clusters) {
  if (C == 128) return prepare_k<128>(max_active_clusters);
  if (C == 256) return prepare_k<256>(max_active_clusters);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_ks_launch(const BwdParams& p, cudaStream_t s, bool pdl) {
  if (p.dplanes != 0) return cudaErrorInvalidValue;  // writes fp32 d_pre only
  if (p.C == 128) return launch_k<128>(p, s, pdl);
  if (p.C == 256) return launch_k<256>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace cfc
