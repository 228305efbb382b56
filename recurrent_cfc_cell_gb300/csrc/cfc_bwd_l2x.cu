// cfc_bwd_l2x.cu -- the BPTT recurrence for large batches: each step's contraction split along
// its reduction over a thread-block cluster, batch rows along the MMA's N side, the partial
// sums exchanged through L2.
//
// The reverse-time recurrence of page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor" (sections "Problem" and "Per-Kernel Breakdown": dh = dH + delta, the gate
// gradients, then delta = W_h^T d_pre for the step before) is, for many batch rows at once, one
// contraction per step: delta^T [C x rows] = W_h^T [C x 4C] times d_pre^T [4C x rows].
//
// A cluster of CS = C / 32 CTAs serves NR (128 or 144) batch rows; CTA `rank` owns channels
// 32 rank .. 32 rank + 31, i.e. the 128 reduction entries k = 4 c + g of those channels (g the
// gate).  Per step, CTA `rank`:
//   1. multiplies its slice of W_h^T (A: [C outputs x 128 k], stationary in shared memory) by
//      its own d_pre slice (B: [NR rows x 128 k], written into shared memory by the same CTA
//      the step before): a partial delta^T [C x NR] in tensor memory.  Both operands carry two
//      fp16 terms, x = hi + lo with hi = fp16(x), lo = fp16(x - hi) (22 significand bits), and
//      the product keeps hi*hi + hi*lo + lo*hi (three MMAs per 16-deep step; what is dropped is
//      below about 2^-21 of each product).  Every output row of W_h^T and every batch row of
//      d_pre is scaled by a power of two into [-2^15, 2^15) before the split, so nothing over-
//      or underflows fp16, and the partial is scaled back exactly when it is read out;
//   2. reduce-scatters the partials over the cluster through L2: the 32 outputs of channel
//      block i go to an exchange buffer in global memory, block (i, rank), and a remote
//      mbarrier arrive on CTA i says they are there; every CTA then sums the CS blocks of its
//      own channels in rank order (a fixed order: bitwise reproducible).  Tensor memory cannot
//      be read by another SM, and a shared-memory exchange of these blocks was slower than L2;
//   3. forms dh = dH + delta and the four gate gradients of its 32 channels for each row,
//      writes them to global memory for the weight gradients (fp32 d_pre, or straight in the
//      contraction's operand rows: bf16 hi and, with two planes, lo = bf16(x - hi)) and writes
//      their two fp16 terms into shared memory as the next step's B.
// The last exchange gives dh0.  15 clusters of 144 rows cover 2048 rows in one wave (GB300
// keeps at most 15 clusters of 8 CTAs resident).
//
// Roles (320 threads): nine epilogue warps (warp w < NR / 16 computes rows 16 w .. 16 w + 15,
// lane = channel pair c / 2 and row parity); warps 0 .. 7 also read the partial out of tensor
// memory (lane quarter w % 4; C = 256: output half w / 4, all rows; C = 128: row half w / 4);
// warp 9 lane 0 loads W_h^T and issues the MMAs.  Every wait is bounded; a timeout is recorded
// in the status word, and all CTAs leave through one final cluster barrier, so none exits while
// another may still arrive on its barriers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kChan = 32;                     // channels per CTA
constexpr int kSlice = 4 * kChan;             // reduction entries per CTA
constexpr int kKSteps = kSlice / 16;          // 16-deep MMA steps per term pair
constexpr int kDrainWarps = 8;
constexpr int kEpiWarps = 9;
constexpr int kThreads = (kEpiWarps + 1) * 32;
constexpr int kEpiBar = 1;                    // named barrier of the epilogue warps
constexpr int kRowsPerWarp = 16;
constexpr int kMaxNR = 144;
constexpr int kWPiece = 16384;                // bytes per bulk copy of the W_h^T image

template <int C, int NR>
struct XShape {
  static constexpr int CS = C / kChan;              // CTAs per cluster
  static constexpr int HALVES = C / 128;            // MMA M = 128 outputs
  static constexpr int W_ATOM = 128 * 128;          // 128 outputs x 64 k fp16, 128-byte rows
  static constexpr int W_HALF = 2 * W_ATOM;         // the two k atoms of one output half
  static constexpr int W_TERM = HALVES * W_HALF;
  static constexpr int W_BYTES = 2 * W_TERM;        // one CTA's image (hi, lo)
  static constexpr int B_ATOM = (NR / 8) * 1024;    // NR rows x 64 k fp16
  static constexpr int B_TERM = 2 * B_ATOM;
  static constexpr int B_BYTES = 2 * B_TERM;
  static constexpr int BLOCK = NR * kChan;          // floats of one exchange block
  static constexpr int PW = NR / kRowsPerWarp;      // epilogue warps with rows
  static constexpr int NBARS = 6;                   // wfull, done[2], b_ready, xfull, spare
  static constexpr int USED = W_BYTES + B_BYTES + 2 * NR * 4 + BLOCK * 4 + NBARS * 8 + 16 + 1024;
  // At least half an SM's shared memory: a CTA takes all 512 tensor-memory columns.
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
  static_assert(NR % 16 == 0 && NR <= kMaxNR && PW <= kEpiWarps, "row tile");
  static_assert(HALVES * NR <= 512, "tensor-memory columns");
  static_assert(W_BYTES % kWPiece == 0, "W image pieces");
};

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16in(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Tensor-memory loads of 8 / 16 consecutive fp32 columns of this warp's 32 lanes, without the
// wait: several are issued back to back and tmem_wait_ld8 (below) completes them.
__device__ __forceinline__ void tmem_ld8_nw(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Ties 8 loaded registers to a point after the wait, so no use of them moves above it.
__device__ __forceinline__ void tmem_after_wait8(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]));
}

// Reads NC (a multiple of 8, at most 64) columns of the partial starting at column c0 (one
// wait for all of them), scales them back and stores them into the exchange block `blk`
// (row-major [rows][32], this lane's output column): in global memory (L2 only), or in this
// CTA's shared memory when `to_smem` (a warp-uniform choice).
template <int NC>
__device__ __forceinline__ void drain_piece(uint32_t dmem, int c0, float os,
                                            const float* __restrict__ ri,
                                            float* __restrict__ blk, bool to_smem) {
  static_assert(NC % 8 == 0 && NC <= 64, "piece");
  uint32_t r[NC];
  float rs[NC];  // the row scales, read before any store (the block may be in shared memory)
#pragma unroll
  for (int j = 0; j < NC; ++j) rs[j] = ri[c0 + j];
#pragma unroll
  for (int j = 0; j + 16 <= NC; j += 16) tmem_ld16_nw(dmem + c0 + j, r + j);
  if constexpr (NC % 16 != 0) tmem_ld8_nw(dmem + c0 + NC - 8, r + NC - 8);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < NC; j += 8) tmem_after_wait8(r + j);
  if (to_smem) {
#pragma unroll
    for (int j = 0; j < NC; ++j) blk[(c0 + j) * kChan] = (__uint_as_float(r[j]) * os) * rs[j];
  } else {
#pragma unroll
    for (int j = 0; j < NC; ++j)
      __stcg(blk + (c0 + j) * kChan, (__uint_as_float(r[j]) * os) * rs[j]);
  }
}


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

// Power-of-two scale for a row whose largest magnitude is m: the exponent e with
// m * 2^e in [2^14, 2^15) (m = f 2^E, f in [0.5, 1): e = 15 - E), clamped to [-126, 126] so that
// both 2^e and 2^-e are normal; 0 for m = 0.
__device__ __forceinline__ int pow2_exponent(float m) {
  if (!(m > 0.f)) return 0;
  int E;
  (void)frexpf(m, &E);
  const int e = 15 - E;
  return e < -126 ? -126 : (e > 126 ? 126 : e);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Byte offset of element (row n, reduction entry k < 128) in one B term of NR rows: K-major,
// 128-byte swizzle, atoms of 64 k.
template <int NR>
__device__ __forceinline__ uint32_t b_offset(int n, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * ((NR / 8) * 1024) + (n >> 3) * 1024 +
                               (n & 7) * 128 + (((chunk & 7) ^ (n & 7)) << 4));
}

// The per-CTA W_h^T image: term (hi, lo), output half, k atom, then a K-major 128-byte-
// swizzled [128 outputs x 64 k] tile; and the power of two each output row was scaled by
// (its inverse is stored).  One warp per (rank, output o): lane = local channel c, its four
// gates are k = 4 c .. 4 c + 3.
template <int C>
__global__ void __launch_bounds__(256) bwd_l2x_split_kernel(const float* __restrict__ W, int n_x,
                                                            int n_in, uint8_t* __restrict__ img,
                                                            float* __restrict__ oscale) {
  using S = XShape<C, 128>;
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= S::CS * C) return;
  const int rank = gw / C, o = gw % C;
  const int ch = kChan * rank + lane;
  float v[4];
  float m = 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    v[g] = __ldg(W + (static_cast<size_t>(g) * C + ch) * n_in + n_x + o);
    m = fmaxf(m, fabsf(v[g]));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  const int e = pow2_exponent(m);
  const float s = pow2f(e);
  __half hi[4], lo[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const float x = v[g] * s;
    hi[g] = __float2half_rn(x);
    lo[g] = __float2half_rn(x - __half2float(hi[g]));
  }
  // k = 4 lane + g: atom lane / 16, 16-byte chunk (lane % 16) / 2, half of the chunk lane % 2.
  const int h = o >> 7, r = o & 127;
  const int chunk = (lane & 15) >> 1;
  const uint32_t off = static_cast<uint32_t>(h * S::W_HALF + (lane >> 4) * S::W_ATOM +
                                             (r >> 3) * 1024 + (r & 7) * 128 +
                                             ((chunk ^ (r & 7)) << 4) + (lane & 1) * 8);
  uint8_t* base = img + static_cast<size_t>(rank) * S::W_BYTES + off;
  *reinterpret_cast<uint2*>(base) = make_uint2(pack_h2(hi[0], hi[1]), pack_h2(hi[2], hi[3]));
  *reinterpret_cast<uint2*>(base + S::W_TERM) =
      make_uint2(pack_h2(lo[0], lo[1]), pack_h2(lo[2], lo[3]));
  if (lane == 0) oscale[rank * C + o] = pow2f(-e);
}

// BF: the cache holds bf16 elements (BwdParams::cache_bf16).
template <int C, int NR, bool BF>
__global__ void __launch_bounds__(kThreads, 1) cfc_bwd_l2x_kernel(const BwdParams p) {
  using S = XShape<C, NR>;
  constexpr int CS = S::CS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sW = smem_addr(sm);
  uint8_t* bterm = sm + S::W_BYTES;
  const uint32_t sB = smem_addr(bterm);
  float* rinv = reinterpret_cast<float*>(sm + S::W_BYTES + S::B_BYTES);  // [2][NR]: 2^-e_row
  float* own = rinv + 2 * NR;  // [NR][32]: this CTA's own exchange block
  uint64_t* bars = reinterpret_cast<uint64_t*>(own + S::BLOCK);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + S::NBARS);
  const uint32_t wfull = smem_addr(&bars[0]);
  const uint32_t done0 = smem_addr(&bars[1]);    // + 8 h: MMAs of output half h committed
  const uint32_t b_ready = smem_addr(&bars[3]);  // next B written (epilogue threads)
  const uint32_t xfull = smem_addr(&bars[4]);    // this CTA's exchange blocks all in L2

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_id_x());
  const int row0 = cid * NR;
  const int B = p.B, K = p.K;
  const uint8_t* wimg = static_cast<const uint8_t*>(p.wsplit);
  const float* oscale = reinterpret_cast<const float*>(wimg + static_cast<size_t>(CS) * S::W_BYTES);
  // Exchange blocks of this cluster: [parity][dest][src][NR][32] fp32 (the blocks with
  // dest == src are not used: each CTA keeps its own in shared memory).
  float* xb = p.xbuf + static_cast<size_t>(cid) * 2 * CS * CS * S::BLOCK;

  if (tid == 0) {
    mbar_init(wfull, 1);
    mbar_init(done0, 1);
    mbar_init(done0 + 8u, 1);
    mbar_init(b_ready, kEpiWarps * 32);
    mbar_init(xfull, kDrainWarps);
    fence_mbar_init_cluster();
  }
  // The W_h^T image, dH and the cache come from earlier kernels.
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (warp == kEpiWarps) {
    tmem_alloc(smem_addr(tslot), 512);
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  cluster_sync_all();  // every CTA's barriers initialised before any remote arrive

  if (warp == kEpiWarps) {
    if (lane == 0) {
      // ---- W_h^T slice into shared memory once, then the MMAs of steps 1 .. K ----
      bool ok = true;
      mbar_arrive_expect_tx(wfull, S::W_BYTES);
      const uint8_t* src = wimg + static_cast<size_t>(rank) * S::W_BYTES;
      for (int i = 0; i < S::W_BYTES / kWPiece; ++i)
        bulk_g2s(sW + i * kWPiece, src + static_cast<size_t>(i) * kWPiece, kWPiece, wfull);
      ok = mbar_wait_bounded_cta(wfull, 0, p.status);
      constexpr uint32_t idesc = idesc_f16in(128, NR);
      int commits = 0;
      for (int n = 1; n <= K && ok; ++n) {
        ok = mbar_wait_bounded_cta(b_ready, (n - 1) & 1, p.status);
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll
        for (int h = 0; h < S::HALVES; ++h) {
          const uint32_t d = tmem + static_cast<uint32_t>(h * NR);
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks) {
            const uint32_t koff = (ks & 3) * 32;  // 16 k = 32 bytes into the atom
            const uint32_t wa = sW + h * S::W_HALF + (ks >> 2) * S::W_ATOM + koff;
            const uint32_t ba = sB + (ks >> 2) * S::B_ATOM + koff;
            const uint64_t a_hi = umma_desc_sw128(wa), a_lo = umma_desc_sw128(wa + S::W_TERM);
            const uint64_t b_hi = umma_desc_sw128(ba), b_lo = umma_desc_sw128(ba + S::B_TERM);
            umma_ss(d, a_hi, b_hi, idesc, ks > 0 ? 1u : 0u);
            umma_ss(d, a_hi, b_lo, idesc, 1u);
            umma_ss(d, a_lo, b_hi, idesc, 1u);
          }
          umma_commit(done0 + 8u * h);
        }
        ++commits;
      }
      // The MMAs committed here finish before tensor memory is freed, whatever else stopped.
      if (!ok && commits > 0)
        for (int h = 0; h < S::HALVES; ++h)
          (void)mbar_wait_bounded_cta(done0 + 8u * h, (commits - 1) & 1, p.status);
    }
  } else {
    // ---- epilogue warps ----
    // Drain role (warps 0 .. 7): tensor-memory lane quarter q holds outputs 32 q .. 32 q + 31
    // of output half dh, i.e. channel block `dest`; columns are batch rows.  The block for this
    // CTA's own channels stays in shared memory (`own`); the others go to L2.
    const int q = warp & 3;
    const int dh = (S::HALVES == 2) ? (warp >> 2) : 0;
    const int dest = 4 * dh + q;
    const int col_lo = (S::HALVES == 2) ? 0 : (warp >> 2) * (NR / 2);
    const bool drainer = warp < kDrainWarps;
    const float os = drainer ? __ldg(oscale + rank * C + 128 * dh + 32 * q + lane) : 0.f;
    const uint32_t dmem = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                          static_cast<uint32_t>(dh * NR);
    // Row role: rows 16 warp + 2 i + (lane >> 4), channels 2 cp, 2 cp + 1 of this CTA.
    const int cp = lane & 15, rsub = lane >> 4;
    const bool has_rows = warp < S::PW;
    const int ch = kChan * rank + 2 * cp;
    bool ok = true;
    for (int n = 0; n <= K && ok; ++n) {
      const int t = K - 1 - n;
      const int par = n & 1;
      if (n > 0) {
        if (drainer) {
          // ---- this step's partial: scaled back, into block (dest, rank) of the exchange ----
          bool dok = mbar_wait_bounded_cta(done0 + 8u * dh, (n - 1) & 1, p.status);
          dok = __all_sync(0xffffffffu, dok);
          if (dok) {
            tc_fence_after_sync();
            const float* ri = rinv + (par ^ 1) * NR;  // row scales of the B this MMA read
            float* blk = dest == rank
                             ? own + lane
                             : xb + (static_cast<size_t>((par * CS + dest) * CS + rank)) * S::BLOCK + lane;
            constexpr int DC = S::HALVES == 2 ? NR : NR / 2;  // columns per drain warp
            const bool mine = dest == rank;
#pragma unroll 1
            for (int pc = 0; pc < DC / 64; ++pc)
              drain_piece<64>(dmem, col_lo + 64 * pc, os, ri, blk, mine);
            if constexpr (DC % 64 != 0)
              drain_piece<DC % 64>(dmem, col_lo + DC - DC % 64, os, ri, blk, mine);
            tc_fence_before_sync();  // the reads precede the next step's MMAs (via b_ready)
            __syncwarp();
            if (dest != rank) fence_acq_rel_gpu();
            if (lane == 0) mbar_arrive_remote(map_to_rank(xfull, dest));
          }
          ok = dok;
        } else if (t >= 0) {
          // ---- warp 8: this step's inputs towards L2 while the exchange runs (per row the
          // CTA's 128-byte slices of dH and of the three cache planes (64 bytes in bf16), and
          // ts) ----
          for (int j = lane; j < 5 * NR; j += 32) {
            const int b = row0 + j / 5, kind = j % 5;
            if (b < B) {
              const size_t tb = static_cast<size_t>(t) * B + b;
              const size_t ce = (tb * 3 + (kind - 1)) * C + kChan * rank;  // cache element
              prefetch_l2(kind == 0   ? static_cast<const void*>(p.dH + tb * C + kChan * rank)
                          : kind == 4 ? static_cast<const void*>(p.ts + tb)
                          : BF
                              ? static_cast<const void*>(reinterpret_cast<const __nv_bfloat16*>(p.cache) + ce)
                              : static_cast<const void*>(p.cache + ce));
            }
          }
        }
        if (ok) ok = mbar_wait_bounded_cluster(xfull, (n - 1) & 1, p.status);
        // All of this CTA's MMAs of the step (they read B) are done before B is rewritten: the
        // exchange alone only implies the half that warp `rank` drained.
        if (ok) ok = mbar_wait_bounded_cta(done0 + 8u * (S::HALVES - 1), (n - 1) & 1, p.status);
        if (bar_or(kEpiBar, kEpiWarps * 32, !ok)) {
          ok = false;
          break;
        }
      }
      if (has_rows) {
        const float* in = xb + static_cast<size_t>(par * CS + rank) * CS * S::BLOCK + 2 * cp;
        // Two batches of 4 rows, unrolled so that the second batch's loads can be in flight
        // while the first one computes.
#pragma unroll
        for (int ib = 0; ib < 2; ++ib) {
          int rr[4];
          bool rv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            rr[i] = kRowsPerWarp * warp + 2 * (4 * ib + i) + rsub;
            rv[i] = row0 + rr[i] < B;
          }
          // This step's inputs and the exchange blocks, all loads issued before any is used
          // (rows past B read row 0 of the step and are zeroed).
          float2 dHv[4], f1[4], f2[4], gg[4];
          float tsv[4];
          const int tt = t >= 0 ? t : 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const size_t tb = static_cast<size_t>(tt) * B + (rv[i] ? row0 + rr[i] : 0);
            dHv[i] = __ldcg(reinterpret_cast<const float2*>(p.dH + tb * C + ch));
            if constexpr (BF) {  // bf16 pairs of channels (ch, ch + 1)
              const unsigned int* cq = reinterpret_cast<const unsigned int*>(
                  reinterpret_cast<const __nv_bfloat16*>(p.cache) + tb * 3 * C + ch);
              const unsigned int a = __ldcg(cq), b2 = __ldcg(cq + C / 2), c2 = __ldcg(cq + C);
              f1[i] = make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
              f2[i] = make_float2(__uint_as_float(b2 << 16), __uint_as_float(b2 & 0xffff0000u));
              gg[i] = make_float2(__uint_as_float(c2 << 16), __uint_as_float(c2 & 0xffff0000u));
            } else {
              const float* cpp = p.cache + tb * 3 * C + ch;
              f1[i] = __ldcg(reinterpret_cast<const float2*>(cpp));
              f2[i] = __ldcg(reinterpret_cast<const float2*>(cpp + C));
              gg[i] = __ldcg(reinterpret_cast<const float2*>(cpp + 2 * C));
            }
            tsv[i] = __ldg(p.ts + tb);
          }
          float2 delta[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) delta[i] = make_float2(0.f, 0.f);
          if (n > 0) {
            float2 x[CS][4];
#pragma unroll
            for (int s = 0; s < CS; ++s)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int off = s * S::BLOCK + rr[i] * kChan;
                x[s][i] = s == rank
                              ? *reinterpret_cast<const float2*>(own + rr[i] * kChan + 2 * cp)
                              : __ldcg(reinterpret_cast<const float2*>(in + off));
              }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int s = 0; s < CS; ++s) {  // rank order: a fixed summation order
                delta[i].x += x[s][i].x;
                delta[i].y += x[s][i].y;
              }
          }
          if (n == K) {  // the last exchange: delta = W_h^T d_pre[0] = dh0
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (rv[i])
                *reinterpret_cast<float2*>(p.dh0 + static_cast<size_t>(row0 + rr[i]) * C + ch) =
                    delta[i];
            continue;
          }
          // ---- d_pre of step t for two channels of each of the 4 rows ----
          float pv[4][2][4];  // [row][channel][gate]
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float z = rv[i] ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float dhv = z * ((c ? dHv[i].y : dHv[i].x) + (c ? delta[i].y : delta[i].x));
              const float a1 = c ? f1[i].y : f1[i].x, a2 = c ? f2[i].y : f2[i].x;
              const float g = c ? gg[i].y : gg[i].x;
              const float ds = dhv * (a2 - a1) * g * (1.f - g);
              pv[i][c][0] = dhv * (1.f - g) * (1.f - a1 * a1);
              pv[i][c][1] = dhv * g * (1.f - a2 * a2);
              pv[i][c][2] = ds * tsv[i];
              pv[i][c][3] = ds;
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (rv[i]) {
              const size_t row = static_cast<size_t>(t) * B + row0 + rr[i];
              if (p.dplanes == 0) {
                float* dpp = p.d_pre + row * 4 * C + ch;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  *reinterpret_cast<float2*>(dpp + static_cast<size_t>(g) * C) =
                      make_float2(pv[i][0][g], pv[i][1][g]);
              } else {
                // Operand row: 2 dpitch bf16 values, hi at k = g C + channel, lo dpitch on.
                __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(p.d_pre) +
                                   row * 2 * static_cast<size_t>(p.dpitch) + ch;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                  uint32_t hi2, lo2;
                  bf16_split2_pair(pv[i][0][g], pv[i][1][g], hi2, lo2);
                  *reinterpret_cast<uint32_t*>(q + static_cast<size_t>(g) * C) = hi2;
                  if (p.dplanes == 2)
                    *reinterpret_cast<uint32_t*>(q + p.dpitch + static_cast<size_t>(g) * C) = lo2;
                }
              }
            }
          // Row scales: the largest magnitude over each row's 128 entries (16 lanes).
          float m[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            m[i] = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int g = 0; g < 4; ++g) m[i] = fmaxf(m[i], fabsf(pv[i][c][g]));
          }
#pragma unroll
          for (int d = 8; d > 0; d >>= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], d));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = pow2_exponent(m[i]);
            const float sc = pow2f(e);
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int gp = 0; gp < 2; ++gp) {
                const float x0 = pv[i][c][2 * gp] * sc, x1 = pv[i][c][2 * gp + 1] * sc;
                f16_split2_pair(x0, x1, hw[2 * c + gp], lw[2 * c + gp]);
              }
            // k = 8 cp .. 8 cp + 7 of row rr[i]: one 16-byte chunk per term.
            const uint32_t off = b_offset<NR>(rr[i], cp);
            *reinterpret_cast<uint4*>(bterm + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(bterm + S::B_TERM + off) =
                make_uint4(lw[0], lw[1], lw[2], lw[3]);
            if (cp == 0) rinv[par * NR + rr[i]] = pow2f(-e);
          }
        }
      }
      if (n == K) break;
      fence_proxy_async_smem();  // the B terms -> visible to the MMAs
      tc_fence_before_sync();
      mbar_arrive(b_ready);
    }
  }

  // Leave together: no CTA exits while another may still arrive on its barriers.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == kEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int C, int NR>
cudaError_t prepare_k(int* max_active_clusters) {
  using S = XShape<C, NR>;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (S::SMEM > optin) {
    *max_active_clusters = 0;
    return cudaSuccess;
  }
  // Both cache dtypes: same launch bounds and shared memory, so the same occupancy.
  auto* kern = cfc_bwd_l2x_kernel<C, NR, false>;
  for (auto* k : {cfc_bwd_l2x_kernel<C, NR, false>, cfc_bwd_l2x_kernel<C, NR, true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
  }
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

template <int C, int NR>
cudaError_t launch_k(const BwdParams& p, cudaStream_t s, bool pdl) {
  using S = XShape<C, NR>;
  LaunchCfg c;
  c.grid = dim3(((p.B + NR - 1) / NR) * S::CS, 1, 1);
  c.block = dim3(kThreads, 1, 1);
  c.smem = S::SMEM;
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(S::CS, 1, 1);
  return p.cache_bf16 ? launch(c, cfc_bwd_l2x_kernel<C, NR, true>, p)
                      : launch(c, cfc_bwd_l2x_kernel<C, NR, false>, p);
}

template <int C>
cudaError_t split_k(const float* W, int n_x, void* img, cudaStream_t s, bool pdl) {
  using S = XShape<C, 128>;
  LaunchCfg c;
  c.grid = dim3((S::CS * C * 32 + 255) / 256, 1, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  uint8_t* base = static_cast<uint8_t*>(img);
  return launch(c, bwd_l2x_split_kernel<C>, W, n_x, n_x + C, base,
                reinterpret_cast<float*>(base + static_cast<size_t>(S::CS) * S::W_BYTES));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

bool bwd_l2x_supported(int C) { return C == 128 || C == 256; }

int bwd_l2x_rows(int B, int max_clusters_128) {
  return (B + 127) / 128 <= max_clusters_128 ? 128 : 144;
}

size_t bwd_l2x_image_bytes(int C) {
  // W_h^T image (C * 512 bytes per CTA, C / 32 CTAs) and the output scales.
  const size_t cs = static_cast<size_t>(C) / kChan;
  return align256(cs * C * 512 + cs * C * sizeof(float));
}

size_t bwd_l2x_ws_bytes(int B, int C) {
  // The exchange blocks of every cluster, for either row tile: [cluster][2][CS][CS][NR][32].
  const size_t cs = static_cast<size_t>(C) / kChan;
  size_t rows = 0;
  for (const int nr : {128, 144}) {
    const size_t r = ((static_cast<size_t>(B) + nr - 1) / nr) * nr;
    rows = r > rows ? r : rows;
  }
  return bwd_l2x_image_bytes(C) + rows * 2 * cs * cs * kChan * sizeof(float);
}

cudaError_t bwd_l2x_prepare(int C, int NR, int* max_active_clusters) {
  if (C == 128 && NR == 128) return prepare_k<128, 128>(max_active_clusters);
  if (C == 128 && NR == 144) return prepare_k<128, 144>(max_active_clusters);
  if (C == 256 && NR == 128) return prepare_k<256, 128>(max_active_clusters);
  if (C == 256 && NR == 144) return prepare_k<256, 144>(max_active_clusters);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_l2x_split(const float* W, int C, int n_x, void* ws, cudaStream_t s, bool pdl) {
  if (C == 128) return split_k<128>(W, n_x, ws, s, pdl);
  if (C == 256) return split_k<256>(W, n_x, ws, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_l2x_launch(const BwdParams& p, int NR, cudaStream_t s, bool pdl) {
  if (p.dplanes < 0 || p.dplanes > 2 || p.xbuf == nullptr) return cudaErrorInvalidValue;
  if (p.dplanes > 0 && (p.dpitch < 4 * p.C || p.dpitch % 8 != 0)) return cudaErrorInvalidValue;
  if (p.C == 128 && NR == 128) return launch_k<128, 128>(p, s, pdl);
  if (p.C == 128 && NR == 144) return launch_k<128, 144>(p, s, pdl);
  if (p.C == 256 && NR == 128) return launch_k<256, 128>(p, s, pdl);
  if (p.C == 256 && NR == 144) return launch_k<256, 144>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace cfc
