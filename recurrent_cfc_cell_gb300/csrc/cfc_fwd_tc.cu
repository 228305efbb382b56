// cfc_fwd_tc.cu -- the forward recurrence with the per-step gate contraction on the
// 5th-generation tensor cores, for large batches.
//
// The recurrence of page "K-loop Parallelization -- Block-per-Batch Kernel Refactor" (section
// "Problem": P = W z + b, then the cell) is, for many batch rows at once, one contraction per
// step: [rows x C] h_{t-1} times [C x 4C] W_h^T, plus the input projection X computed before
// the loop.  The pages note that a bigger batch wants mixed-precision matrix hardware
// (section "Headline Numbers").  Here each step's contraction runs on tcgen05 with fp32-level
// accuracy.  Both operands are split into two fp16 terms, x = hi + lo with hi = fp16(x) and
// lo = fp16(x - hi), carrying 22 significand bits.  The product keeps hi*hi + hi*lo + lo*hi,
// three MMAs per 16-deep step; what is dropped is below about 2^-21 of each product.  h lies
// in (-1, 1).  Each row of W is scaled by a power of two into [-1, 1) before the split, and
// the result is scaled back exactly, so no weight over- or underflows fp16.
//
// Layout: a thread-block cluster of CS = C / 32 CTAs serves NR = 128 or 144 batch rows; CTA
// `rank` owns channels 32 rank .. 32 rank + 31, i.e. 128 gate rows of W.  Per CTA:
//   tensor memory  D^T [128 gate rows (lanes) x NR batch rows (columns)] fp32, then the CTA's
//                  W_h^T slice as the A operand (lane 4c + g = gate g of local channel c, k
//                  along columns in fp16 pairs), two terms of C / 2 columns each;
//   shared memory  h_{t-1} as the B operand, two fp16 terms [C x NR] in the non-swizzled
//                  K-major layout [k / 8][row / 8][8 rows][16 bytes], so the 32 values of
//                  k that one CTA produces form one contiguous slab per term.
// Roles (320 threads): eight epilogue warps, a control warp whose lane 0 issues the MMAs and
// an exchange warp whose lane 0 moves the slabs.  A step t: the control thread issues the
// MMAs slab by slab as the slabs of h_{t-1} land (its own first) and commits them to `done`;
// the epilogue warps wait for `done`, read D^T and add X (a channel's four gates sit in four
// adjacent lanes; a 4 x 4 transpose inside each lane quad gives every lane all four gates of
// one row), apply the cell, write H and the cache and write h_t's two terms into the CTA's
// own slab, then mark it full.  The exchange thread copies that slab to the CTA's slot of an
// exchange buffer in global memory (bulk copy, completion awaited), announces it by a remote
// mbarrier arrive on every other CTA, and bulk-loads the other CTAs' slabs of h_t from L2 as
// they are announced.  The slabs of the cluster used to travel between shared memories
// (bulk copies into distributed shared memory); on GB300 with 15 clusters of 8 CTAs those
// took 4 to 6 us per step to land against about 2 us through L2.  A slab of the exchange
// buffer is rewritten two steps later (slots alternate with the step parity, and so do the
// announcing barriers): by then every CTA has loaded it, because it needed this CTA's next
// slab first.  No CTA waits for another except for the data it reads.  Every wait is
// bounded; a timeout is recorded in the status word and every role leaves its loop.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kGC = 4 * kFwdChanPerCta;          // gate rows per CTA (MMA M)
constexpr int kEpiWarps = 8;                     // epilogue warps (two per TMEM lane quarter)
constexpr int kCtlWarp = kEpiWarps;              // lane 0 issues the MMAs
constexpr int kXchWarp = kEpiWarps + 1;          // lane 0 runs the exchange
constexpr int kTcThreads = (kEpiWarps + 2) * 32;
constexpr int kTerms = 2;                        // fp16 terms per operand
constexpr uint32_t kACol0 = 256;                 // W_h^T terms start here; D^T takes NR columns
// Fused input projection: W_u^T as three bf16 terms of kUMax / 2 columns each from kUCol0
// (between D^T's at most 144 columns and W_h^T), u_t as three bf16 terms in shared memory.
constexpr int kUTerms = 3;
constexpr int kUMax = 64;                        // inputs the fused form takes (n_x <= 64)
constexpr uint32_t kUCol0 = 160;
static_assert(kUMax == kFwdFuseMaxInputs, "fused input width");
static_assert(kUCol0 + kUTerms * kUMax / 2 <= kACol0, "W_u^T below W_h^T in tensor memory");

// NR: batch rows per cluster (MMA N), 128 or 144.  144 lets 15 clusters cover 2048 rows:
// GB300 keeps at most 15 clusters of 8 CTAs resident, so 16 clusters of 128 rows ran in two
// waves.
template <int CS, int NR, bool FU = false>
struct TcShape {
  static constexpr int C = kFwdChanPerCta * CS;
  static constexpr int TERM = C * NR * 2;        // bytes of one fp16 term of h
  static constexpr int SLAB = NR * kFwdChanPerCta * 2;  // one CTA's k range of one h term
  static constexpr int XSLOT = kTerms * SLAB;    // one CTA's exchange slot: its slab, both terms
  static constexpr int HR = NR / 2;              // rows of one epilogue warp half
  static constexpr int ACOLS = C / 2;            // TMEM columns of one term of W_h^T
  // u_t (fused form): [k / 8][n / 8][8 rows][16 B] with k groups ULBO bytes apart, 16 more than
  // packed, so that lanes storing eight k groups of one row hit eight different bank groups.
  static constexpr int ULBO = NR * 16 + 16;
  static constexpr int UTERM = kUMax / 8 * ULBO;  // bytes of one bf16 term of u_t
  static constexpr int UBYTES = FU ? kUTerms * UTERM : 0;
  static constexpr int NBARS = 3 * CS + 3;       // full[CS], done, fin, ufull, ready[2][CS]
  static_assert(NR % 16 == 0 && HR % 8 == 0 && NR <= 256, "row tile");
  static_assert(NR <= static_cast<int>(kUCol0), "D^T below W_u^T");
  // h terms, u terms, each epilogue warp's ts, barriers, TMEM slot, alignment.
  static constexpr int USED =
      kTerms * TERM + UBYTES + kEpiWarps * HR * 4 + NBARS * 8 + 16 + 128;
  // At least half an SM's shared memory: a CTA takes all 512 tensor-memory columns, so two
  // CTAs on one SM would leave the second waiting in tcgen05.alloc while its cluster waits on
  // it.
  static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

struct Split2 {
  __half t[2];
};
__device__ __forceinline__ Split2 split2(float x) {
  Split2 s;
  s.t[0] = __float2half_rn(x);
  s.t[1] = __float2half_rn(x - __half2float(s.t[0]));
  return s;
}
__device__ __forceinline__ uint32_t pack2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}
// Instruction descriptor of kind::f16 with fp16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16in(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Three bf16 terms x = hi + mid + lo (8 significand bits each, so the three carry all 24 of
// fp32; each difference is exact in fp32), packed in pairs: pk[term] = (term of a, of b) with
// a in the low half, one packed conversion per term.
__device__ __forceinline__ void split3_pair(float a, float b, uint32_t (&pk)[kUTerms]) {
  pk[0] = bf16x2_rn(a, b);
  const float ar = a - bf16_lo_f32(pk[0]), br = b - bf16_hi_f32(pk[0]);
  pk[1] = bf16x2_rn(ar, br);
  pk[2] = bf16x2_rn(ar - bf16_lo_f32(pk[1]), br - bf16_hi_f32(pk[1]));
}

// Byte offset of element (row n, k) in one h term of NR rows: [k / 8][n / 8][n % 8][k % 8].
template <int NR>
__device__ __forceinline__ uint32_t hterm_offset(int n, int k) {
  return static_cast<uint32_t>(((k >> 3) * (NR / 8) + (n >> 3)) * 128 + (n & 7) * 16 +
                               (k & 7) * 2);
}

// Tensor-memory load of 8 consecutive fp32 columns of this warp's 32 lanes.
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

// Shared-memory operand descriptor, no swizzle, K-major: `lbo` bytes between core matrices
// along k, `sbo` bytes between core matrices along the rows.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version; layout type 0 (no swizzle)
  return d;
}

// D (tensor memory) += A (tensor memory) * B (shared memory descriptor).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 32 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// FU: the input projection is fused (X = W_u u_t + b is not read from memory: u_t enters the
// step's contraction, b the epilogue).
template <int CS, int NR, bool BF, bool FU>
__global__ void __launch_bounds__(kTcThreads, 1) cfc_fwd_tc_kernel(const FwdParams p) {
  using S = TcShape<CS, NR, FU>;
  constexpr int HR = S::HR;
  constexpr int C = S::C;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* sm = smem_raw + ((128u - (raw & 127u)) & 127u);
  uint8_t* hb = sm;                                                     // [2][TERM]
  uint8_t* ub = sm + kTerms * S::TERM;                                  // FU: [3][UTERM]
  float* ts_w = reinterpret_cast<float*>(ub + S::UBYTES);               // [kEpiWarps][HR]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ts_w + kEpiWarps * HR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + S::NBARS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cluster = static_cast<int>(cluster_id_x());
  const int n_clusters = static_cast<int>(gridDim.x) / CS;
  const int row0 = cluster * NR;
  const int B = p.B, K = p.K, n_x = p.n_x, n_in = p.n_in;
  const uint32_t full0 = smem_addr(&bars[0]);          // full[j]: slab j of the step's h in place
  const uint32_t done_bar = smem_addr(&bars[CS]);      // this CTA's MMAs of the step are done
  const uint32_t fin_bar = smem_addr(&bars[CS + 1]);   // every MMA of this CTA is done (exit)
  const uint32_t ufull = smem_addr(&bars[CS + 2]);     // FU: u of the step in place, D^T free
  const uint32_t ready0 = smem_addr(&bars[CS + 3]);    // ready[par][j]: CTA j's slab is in L2
  const int KU = (n_x + 15) & ~15;                     // FU: inputs padded to whole MMA steps
  uint8_t* const xch = static_cast<uint8_t*>(p.xch);
  // Exchange slot of CTA r of this cluster for step parity par.
  auto slot = [&](int par, int r) {
    return xch + static_cast<size_t>((par * n_clusters + cluster) * CS + r) * S::XSLOT;
  };

  grid_dep_launch_dependents();
  if (tid == 0) {
    // The own slab is filled by the eight epilogue warps, the others by one bulk load each.
    for (int j = 0; j < CS; ++j) mbar_init(full0 + 8u * j, j == rank ? kEpiWarps : 1);
    mbar_init(done_bar, 1);
    mbar_init(fin_bar, 1);
    mbar_init(ufull, kEpiWarps);
    for (int i = 0; i < 2 * CS; ++i) mbar_init(ready0 + 8u * i, kEpiWarps);
    fence_mbar_init_cluster();
  }
  if (warp == kCtlWarp) {
    tmem_alloc(smem_addr(tslot), 512);
    tc_fence_before_sync();
  }
  // X comes from the projection kernel in place in H / cache (unfused form), and the previous
  // kernel may still read what this one writes: wait for it before any global access.
  grid_dep_wait();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  // This thread's role in the epilogue warps: TMEM lane quarter q, rows HR hh .. HR hh + HR - 1,
  // gate g of local channel c (lane 4c + g of the quarter's 32 lanes).
  const int q = warp & 3, hh = (warp >> 2) & 1;
  const int c = (32 * q + lane) >> 2, g = lane & 3;
  const int ch = kFwdChanPerCta * rank + c;

  // FU: u_t of the cluster's rows -> the three bf16 terms of the u operand (epilogue warps,
  // loaded into registers one step ahead).  Item (row n, inputs k0 .. k0 + 7), the eight k
  // groups of a row in eight consecutive lanes: a warp's loads touch 4 rows (8 lines of 128
  // bytes, not 32), and its 16-byte stores, with the k groups ULBO apart, 32 distinct bank
  // slots per 128 bytes.  Zero beyond B and n_x.
  constexpr int kUItems = (NR * kUMax / 8 + kEpiWarps * 32 - 1) / (kEpiWarps * 32);
  float un[FU ? kUItems : 1][8];
  auto load_u = [&](int t) {
    if constexpr (FU) {
      const bool vec = (n_x & 3) == 0;
#pragma unroll
      for (int m = 0; m < kUItems; ++m) {
        const int it = tid + m * kEpiWarps * 32;
        const int n = it / (kUMax / 8), k0 = 8 * (it % (kUMax / 8)), b = row0 + n;
#pragma unroll
        for (int i = 0; i < 8; ++i) un[m][i] = 0.f;
        if (n < NR && k0 < KU && b < B) {
          const float* src = p.u + (static_cast<size_t>(t) * B + b) * n_x + k0;
          if (vec && k0 + 8 <= n_x) {
            const float4 q0 = ld_early_f4(src);
            const float4 q1 = ld_early_f4(src + 4);
            un[m][0] = q0.x; un[m][1] = q0.y; un[m][2] = q0.z; un[m][3] = q0.w;
            un[m][4] = q1.x; un[m][5] = q1.y; un[m][6] = q1.z; un[m][7] = q1.w;
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (k0 + i < n_x) un[m][i] = ld_early(src + i);
          }
        }
      }
    }
  };
  auto store_u = [&]() {
    if constexpr (FU) {
#pragma unroll
      for (int m = 0; m < kUItems; ++m) {
        const int it = tid + m * kEpiWarps * 32;
        const int n = it / (kUMax / 8), k0 = 8 * (it % (kUMax / 8));
        if (n < NR && k0 < KU) {
          uint32_t w[kUTerms][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t pk[kUTerms];
            split3_pair(un[m][2 * i], un[m][2 * i + 1], pk);
#pragma unroll
            for (int tm = 0; tm < kUTerms; ++tm) w[tm][i] = pk[tm];
          }
          const uint32_t off = static_cast<uint32_t>((k0 >> 3) * S::ULBO + (n >> 3) * 128 +
                                                     (n & 7) * 16);
#pragma unroll
          for (int tm = 0; tm < kUTerms; ++tm)
            *reinterpret_cast<uint4*>(ub + tm * S::UTERM + off) =
                make_uint4(w[tm][0], w[tm][1], w[tm][2], w[tm][3]);
        }
      }
    }
  };

  float wunscale = 1.f;  // 2^e: this lane's W row was scaled by 2^-e before the split
  if (warp < kEpiWarps) {
    // ---- W_h^T slice -> tensor memory (two fp16 terms); the two warps of a lane quarter
    // take the two halves of k.  Row scale: max|W| * 2^-e in [0.5, 1). ----
    const float* wrow = p.W + (static_cast<size_t>(g) * C + ch) * n_in + n_x;
    float wmax = 0.f;
    for (int k = 0; k < C; ++k) wmax = fmaxf(wmax, fabsf(__ldg(wrow + k)));
    int e = 0;
    if (wmax > 0.f) (void)frexpf(wmax, &e);
    const float wscale = ldexpf(1.f, -e);
    wunscale = ldexpf(1.f, e);
    for (int k0 = hh * (C / 2); k0 < (hh + 1) * (C / 2); k0 += 64) {
      uint32_t r0[32], r1[32];
#pragma unroll
      for (int cc = 0; cc < 32; ++cc) {
        const Split2 a = split2(__ldg(wrow + k0 + 2 * cc) * wscale);
        const Split2 b = split2(__ldg(wrow + k0 + 2 * cc + 1) * wscale);
        r0[cc] = pack2(a.t[0], b.t[0]);
        r1[cc] = pack2(a.t[1], b.t[1]);
      }
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + kACol0 + k0 / 2;
      tmem_st32(ta, r0);
      tmem_st32(ta + S::ACOLS, r1);
    }
    if constexpr (FU) {
      // ---- W_u^T (same row scale) -> tensor memory, three bf16 terms; the two warps of a
      // lane quarter take inputs 0 .. 31 and 32 .. 63 (zero beyond n_x). ----
      const float* urow = p.W + (static_cast<size_t>(g) * C + ch) * n_in;
      uint32_t r[kUTerms][16];
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        const int k = kUMax / 2 * hh + 2 * cc;
        const float a = (k < n_x) ? __ldg(urow + k) * wscale : 0.f;
        const float b = (k + 1 < n_x) ? __ldg(urow + k + 1) * wscale : 0.f;
        uint32_t pk[kUTerms];
        split3_pair(a, b, pk);
#pragma unroll
        for (int tm = 0; tm < kUTerms; ++tm) r[tm][cc] = pk[tm];
      }
      const uint32_t tu = tmem + (static_cast<uint32_t>(32 * q) << 16) + kUCol0 + 16 * hh;
#pragma unroll
      for (int tm = 0; tm < kUTerms; ++tm) tmem_st16(tu + tm * (kUMax / 2), r[tm]);
      load_u(0);
      store_u();
      if (K > 1) load_u(1);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    // ---- h0 -> this CTA's slab of the h buffer and its exchange slot of step parity 0
    // (lanes g = 1, 2 write term g - 1). ----
    if (g == 1 || g == 2) {
      uint8_t* const xs = slot(0, rank) + (g - 1) * S::SLAB - rank * S::SLAB;
      for (int i = 0; i < HR; ++i) {
        const int r = HR * hh + i, b = row0 + r;
        const float h = (b < B) ? __ldg(p.h0 + static_cast<size_t>(b) * C + ch) : 0.f;
        const uint32_t off = hterm_offset<NR>(r, ch);
        const __half v = split2(h).t[g - 1];
        *reinterpret_cast<__half*>(hb + (g - 1) * S::TERM + off) = v;
        __stcg(reinterpret_cast<unsigned short*>(xs + off), __half_as_ushort(v));
      }
    }
    // ts of step 0 for this warp's rows (each warp keeps its own copy).
    for (int i = lane; i < HR; i += 32) {
      const int b = row0 + HR * hh + i;
      ts_w[warp * HR + i] = (b < B) ? __ldg(p.ts + b) : 0.f;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  cluster_sync_all();  // every CTA: barriers set up (remote arrives may follow), W_h^T in place
  if (warp < kEpiWarps) {
    // The h0 slab is in place here and in L2: mark it full and announce it.
    fence_acq_rel_gpu();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(full0 + 8u * rank);
      if (FU) mbar_arrive(ufull);  // u_0 in place (written before the CTA barrier above)
    } else if (lane < CS) {
      mbar_arrive_remote(map_to_rank(ready0 + 8u * rank, (rank + lane) % CS));
    }
  }

  if (warp == kCtlWarp) {
    // ================= control thread: the MMAs =================
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16in(kGC, NR);
      const uint64_t bdesc0 = desc_kmajor(smem_addr(hb), (NR / 8) * 128, 128);
      const uint32_t idesc_u = umma_idesc_bf16(kGC, NR);
      const uint64_t udesc0 = desc_kmajor(smem_addr(ub), S::ULBO, 128);
      bool ok = true;
      for (int t = 0; t < K && ok; ++t) {
        uint32_t acc = 0;
        for (int jj = 0; jj < CS; ++jj) {
          const int j = (rank + jj) % CS;  // own slab first, then in rank order
          ok = mbar_wait_bounded_cta(full0 + 8u * j, t & 1, p.status);
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {  // the two 16-deep steps of slab j
            const int s = 2 * j + s2;
            const uint32_t a0 = tmem + kACol0 + 8 * s;
            // Descriptor of B term 0 at this k step; the start-address field counts 16 bytes,
            // so term 1 is a fixed add away.
            const uint64_t d0 = bdesc0 + static_cast<uint64_t>(s * ((NR * 32) >> 4));
            const uint64_t d1 = d0 + (S::TERM >> 4);
            // (A term, B term): hi*hi, hi*lo, lo*hi
            umma_tmem_a(tmem, a0, d0, idesc, acc);
            acc = 1;
            umma_tmem_a(tmem, a0, d1, idesc, 1);
            umma_tmem_a(tmem, a0 + S::ACOLS, d0, idesc, 1);
          }
          if (FU && jj == 0) {
            // W_u u_t right after the own slab (whose wait also says the epilogue has read
            // D^T), while the other CTAs' slabs are still on their way.
            ok = mbar_wait_bounded_cta(ufull, t & 1, p.status);
            if (!ok) break;
            tc_fence_after_sync();
            for (int s = 0; s < KU / 16; ++s) {
              const uint32_t a0 = tmem + kUCol0 + 8 * s;
              const uint64_t d0 = udesc0 + static_cast<uint64_t>(s * ((2 * S::ULBO) >> 4));
              constexpr uint32_t UT = S::UTERM >> 4, AT = kUMax / 2;
              // (A term, B term): hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid
              umma_tmem_a(tmem, a0, d0, idesc_u, 1);
              umma_tmem_a(tmem, a0, d0 + UT, idesc_u, 1);
              umma_tmem_a(tmem, a0 + AT, d0, idesc_u, 1);
              umma_tmem_a(tmem, a0, d0 + 2 * UT, idesc_u, 1);
              umma_tmem_a(tmem, a0 + 2 * AT, d0, idesc_u, 1);
              umma_tmem_a(tmem, a0 + AT, d0 + UT, idesc_u, 1);
            }
          }
        }
        if (ok) umma_commit(done_bar);
      }
      // Every MMA this thread issued has completed before tensor memory is freed.
      umma_commit(fin_bar);
      (void)mbar_wait_bounded_cta(fin_bar, 0, p.status);
    }
  } else if (warp == kXchWarp) {
    // ================= exchange warp =================
    // Step s multiplies h_{s-1}.  Once this CTA's MMAs of step s - 1 are done (its epilogue
    // has filled the own slab), lane jj = 1 .. CS - 1 loads slab rank + jj from L2 as soon as
    // all eight epilogue warps of that CTA have announced it.
    const uint32_t hb0 = smem_addr(hb);
    const bool peer = lane >= 1 && lane < CS;
    const int j = (rank + lane) % CS;  // the slab this lane loads
    bool ok = true;
    int armed = -1;  // the last step whose slab this lane requested
    for (int s = 0; s < K; ++s) {
      const int par = s & 1;
      if (lane == 0) ok = mbar_wait_bounded_cta(full0 + 8u * rank, s & 1, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t rb = ready0 + 8u * (par * CS + j);
      bool pending = peer;
      const uint64_t t0 = global_timer_ns();
      for (uint32_t it = 1; __any_sync(0xffffffffu, pending); ++it) {
        if (pending && mbar_test_wait_cluster(rb, (s >> 1) & 1)) {
          fence_proxy_async_global();
          const uint32_t fb = full0 + 8u * j;
          mbar_arrive_expect_tx(fb, S::XSLOT);
          const uint8_t* const src = slot(par, j);
          for (int tm = 0; tm < kTerms; ++tm)
            bulk_g2s(hb0 + tm * S::TERM + j * S::SLAB, src + tm * S::SLAB, S::SLAB, fb);
          armed = s;
          pending = false;
        }
        if ((it & 255u) == 0u &&
            __any_sync(0xffffffffu, global_timer_ns() - t0 > kWaitLimitNs)) {  // warp-uniform
          if (pending) atomicExch(p.status, kStatusTimeout);
          ok = false;
          break;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
    }
    // No bulk load into this CTA's shared memory is in flight when it exits (they read L2
    // only, so they complete).
    if (armed >= 0) (void)mbar_wait_bounded_cta(full0 + 8u * j, armed & 1, p.status);
  } else {
    // ================= epilogue warps =================
    // Unfused: X of (gate g, channel ch) for rows row0 + HR hh + i, i < HR, of step t, in the
    // layout of H (gate 0) or cache (gates 1-3): in place there unless the outputs are bf16.
    // Fused: the bias of (gate g, channel ch) instead.
    const size_t xrow = (g == 0) ? static_cast<size_t>(C) : 3ull * C;
    const float* xbase = ((g == 0) ? p.xH : p.xcache + static_cast<size_t>(g - 1) * C) + ch;
    constexpr bool obf = BF;  // H and the cache stored as bf16
    const int rfirst = row0 + HR * hh;
    int nvalid = B - rfirst;
    nvalid = nvalid < 0 ? 0 : (nvalid > HR ? HR : nvalid);
    const float bv = FU ? __ldg(p.bias + g * C + ch) : 0.f;
    float xv[FU ? 1 : HR];
    auto load_x = [&](int t) {
      if constexpr (!FU) {
        const float* xp = xbase + (static_cast<size_t>(t) * B + rfirst) * xrow;
#pragma unroll
        for (int i = 0; i < HR; ++i) xv[i] = (i < nvalid) ? ld_early_cg(xp + i * xrow) : 0.f;
      }
    };
    // ts of the next step for this warp's rows: lane i holds rows i, i + 32, ...
    constexpr int kTsPerLane = (HR + 31) / 32;
    float tsn[kTsPerLane];
    auto load_ts = [&](int t) {
#pragma unroll
      for (int k = 0; k < kTsPerLane; ++k) {
        const int i = lane + 32 * k, b = rfirst + i;
        tsn[k] = (i < HR && b < B) ? __ldg(p.ts + static_cast<size_t>(t) * B + b) : 0.f;
      }
    };
    float* const tsw = ts_w + warp * HR;
    load_x(0);
    for (int t = 0; t < K; ++t) {
      bool ok = mbar_wait_bounded_cta(done_bar, t & 1, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      if (t > 0) {
        __syncwarp();  // the previous step's reads of tsw are done
#pragma unroll
        for (int k = 0; k < kTsPerLane; ++k)
          if (lane + 32 * k < HR) tsw[lane + 32 * k] = tsn[k];
        __syncwarp();
      }
      // The H / cache stores of the warp half's last 8 rows (when HR % 16 == 8) are issued
      // after the release fence and the announcements below: the fence waits for every store
      // the thread has in flight, and these would be the youngest.
      float dfv[2][4];
      size_t dfh[2], dfc[2];
      bool dfo[2] = {false, false};
      {
        const float* tsr = tsw;
        const size_t ho = (static_cast<size_t>(t) * B + rfirst) * C + ch;  // element offsets
        const size_t co = (static_cast<size_t>(t) * B + rfirst) * 3 * C + ch;
        const uint32_t dq = tmem + (static_cast<uint32_t>(32 * q) << 16) + HR * hh;
        // h_t is the operand of step t + 1: its exchange slot has that step's parity.
        uint8_t* const xs = slot((t + 1) & 1, rank) - rank * S::SLAB;
        // Rows ibase .. ibase + n - 1 of this warp half (n = 16, or 8 for the tail of 72).
        auto rows = [&](float (&P)[16], int ibase, int n, bool defer) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < n) P[i] = fmaf(P[i], wunscale, FU ? bv : xv[FU ? 0 : ibase + i]);
#pragma unroll
          for (int i0 = 0; i0 < 16; i0 += 4) {
            if (i0 >= n) break;
            // 4 x 4 transpose within the lane quad: lane g held gate g of rows i0 .. i0 + 3,
            // afterwards it holds the four gates of row i0 + g.
            float v[4] = {P[i0], P[i0 + 1], P[i0 + 2], P[i0 + 3]};
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                if (jj & m) continue;
                const bool up = (g & m) != 0;
                const float r = __shfl_xor_sync(0xffffffffu, up ? v[jj] : v[jj + m], m);
                if (up) v[jj] = r;
                else v[jj + m] = r;
              }
            }
            const int ri = ibase + i0 + g;  // this lane's row among the warp half's HR
            const float ff1 = fmaf(2.f, sigmoid_fast(2.f * v[0]), -1.f);
            const float ff2 = fmaf(2.f, sigmoid_fast(2.f * v[1]), -1.f);
            const float gt = sigmoid_fast(fmaf(v[2], tsr[ri], v[3]));
            const float h = ff1 * (1.f - gt) + gt * ff2;
            if (defer) {
              const int j = i0 >> 2;
              dfo[j] = ri < nvalid;
              dfv[j][0] = h; dfv[j][1] = ff1; dfv[j][2] = ff2; dfv[j][3] = gt;
              dfh[j] = ho + static_cast<size_t>(ri) * C;
              dfc[j] = co + static_cast<size_t>(ri) * 3 * C;
            } else if (ri < nvalid) {
              const size_t hi = ho + static_cast<size_t>(ri) * C;
              const size_t ci = co + static_cast<size_t>(ri) * 3 * C;
              if constexpr (obf) {
                __nv_bfloat16* hb16 = reinterpret_cast<__nv_bfloat16*>(p.H);
                __nv_bfloat16* cb16 = reinterpret_cast<__nv_bfloat16*>(p.cache);
                hb16[hi] = __float2bfloat16_rn(h);
                cb16[ci] = __float2bfloat16_rn(ff1);
                cb16[ci + C] = __float2bfloat16_rn(ff2);
                cb16[ci + 2 * C] = __float2bfloat16_rn(gt);
              } else {
                p.H[hi] = h;
                p.cache[ci] = ff1;
                p.cache[ci + C] = ff2;
                p.cache[ci + 2 * C] = gt;
              }
            }
            const Split2 sp = split2(h);
            const uint32_t off = hterm_offset<NR>(HR * hh + ri, ch);
            uint8_t* dst = hb + off;
            *reinterpret_cast<__half*>(dst) = sp.t[0];
            *reinterpret_cast<__half*>(dst + S::TERM) = sp.t[1];
            if (t + 1 < K) {
              __stcg(reinterpret_cast<unsigned short*>(xs + off), __half_as_ushort(sp.t[0]));
              __stcg(reinterpret_cast<unsigned short*>(xs + off + S::SLAB),
                     __half_as_ushort(sp.t[1]));
            }
          }
        };
#pragma unroll
        for (int cc = 0; cc < HR / 16; ++cc) {
          float P[16];
          tmem_ld16(dq + 16 * cc, P);
          rows(P, 16 * cc, 16, false);
        }
        if constexpr (HR % 16 == 8) {
          float P[16];
          float P8[8];
          tmem_ld8(dq + HR - 8, P8);
#pragma unroll
          for (int i = 0; i < 8; ++i) P[i] = P8[i];
#pragma unroll
          for (int i = 8; i < 16; ++i) P[i] = 0.f;
          rows(P, HR - 8, 8, true);
        }
      }
      fence_proxy_async_smem();  // h_t's terms -> visible to the MMAs
      tc_fence_before_sync();    // tensor-memory loads done before the next step's MMAs
      if (t + 1 < K) {
        fence_acq_rel_gpu();     // h_t's terms in L2 before the announcements below
        __syncwarp();
        // This warp's part of h_t: in the own slab (lane 0), in L2 for every other CTA.
        if (lane == 0) mbar_arrive(full0 + 8u * rank);
        else if (lane < CS)
          mbar_arrive_remote(
              map_to_rank(ready0 + 8u * (((t + 1) & 1) * CS + rank), (rank + lane) % CS));
        if constexpr (FU) {
          // u_{t+1} (in registers) -> the u operand (the MMAs of step t that read it are done:
          // `done` was waited above); then the loads of u_{t+2}.
          store_u();
          if (t + 2 < K) load_u(t + 2);
          fence_proxy_async_smem();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(ufull);
        } else {
          load_x(t + 1);  // in flight while the exchange and the next step's MMAs run
        }
        load_ts(t + 1);
      }
      if constexpr (HR % 16 == 8) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (dfo[j]) {
            if constexpr (obf) {
              __nv_bfloat16* hb16 = reinterpret_cast<__nv_bfloat16*>(p.H);
              __nv_bfloat16* cb16 = reinterpret_cast<__nv_bfloat16*>(p.cache);
              hb16[dfh[j]] = __float2bfloat16_rn(dfv[j][0]);
              cb16[dfc[j]] = __float2bfloat16_rn(dfv[j][1]);
              cb16[dfc[j] + C] = __float2bfloat16_rn(dfv[j][2]);
              cb16[dfc[j] + 2 * C] = __float2bfloat16_rn(dfv[j][3]);
            } else {
              p.H[dfh[j]] = dfv[j][0];
              p.cache[dfc[j]] = dfv[j][1];
              p.cache[dfc[j] + C] = dfv[j][2];
              p.cache[dfc[j] + 2 * C] = dfv[j][3];
            }
          }
      }
    }
  }

  // Leave together: no CTA exits while another may still address its shared memory or arrive
  // on its barriers.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == kCtlWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int CS, int NR>
cudaError_t prepare_k(int* max_active) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  // The fused form needs the most shared memory; the occupancy asked for is its.
  const int smem = TcShape<CS, NR, false>::SMEM, smem_fu = TcShape<CS, NR, true>::SMEM;
  if (smem_fu > optin) {
    *max_active = 0;
    return cudaSuccess;
  }
  for (auto* k : {cfc_fwd_tc_kernel<CS, NR, false, false>, cfc_fwd_tc_kernel<CS, NR, true, false>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  for (auto* k : {cfc_fwd_tc_kernel<CS, NR, false, true>, cfc_fwd_tc_kernel<CS, NR, true, true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_fu);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_fu;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_active, cfc_fwd_tc_kernel<CS, NR, false, true>, &cfg);
}

template <int CS, int NR>
cudaError_t launch_k(const FwdParams& p, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3(((p.B + NR - 1) / NR) * CS, 1, 1);
  c.block = dim3(kTcThreads, 1, 1);
  const bool fuse = p.u != nullptr;
  c.smem = fuse ? TcShape<CS, NR, true>::SMEM : TcShape<CS, NR, false>::SMEM;
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(CS, 1, 1);
  if (fuse)
    return p.out_bf16 ? launch(c, cfc_fwd_tc_kernel<CS, NR, true, true>, p)
                      : launch(c, cfc_fwd_tc_kernel<CS, NR, false, true>, p);
  return p.out_bf16 ? launch(c, cfc_fwd_tc_kernel<CS, NR, true, false>, p)
                    : launch(c, cfc_fwd_tc_kernel<CS, NR, false, false>, p);
}

}  // namespace

bool fwd_tc_supported(int C) { return C == 4 * kFwdChanPerCta || C == 8 * kFwdChanPerCta; }

// Two step parities x clusters x CTAs x one slot (both terms of a CTA's slab): 8 C bytes per
// row of the padded batch, for whichever row tile (128 or 144) the launch takes.
size_t fwd_tc_xch_bytes(int B, int C) {
  const size_t r128 = static_cast<size_t>((B + 127) / 128) * 128;
  const size_t r144 = static_cast<size_t>((B + 143) / 144) * 144;
  return 8 * static_cast<size_t>(C) * (r128 > r144 ? r128 : r144);
}

// `rows`: batch rows per cluster, 128 or 144 (FwdParams::R at launch).
cudaError_t fwd_tc_prepare(int C, int rows, int* max_active_clusters) {
  if (C == 4 * kFwdChanPerCta)
    return rows == 144 ? prepare_k<4, 144>(max_active_clusters) : prepare_k<4, 128>(max_active_clusters);
  if (C == 8 * kFwdChanPerCta)
    return rows == 144 ? prepare_k<8, 144>(max_active_clusters) : prepare_k<8, 128>(max_active_clusters);
  return cudaErrorInvalidValue;
}

cudaError_t fwd_tc_launch(const FwdParams& p, cudaStream_t s, bool pdl) {
  if (p.C == 4 * kFwdChanPerCta)
    return p.R == 144 ? launch_k<4, 144>(p, s, pdl) : launch_k<4, 128>(p, s, pdl);
  if (p.C == 8 * kFwdChanPerCta)
    return p.R == 144 ? launch_k<8, 144>(p, s, pdl) : launch_k<8, 128>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace cfc
