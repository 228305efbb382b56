// cfc_contract.cu -- the backward pass's two dense contractions over the B*K rows, fed by TMA:
//
//   dW[m][n] = sum_{r < B*K} d_pre[r][m] * z[r][n],   m < 4C, n <= n_in (z[r][n_in] = 1: db)
//   du[r][k] = sum_{m < 4C}  d_pre[r][m] * W[m][k],   k < n_x
//
// z[r] = [u[r] ; h_{r-B} ; 1] with h_{r-B} = h0[r] for the first B rows.  The DQN plan on page
// "H100 Epoch Optimization Phase 2" (Task 2) replaces per-sample atomic weight-gradient
// accumulation by one GEMM over the batch, "dW = dY^T X"; here the sum runs over batch and time.
//
// Operand forms (the weight-gradient mode):
//   accurate  every fp32 operand x is held as two bf16 planes, hi = bf16(x) and
//             lo = bf16(x - hi) (16 significand bits), and a tile product is hi*hi + hi*lo +
//             lo*hi: three tcgen05.mma kind::f16 per 16-deep step, fp32 accumulation in tensor
//             memory; the dropped terms are below 2^-16 of the product;
//   bf16      the hi plane alone, one MMA per step (relative error ~2^-9 per product);
//   tf32      the fp32 operands, tcgen05.mma kind::tf32 (10 explicit mantissa bits).  This
//             form reads every operand K-major: the weight gradient takes transposed copies of
//             d_pre and z (transpose_kernel), since the layout the tensor cores want for
//             MN-major 32-bit operands differs from the 16-bit one used here.
// The planes are written by the producers: d_pre's by the BPTT recurrence (or the split kernel
// below), z's and W_u^T's by build_operands_kernel.  So the contraction itself converts
// nothing: every operand tile arrives by a 2-D TMA copy (128-byte swizzle) in the layout the
// tensor cores read, and out-of-range rows and columns arrive as zeros from the copy itself.
//
// Layouts.  The weight gradient reduces over the rows r of d_pre [r][m] and z [r][n], so both
// of its operands are MN-major (the output index is the contiguous one); the input gradient
// reduces over m, the contiguous index of d_pre, and its operands are K-major.  A 128-byte
// swizzle atom is 8 rows of 128 bytes (64 bf16 or 32 fp32); a K-major tile stacks atoms along
// the output index (8 rows each), an MN-major tile stacks them along the reduction index, one
// column of atoms per 128 bytes of output index.
//
// Roles (one CTA = one output tile over one range of the reduction): warp 8 lane 0 issues the
// TMA copies of each stage, warp 9 lane 0 issues the MMAs and commits each stage back, warps
// 0-7 read the accumulators (tcgen05.ld) once the last MMA has completed and store them.  When
// there are fewer output tiles than SMs the reduction is split and reduce_axis0 sums the split
// partials in order (the split depends only on the sizes, so results are bitwise
// reproducible).
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kCEpiWarps = 8;
constexpr int kCThreads = (kCEpiWarps + 2) * 32;  // + TMA warp + MMA warp
constexpr int kCMaxStages = 8;
constexpr int kAtomBytes = 128;                   // bytes of one swizzle-atom row

// Elements of the operand type per 128-byte atom row.
template <int FORM>
struct Form {
  static constexpr int kElem = FORM == kFormTf32 ? 4 : 2;
  static constexpr int kAtom = kAtomBytes / kElem;          // 64 bf16 or 32 fp32
  static constexpr int kTerms = FORM == kFormBf16x2 ? 2 : 1;
  static constexpr int kKStep = FORM == kFormTf32 ? 8 : 16;  // reduction depth of one MMA
};

struct CArgs {
  int M, N;             // rows and columns of the result
  int n_tile;           // columns of a tile
  int m_tiles, n_tiles;
  int n_kb;             // k-blocks of the reduction (kd entries each)
  int kd;               // reduction entries per k-block: a multiple of 16 for MN-major
                        // tiles, the atom row (kAtom) for K-major ones
  int kb_per_split;
  int stages;
  float* out;           // [splits][M][ldo] (split_stride floats apart)
  int ldo, n_store;     // row pitch of out; columns stored per row (< N allowed)
  size_t split_stride;
  int* status;
  // 0: wait for the previous kernel before any copy, then release dependents.  1: the operands
  // are known to be complete when this kernel starts (the previous kernel released its
  // dependents only after its own wait); release dependents at once and wait for the previous
  // kernel only at the end, so this kernel runs beside it and its completion still implies the
  // previous kernel's.
  int defer_wait;
};

// TMA: a 2-D tile of `tmap` at (x, y) (x: the contiguous index) into shared memory at `dst`,
// completing as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Shared-memory matrix descriptor of an MN-major operand in 128-byte-swizzled atoms: `lbo` is
// the byte distance between atoms along the output index, `sbo` between groups of 8 reduction
// rows (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator, A / B of the form's type, MN-major flags, M x N.
template <int FORM>
__host__ __device__ constexpr uint32_t idesc_form(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) |                                    // D: fp32
         ((FORM == kFormTf32 ? 2u : 1u) << 7) |         // A: tf32 (kind::tf32) or bf16
         ((FORM == kFormTf32 ? 2u : 1u) << 10) |        // B: likewise
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <int FORM>
__device__ __forceinline__ void umma_form(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (FORM == kFormTf32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
  }
}

// One CTA: output tile `tile` (m-tile fastest) over the reduction blocks of split `split`.
// Maps: a0 / b0 the hi planes (or the fp32 operands), a1 / b1 the lo planes (accurate form).
template <int FORM, bool A_MN, bool B_MN, int MT>
__global__ void __launch_bounds__(kCThreads, 1)
    contract_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                    const __grid_constant__ CUtensorMap b0, const __grid_constant__ CUtensorMap b1,
                    const CArgs g) {
  using F = Form<FORM>;
  constexpr int kTerms = F::kTerms;
  // Reduction entries of one stage: MN-major tiles take g.kd rows of 128-byte atoms, K-major
  // tiles one atom row (the swizzle width) per output row.
  const int kd = A_MN ? g.kd : F::kAtom;
  const uint32_t rb = static_cast<uint32_t>(kd) * F::kElem;  // bytes per output index
  const uint32_t kABytes = MT * 128 * rb;                    // one term of A: MT*128 outputs
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(base);
  const uint32_t b_bytes = static_cast<uint32_t>(g.n_tile) * rb;
  const uint32_t stage_bytes = kTerms * (kABytes + b_bytes);
  const int stages = g.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + stages * stage_bytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kCMaxStages + 1);
  const uint32_t full0 = smem_addr(&bars[0]);
  const uint32_t empty0 = smem_addr(&bars[kCMaxStages]);
  const uint32_t accb = smem_addr(&bars[2 * kCMaxStages]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles = g.m_tiles * g.n_tiles;
  const int tile = blockIdx.x % tiles, split = blockIdx.x / tiles;
  const int m0 = (tile % g.m_tiles) * (MT * 128);
  const int n0 = (tile / g.m_tiles) * g.n_tile;
  const int kb0 = split * g.kb_per_split;
  const int nk = min(g.kb_per_split, g.n_kb - kb0);
  uint32_t acc_cols = 32;
  while (acc_cols < static_cast<uint32_t>(g.n_tile)) acc_cols <<= 1;
  const uint32_t ncols = acc_cols * MT;

  if (g.defer_wait) grid_dep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(accb, 1);
    fence_mbar_init_cluster();
  }
  if (warp == kCEpiWarps && lane == 0) {
    tma_prefetch_desc(&a0);
    tma_prefetch_desc(&b0);
  }
  // The operands come from the previous kernels; tensor memory is taken only after they have
  // finished, so this kernel never waits for columns a running predecessor holds.  (With a
  // deferred wait the predecessor holds no tensor memory: it is the weight-gradient contraction,
  // whose CTAs leave no room on their SM for this one's shared memory, or the columns it holds
  // leave room for these.)
  if (!g.defer_wait) {
    grid_dep_wait();
    grid_dep_launch_dependents();
  }
  if (warp == kCEpiWarps) {
    tmem_alloc(smem_addr(tslot), ncols);
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kCEpiWarps) {
    if (lane == 0) {
      // ---- TMA producer ----
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % stages;
        if (i >= stages) ok = mbar_wait_bounded_cta(empty0 + 8u * s, (i / stages - 1) & 1, g.status);
        if (!ok) break;
        const uint32_t bar = full0 + 8u * s;
        mbar_arrive_expect_tx(bar, stage_bytes);
        const uint32_t st = sbase + s * stage_bytes;
        const int kb = kb0 + i;
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
          const CUtensorMap* ma = t == 0 ? &a0 : &a1;
          const CUtensorMap* mb = t == 0 ? &b0 : &b1;
          const uint32_t sa = st + t * kABytes;
          const uint32_t sb = st + kTerms * kABytes + t * b_bytes;
          if constexpr (A_MN) {
            // box {kAtom outputs, kd reduction rows}: one atom column per box
#pragma unroll
            for (int a = 0; a < MT * 128 / F::kAtom; ++a)
              tma_load_2d(sa + a * (kd * kAtomBytes), ma, m0 + a * F::kAtom, kb * kd, bar);
          } else {
            tma_load_2d(sa, ma, kb * F::kAtom, m0, bar);  // box {kAtom, MT*128 rows}
          }
          if constexpr (B_MN) {
            for (int a = 0; a < g.n_tile / F::kAtom; ++a)
              tma_load_2d(sb + a * (kd * kAtomBytes), mb, n0 + a * F::kAtom, kb * kd, bar);
          } else {
            tma_load_2d(sb, mb, kb * F::kAtom, n0, bar);  // box {kAtom, n_tile rows}
          }
        }
        ++issued;
      }
      // After an early stop no copy into this CTA's shared memory may still be in flight when
      // it exits (copies from global memory always complete).
      if (!ok)
        for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
          (void)mbar_wait_bounded_cta(full0 + 8u * (i % stages), (i / stages) & 1, g.status);
    }
  } else if (warp == kCEpiWarps + 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      const uint32_t idesc = idesc_form<FORM>(128, g.n_tile, A_MN, B_MN);
      // MN-major: atoms along the output index are kd reduction rows x 128 B apart, groups
      // of 8 reduction rows 1024 B apart; one MMA step spans kKStep / 8 groups.
      const uint32_t kLbo = static_cast<uint32_t>(kd) * kAtomBytes;
      constexpr uint32_t kSbo = 1024;
      const int ksteps = kd / F::kKStep;
      constexpr uint32_t kMnStep = (F::kKStep / 8) * 1024;
      constexpr uint32_t kKStepBytes = F::kKStep * F::kElem;  // K-major: 32 B per step
      uint32_t acc = 0;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int s = i % stages;
        ok = mbar_wait_bounded_cta(full0 + 8u * s, (i / stages) & 1, g.status);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t st = sbase + s * stage_bytes;
        const uint32_t sb = st + kTerms * kABytes;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t d = tmem + mt * acc_cols;
          const uint32_t sa = st + mt * (128 * rb);
#pragma unroll 4
          for (int j = 0; j < ksteps; ++j) {
            uint64_t ad[kTerms], bd[kTerms];
#pragma unroll
            for (int t = 0; t < kTerms; ++t) {
              ad[t] = A_MN ? desc_mn_sw128(sa + t * kABytes + j * kMnStep, kLbo, kSbo)
                           : umma_desc_sw128(sa + t * kABytes + j * kKStepBytes);
              bd[t] = B_MN ? desc_mn_sw128(sb + t * b_bytes + j * kMnStep, kLbo, kSbo)
                           : umma_desc_sw128(sb + t * b_bytes + j * kKStepBytes);
            }
            const uint32_t first = (i == 0 && j == 0) ? acc : 1u;
            umma_form<FORM>(d, ad[0], bd[0], idesc, first);
            if constexpr (kTerms == 2) {
              umma_form<FORM>(d, ad[0], bd[1], idesc, 1);  // hi * lo
              umma_form<FORM>(d, ad[1], bd[0], idesc, 1);  // lo * hi
            }
          }
        }
        umma_commit(empty0 + 8u * s);  // the stage may be refilled once these MMAs are done
      }
      umma_commit(accb);
      // The MMAs issued here finish before tensor memory is freed, whatever the other roles
      // did: they depend on nothing outside this CTA.
      (void)mbar_wait_bounded_cta(accb, 0, g.status);
    }
  } else {
    // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) ..; warps w and w + 4 take
    // alternate 16-column chunks ----
    bool ok = mbar_wait_bounded_cta(accb, 0, g.status);
    tc_fence_after_sync();
    const int q = warp & 3, h = warp >> 2;
    const bool vec = (g.ldo % 4) == 0;
    float* outs = g.out + static_cast<size_t>(split) * g.split_stride;
#pragma unroll 1
    for (int mt = 0; mt < MT; ++mt) {
      const int m = m0 + mt * 128 + 32 * q + lane;
      float* orow = outs + static_cast<size_t>(m) * g.ldo;
#pragma unroll 1
      for (int c0 = 16 * h; c0 < g.n_tile; c0 += 32) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + mt * acc_cols + c0, v);
        if (!ok || m >= g.M) continue;
        const int n = n0 + c0;
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
          const int nc = n + c;
          if (vec && nc + 3 < g.n_store) {
            *reinterpret_cast<float4*>(orow + nc) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (nc + e < g.n_store) orow[nc + e] = v[c + e];
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kCEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, ncols);
  }
  if (g.defer_wait) grid_dep_wait();
}

// ---- operand producers -------------------------------------------------------------------

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Eight consecutive values of one operand row -> their 16-byte hi chunk (and lo chunk, `pitch`
// elements further on) at element `col` of the row starting at `row` (bf16 forms), or two
// 16-byte fp32 chunks (tf32; `col` then counts floats).
template <int FORM>
__device__ __forceinline__ void put8(uint8_t* row, int pitch, int col, const float (&v)[8]) {
  if constexpr (FORM == kFormTf32) {
    float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(row) + col);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    __nv_bfloat16 h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) split_bf16(v[e], h[e], l[e]);
    __nv_bfloat16* r16 = reinterpret_cast<__nv_bfloat16*>(row);
    *reinterpret_cast<uint4*>(r16 + col) =
        make_uint4(pack2(h[0], h[1]), pack2(h[2], h[3]), pack2(h[4], h[5]), pack2(h[6], h[7]));
    if constexpr (FORM == kFormBf16x2)
      *reinterpret_cast<uint4*>(r16 + pitch + col) =
          make_uint4(pack2(l[0], l[1]), pack2(l[2], l[3]), pack2(l[4], l[5]), pack2(l[6], l[7]));
  }
}

// z rows [u ; h_{t-1} ; 1] (h_{-1} = h0) and W_u^T rows (wt[k][m] = W[m][k]) in the operand form,
// eight columns per item.  Columns past the valid ones are written as zeros up to the next
// multiple of 8 (the pitches are multiples of 8); the contraction never reads beyond them.
// HB: H holds bf16 elements.
template <int FORM, bool HB>
__global__ void __launch_bounds__(1024)
    build_operands_kernel(const float* __restrict__ u, const void* __restrict__ H,
                          const float* __restrict__ h0, const float* __restrict__ W, int B,
                          int BK, int C, int n_x, int M, uint8_t* z, int zp, uint8_t* wt,
                          int mp) {
  // u, H, h0 and W are complete when this kernel starts: it follows either nothing of the same
  // call, or a kernel that releases its dependents only after its own dependency wait (the
  // BPTT recurrence, the d_pre split).  So the build runs beside that kernel and waits for it
  // only at the end, which keeps "this kernel complete" implying "every earlier kernel
  // complete" for the contractions that wait on it.
  grid_dep_launch_dependents();
  const int n_in = n_x + C, zn = n_in + 1;  // M: the W rows (gate rows) of W_u^T
  const int zg = (zn + 7) / 8, wg = (M + 7) / 8;  // 8-column groups per row
  const long long z_items = static_cast<long long>(BK) * zg;
  const long long total = z_items + static_cast<long long>(n_x) * wg;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // Whole 16-byte loads when u's and H's rows start on 16 bytes (n_x, C multiples of 4): an
  // item of 8 columns then lies wholly in u, wholly in h, or straddles the end of a region.
  const bool vec = (n_x & 3) == 0 && (C & 3) == 0;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += stride) {
    float v[8];
    if (i < z_items) {
      const int r = static_cast<int>(i / zg), c0 = 8 * static_cast<int>(i - static_cast<long long>(r) * zg);
      // h_{t-1}: h0 for the first step, else the previous step's row of H (fp32 or bf16).
      const float* hrow = r < B ? h0 + static_cast<size_t>(r) * C
                                : static_cast<const float*>(H) + static_cast<size_t>(r - B) * C;
      const bool in_u = c0 + 8 <= n_x, in_h = c0 >= n_x && c0 + 8 <= n_in;
      if (vec && in_u) {
        const float4* src = reinterpret_cast<const float4*>(u + static_cast<size_t>(r) * n_x + c0);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else if (vec && in_h && (!HB || r < B)) {
        const float4* src = reinterpret_cast<const float4*>(hrow + (c0 - n_x));
        const float4 a = __ldg(src), b = __ldg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else if (HB && vec && in_h && (C & 7) == 0 && (n_x & 7) == 0) {
        // Eight bf16 values of H: one 16-byte load (the row start and c0 - n_x are multiples
        // of 8 elements).
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(H) + static_cast<size_t>(r - B) * C + (c0 - n_x)));
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = __uint_as_float(q[e] << 16);
          v[2 * e + 1] = __uint_as_float(q[e] & 0xFFFF0000u);
        }
      } else if constexpr (HB) {
        const __nv_bfloat16* hrow16 =
            static_cast<const __nv_bfloat16*>(H) + static_cast<size_t>(r < B ? 0 : r - B) * C;
        const bool from_h0 = r < B;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int n = c0 + e;
          v[e] = n < n_x ? __ldg(u + static_cast<size_t>(r) * n_x + n)
               : n < n_in ? (from_h0 ? __ldg(hrow + (n - n_x)) : __bfloat162float(hrow16[n - n_x]))
               : n == n_in ? 1.f : 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int n = c0 + e;
          v[e] = n < n_x ? __ldg(u + static_cast<size_t>(r) * n_x + n)
               : n < n_in ? __ldg(hrow + (n - n_x))
               : n == n_in ? 1.f : 0.f;
        }
      }
      put8<FORM>(z + static_cast<size_t>(r) * 4 * zp, zp, c0, v);
    } else {
      const long long j = i - z_items;
      const int k = static_cast<int>(j / wg), m0 = 8 * static_cast<int>(j - static_cast<long long>(k) * wg);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = m0 + e < M ? __ldg(W + static_cast<size_t>(m0 + e) * n_in + k) : 0.f;
      put8<FORM>(wt + static_cast<size_t>(k) * 4 * mp, mp, m0, v);
    }
  }
  grid_dep_wait();
}

// fp32 d_pre rows [BK][M] -> bf16 operand rows (pitch mp, 4 mp bytes per row).  One warp per
// row reads the whole row into registers before any lane writes, so the split may run in place
// when a row's operand bytes are its fp32 bytes (mp == M): every row is rewritten from its own
// values only.
template <int FORM>
__global__ void split_dpre_kernel(const float* d_pre, int BK, int M, int mp, uint8_t* planes) {
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int groups = (M + 7) / 8;  // 8-value groups of a row (M is a multiple of 4)
  constexpr int kMaxPerLane = (4 * kMaxChannels / 8 + 31) / 32;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < BK; r += warps) {
    const float* src = d_pre + static_cast<size_t>(r) * M;
    float v[kMaxPerLane][8];
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int c0 = 8 * (lane + 32 * q);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[q][e] = c0 + e < M ? src[c0 + e] : 0.f;
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int g = lane + 32 * q;
      if (g < groups) put8<FORM>(planes + static_cast<size_t>(r) * 4 * mp, mp, 8 * g, v[q]);
    }
    __syncwarp();
  }
}

// dst[c][r] = src[r][c] for r < rows, c < cols (fp32; src rows `sp` floats apart, dst rows
// `dp` floats apart), through 32 x 32 shared-memory tiles so both sides are coalesced.
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ src, int rows,
                                                        int cols, int sp, float* __restrict__ dst,
                                                        int dp) {
  __shared__ float tile[32][33];
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int r = r0 + ty + k, c = c0 + tx;
    tile[ty + k][tx] = (r < rows && c < cols) ? src[static_cast<size_t>(r) * sp + c] : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 32; k += 8) {
    const int c = c0 + ty + k, r = r0 + tx;
    if (c < cols && r < rows) dst[static_cast<size_t>(c) * dp + r] = tile[tx][ty + k];
  }
}

// ---- host side -----------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// 2-D tensor map over rows of `inner` valid elements, `row_bytes` apart; box {box_inner,
// box_outer}; 128-byte swizzle; reads outside [inner) x [outer) return zeros.
cudaError_t make_map(CUtensorMap* m, bool f32, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int atom_of(int form) { return form == kFormTf32 ? 32 : 64; }
int terms_of(int form) { return form == kFormBf16x2 ? 2 : 1; }

template <int FORM, bool A_MN, bool B_MN, int MT>
cudaError_t launch_contract(const ContractPlan& pl, const CUtensorMap& a0, const CUtensorMap& a1,
                            const CUtensorMap& b0, const CUtensorMap& b1, const CArgs& g,
                            cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3(pl.m_tiles * pl.n_tiles * pl.splits, 1, 1);
  c.block = dim3(kCThreads, 1, 1);
  c.smem = pl.smem;
  c.stream = s;
  c.pdl = pdl;
  return launch(c, contract_kernel<FORM, A_MN, B_MN, MT>, a0, a1, b0, b1, g);
}

// The kernels each form launches: bf16 forms read the weight gradient's operands MN-major,
// tf32 reads everything K-major.
template <int FORM>
cudaError_t set_attrs_form(int max_smem) {
  constexpr bool mn = FORM != kFormTf32;
  const void* k[] = {reinterpret_cast<const void*>(contract_kernel<FORM, mn, mn, 1>),
                     reinterpret_cast<const void*>(contract_kernel<FORM, mn, mn, 2>),
                     reinterpret_cast<const void*>(contract_kernel<FORM, false, false, 1>)};
  for (const void* f : k) {
    const cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Bytes of one stage: `rb` bytes per output index (kd entries of an MN-major tile, or one
// 128-byte atom row of a K-major one).
size_t stage_bytes(int form, int mt, int n_tile, int rb) {
  return static_cast<size_t>(terms_of(form)) * (mt * 128 + n_tile) * rb;
}

int row_bytes(int form, int kd, bool mn) {
  return mn ? kd * (form == kFormTf32 ? 4 : 2) : kAtomBytes;
}

// Stages: as many as fit (at most `max_stages`), leaving room for alignment and barriers.
ContractPlan finish_plan(ContractPlan p, int form, int max_stages, int smem_budget, bool mn) {
  const size_t sb = stage_bytes(form, p.mt, p.n_tile, row_bytes(form, p.kd, mn));
  const size_t extra = 1024 + (2 * kCMaxStages + 2) * 8 + 16;
  int st = static_cast<int>((smem_budget - extra) / sb);
  if (st > max_stages) st = max_stages;
  if (st > kCMaxStages) st = kCMaxStages;
  p.stages = st;
  p.smem = st * sb + extra;
  return p;
}

}  // namespace

int contract_z_pitch(int n_in, int form) {
  (void)form;
  return (n_in + 1 + 7) & ~7;
}
int contract_m_pitch(int C, int form) {
  return form == kFormTf32 ? 4 * C : (4 * C + 7) & ~7;  // tf32: the fp32 d_pre rows as written
}
int contract_wt_pitch(int C) { return (4 * C + 7) & ~7; }

// Weight gradient: rows 4C, columns n_in + 1 (the last is db), reduction B*K.  Column tiles are
// whole atoms (MN-major B), at most 256 wide; two 128-row accumulators per CTA when there are
// enough rows, so each z tile feeds 256 rows of the result.  The reduction is split so the
// CTAs fill about one wave of a fixed 148 (a constant, not the device's SM count: the split,
// hence the summation order, depends only on the sizes).
ContractPlan dw_contract_plan(int B, int K, int C, int n_x, int form, int smem_budget) {
  return dw_contract_plan_mn(B * K, 4 * C, n_x + C + 1, form, smem_budget);
}

// Rows (B*K) below which both contractions are split, sized together: a tiny problem is all
// latency, so more and shorter CTAs help, and one launch merges both sets of partials.
constexpr int kJointSplitMaxRows = 8192;
// Reduction rows per stage of the MN-major (bf16) weight gradient above that size: 32 rows
// give twice the stages of 64 in the same shared memory (four of 56 KB at 256 x 192 tiles,
// accurate form), so each stage's copy has three stages of MMAs to land behind.
constexpr int kMnDeepKd = 32;

ContractPlan dw_contract_plan_mn(int BK, int M, int N, int form, int smem_budget) {
  ContractPlan p{};
  // Column tiles: whole 128-byte atoms for MN-major operands (bf16), multiples of 16 (K-major).
  const int atom = form == kFormTf32 ? 16 : atom_of(form);
  p.mt = M >= 256 ? 2 : 1;
  p.n_tiles = (N + 255) / 256;
  int nt = (N + p.n_tiles - 1) / p.n_tiles;
  p.n_tile = (nt + atom - 1) / atom * atom;
  if (p.n_tile > 256) {  // a whole number of atoms per tile may need one more tile
    ++p.n_tiles;
    nt = (N + p.n_tiles - 1) / p.n_tiles;
    p.n_tile = (nt + atom - 1) / atom * atom;
  }
  const bool mn = form != kFormTf32;
  p.kd = mn && BK >= kJointSplitMaxRows ? kMnDeepKd : atom_of(form);
  // Two stages of two accumulators must fit; otherwise one accumulator per CTA.
  if (p.mt == 2 &&
      2 * stage_bytes(form, 2, p.n_tile, row_bytes(form, p.kd, mn)) + 2048 >
          static_cast<size_t>(smem_budget))
    p.mt = 1;
  p.m_tiles = (M + 128 * p.mt - 1) / (128 * p.mt);
  p.n_kb = (BK + p.kd - 1) / p.kd;
  const int tiles = p.m_tiles * p.n_tiles;
  // At least four k-blocks per split: the copies of a CTA's blocks are in flight together, so
  // a longer range costs little, and every split adds a partial block to the merge.
  int s0 = tiles < 148 ? 148 / tiles : 1;
  if (s0 > (p.n_kb + 3) / 4) s0 = (p.n_kb + 3) / 4;
  if (s0 < 1) s0 = 1;
  p.kb_per_split = (p.n_kb + s0 - 1) / s0;
  p.splits = (p.n_kb + p.kb_per_split - 1) / p.kb_per_split;
  return finish_plan(p, form, 8, smem_budget, mn);
}

// Input gradient: rows B*K, columns n_x, reduction 4C; one 128-row tile per CTA, not split.
// At most two stages' worth of shared memory per CTA, so two CTAs share an SM and one's set-up
// and stores overlap the other's copies.
ContractPlan du_contract_plan(int B, int K, int C, int n_x, int form, int smem_budget) {
  return du_contract_plan_mn(B * K, 4 * C, n_x, form, smem_budget);
}

ContractPlan du_contract_plan_mn(int BK, int M, int n_x, int form, int smem_budget) {
  ContractPlan p{};
  const int atom = atom_of(form);
  p.mt = 1;
  p.n_tiles = (n_x + 255) / 256;
  const int nt = (n_x + p.n_tiles - 1) / p.n_tiles;
  p.n_tile = (nt + 15) / 16 * 16;
  p.m_tiles = (BK + 127) / 128;
  p.kd = atom;
  p.n_kb = (M + atom - 1) / atom;
  p.kb_per_split = p.n_kb;
  p.splits = 1;
  return finish_plan(p, form, 4, smem_budget / 2 - 1024, false);
}


void contract_plans(int B, int K, int C, int n_x, int form, int smem_budget, ContractPlan* pw,
                    ContractPlan* pu) {
  contract_plans_mn(B * K, 4 * C, n_x + C + 1, n_x, form, smem_budget, pw, pu);
}

void contract_plans_mn(int BK, int M, int N, int n_x, int form, int smem_budget, ContractPlan* pw,
                       ContractPlan* pu) {
  *pw = dw_contract_plan_mn(BK, M, N, form, smem_budget);
  *pu = du_contract_plan_mn(BK, M, n_x, form, smem_budget);
  if (BK >= kJointSplitMaxRows) return;
  // One 128-row accumulator per dW CTA, and the smallest common k-blocks-per-split whose CTAs
  // fit a fixed budget of one wave (a constant, not the device's SM count: the splits, hence
  // the summation orders, depend only on the sizes).
  constexpr int kBudget = 148;
  ContractPlan w = *pw;
  w.mt = 1;
  w.m_tiles = (M + 127) / 128;
  const int tw = w.m_tiles * w.n_tiles, tu = pu->m_tiles * pu->n_tiles;
  int kbps = 1;
  const int kmax = w.n_kb > pu->n_kb ? w.n_kb : pu->n_kb;
  while (kbps < kmax &&
         tw * ((w.n_kb + kbps - 1) / kbps) + tu * ((pu->n_kb + kbps - 1) / kbps) > kBudget)
    ++kbps;
  for (ContractPlan* p : {&w, pu}) {
    p->kb_per_split = kbps < p->n_kb ? kbps : p->n_kb;
    p->splits = (p->n_kb + p->kb_per_split - 1) / p->kb_per_split;
  }
  *pw = finish_plan(w, form, 8, smem_budget, form != kFormTf32);
}

cudaError_t contract_prepare(int max_smem) {
  cudaError_t e = set_attrs_form<kFormBf16x2>(max_smem);
  if (e == cudaSuccess) e = set_attrs_form<kFormBf16>(max_smem);
  if (e == cudaSuccess) e = set_attrs_form<kFormTf32>(max_smem);
  if (e == cudaSuccess && !encode_fn()) e = cudaErrorNotSupported;
  return e;
}

namespace {
LaunchCfg grid_stride_cfg(long long items, cudaStream_t s, bool pdl) {
  LaunchCfg c;
  const long long blocks = (items + 255) / 256;
  c.grid = dim3(static_cast<unsigned>(blocks < 148 * 16 ? (blocks > 0 ? blocks : 1) : 148 * 16), 1, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return c;
}
}  // namespace

cudaError_t build_operands_launch(int form, const float* u, const void* H, int h_bf16,
                                  const float* h0,
                                  const float* W, int B, int K, int C, int n_x, void* z, void* wt,
                                  cudaStream_t s, bool pdl, int M, int ctas) {
  const int BK = B * K;
  if (M <= 0) M = 4 * C;
  const long long items = static_cast<long long>(BK) * ((n_x + C + 1 + 7) / 8) +
                          static_cast<long long>(n_x) * ((M + 7) / 8);
  LaunchCfg c = grid_stride_cfg(items, s, pdl);
  if (c.grid.x > 2 * 148) c.grid.x = 2 * 148;  // resident beside the kernel it runs next to
  if (ctas > 0) {
    // 1024 threads at 48 registers: one CTA per SM, and none beside a CTA that holds more than
    // a quarter of the SM's registers.
    c.grid = dim3(static_cast<unsigned>(ctas), 1, 1);
    c.block = dim3(1024, 1, 1);
  }
  const int zp = contract_z_pitch(n_x + C, form), mp = (M + 7) & ~7;  // W_u^T row pitch
  uint8_t* z8 = static_cast<uint8_t*>(z);
  uint8_t* w8 = static_cast<uint8_t*>(wt);
  if (h_bf16) {  // the bf16-state backward: single-pass bf16 operands only
    if (form != kFormBf16) return cudaErrorInvalidValue;
    return launch(c, build_operands_kernel<kFormBf16, true>, u, H, h0, W, B, BK, C, n_x, M, z8, zp, w8, mp);
  }
  switch (form) {
    case kFormBf16x2:
      return launch(c, build_operands_kernel<kFormBf16x2, false>, u, H, h0, W, B, BK, C, n_x, M, z8, zp, w8, mp);
    case kFormBf16:
      return launch(c, build_operands_kernel<kFormBf16, false>, u, H, h0, W, B, BK, C, n_x, M, z8, zp, w8, mp);
    default:
      return launch(c, build_operands_kernel<kFormTf32, false>, u, H, h0, W, B, BK, C, n_x, M, z8, zp, w8, mp);
  }
}

int contract_bk_pitch(int BK) { return (BK + 3) & ~3; }

cudaError_t transpose_launch(const float* src, int rows, int cols, int sp, float* dst, int dp,
                             cudaStream_t s, bool pdl) {
  LaunchCfg c;
  c.grid = dim3((cols + 31) / 32, (rows + 31) / 32, 1);
  c.block = dim3(256, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  return launch(c, transpose_kernel, src, rows, cols, sp, dst, dp);
}

cudaError_t split_dpre_launch(int form, const float* d_pre, int BK, int C, void* planes,
                              cudaStream_t s, bool pdl) {
  const LaunchCfg c = grid_stride_cfg(32LL * BK, s, pdl);
  const int mp = contract_m_pitch(C, form);
  uint8_t* p8 = static_cast<uint8_t*>(planes);
  if (form == kFormBf16x2) return launch(c, split_dpre_kernel<kFormBf16x2>, d_pre, BK, 4 * C, mp, p8);
  return launch(c, split_dpre_kernel<kFormBf16>, d_pre, BK, 4 * C, mp, p8);
}

// dW partials [splits][4C][ldo] from the d_pre operand and z (operand rows of 4 * pitch bytes;
// the lo plane starts 2 * pitch bytes into each row).  tf32: `dpre` is d_pre^T [4C][bkp] and
// `z` is z^T [n_in + 1][bkp] (fp32, bkp = B*K rounded up to 4), both K-major.
cudaError_t dw_contract_launch(const ContractPlan& pl, int form, const void* dpre, const void* z,
                               int B, int K, int C, int n_x, float* partial, int ldo,
                               int* status, cudaStream_t s, bool pdl) {
  return dw_contract_launch_mn(pl, form, dpre, z, B * K, 4 * C, n_x + C + 1,
                               contract_m_pitch(C, form), contract_z_pitch(n_x + C, form),
                               partial, ldo, status, s, pdl);
}

cudaError_t dw_contract_launch_mn(const ContractPlan& pl, int form, const void* dpre,
                                  const void* z, int BK, int M, int N, int mp, int zp,
                                  float* partial, int ldo, int* status, cudaStream_t s,
                                  bool pdl) {
  const bool f32 = form == kFormTf32;
  const int atom = atom_of(form);
  const uint8_t* d8 = static_cast<const uint8_t*>(dpre);
  const uint8_t* z8 = static_cast<const uint8_t*>(z);
  CUtensorMap a0, a1, b0, b1;
  cudaError_t e;
  if (f32) {
    const uint64_t row = 4ull * contract_bk_pitch(BK);
    e = make_map(&a0, true, d8, BK, M, row, atom, 128 * pl.mt);
    if (e == cudaSuccess) e = make_map(&b0, true, z8, BK, N, row, atom, pl.n_tile);
  } else {
    e = make_map(&a0, false, d8, M, BK, 4ull * mp, atom, pl.kd);
    if (e == cudaSuccess) e = make_map(&b0, false, z8, N, BK, 4ull * zp, atom, pl.kd);
  }
  a1 = a0;
  b1 = b0;
  if (e == cudaSuccess && form == kFormBf16x2) {
    e = make_map(&a1, false, d8 + 2 * mp, M, BK, 4ull * mp, atom, pl.kd);
    if (e == cudaSuccess) e = make_map(&b1, false, z8 + 2 * zp, N, BK, 4ull * zp, atom, pl.kd);
  }
  if (e != cudaSuccess) return e;
  CArgs g{};
  g.M = M; g.N = N; g.n_tile = pl.n_tile; g.m_tiles = pl.m_tiles; g.n_tiles = pl.n_tiles;
  g.n_kb = pl.n_kb; g.kd = pl.kd; g.kb_per_split = pl.kb_per_split; g.stages = pl.stages;
  g.out = partial; g.ldo = ldo; g.n_store = ldo < N ? ldo : N;
  g.split_stride = static_cast<size_t>(M) * ldo;
  g.status = status;
  g.defer_wait = 0;
  switch (form * 2 + (pl.mt == 2)) {
    case kFormBf16x2 * 2: return launch_contract<kFormBf16x2, true, true, 1>(pl, a0, a1, b0, b1, g, s, pdl);
    case kFormBf16x2 * 2 + 1: return launch_contract<kFormBf16x2, true, true, 2>(pl, a0, a1, b0, b1, g, s, pdl);
    case kFormBf16 * 2: return launch_contract<kFormBf16, true, true, 1>(pl, a0, a1, b0, b1, g, s, pdl);
    case kFormBf16 * 2 + 1: return launch_contract<kFormBf16, true, true, 2>(pl, a0, a1, b0, b1, g, s, pdl);
    case kFormTf32 * 2: return launch_contract<kFormTf32, false, false, 1>(pl, a0, a1, b0, b1, g, s, pdl);
    default: return launch_contract<kFormTf32, false, false, 2>(pl, a0, a1, b0, b1, g, s, pdl);
  }
}

// du [B*K][n_x] from the d_pre operand and W_u^T.
cudaError_t du_contract_launch(const ContractPlan& pl, int form, const void* dpre, const void* wt,
                               int B, int K, int C, int n_x, float* du, int* status,
                               cudaStream_t s, bool pdl, bool defer_wait) {
  return du_contract_launch_mn(pl, form, dpre, wt, B * K, 4 * C, n_x, contract_m_pitch(C, form),
                               contract_wt_pitch(C), du, status, s, pdl, defer_wait);
}

cudaError_t du_contract_launch_mn(const ContractPlan& pl, int form, const void* dpre,
                                  const void* wt, int BK, int M, int n_x, int mp, int wp,
                                  float* du, int* status, cudaStream_t s, bool pdl,
                                  bool defer_wait) {
  const bool f32 = form == kFormTf32;
  const int atom = atom_of(form);
  const uint8_t* d8 = static_cast<const uint8_t*>(dpre);
  const uint8_t* w8 = static_cast<const uint8_t*>(wt);
  CUtensorMap a0, a1, b0, b1;
  cudaError_t e = make_map(&a0, f32, d8, M, BK, 4ull * mp, atom, 128);
  if (e == cudaSuccess) e = make_map(&b0, f32, w8, M, n_x, 4ull * wp, atom, pl.n_tile);
  a1 = a0;
  b1 = b0;
  if (e == cudaSuccess && form == kFormBf16x2) {
    e = make_map(&a1, f32, d8 + 2 * mp, M, BK, 4ull * mp, atom, 128);
    if (e == cudaSuccess) e = make_map(&b1, f32, w8 + 2 * wp, M, n_x, 4ull * wp, atom, pl.n_tile);
  }
  if (e != cudaSuccess) return e;
  CArgs g{};
  g.M = BK; g.N = n_x; g.n_tile = pl.n_tile; g.m_tiles = pl.m_tiles; g.n_tiles = pl.n_tiles;
  g.n_kb = pl.n_kb; g.kd = pl.kd; g.kb_per_split = pl.kb_per_split; g.stages = pl.stages;
  g.out = du; g.ldo = n_x; g.n_store = n_x;
  g.split_stride = static_cast<size_t>(BK) * n_x;  // split partials, when the plan splits
  g.status = status;
  g.defer_wait = defer_wait ? 1 : 0;
  switch (form) {
    case kFormBf16x2: return launch_contract<kFormBf16x2, false, false, 1>(pl, a0, a1, b0, b1, g, s, pdl);
    case kFormBf16: return launch_contract<kFormBf16, false, false, 1>(pl, a0, a1, b0, b1, g, s, pdl);
    default: return launch_contract<kFormTf32, false, false, 1>(pl, a0, a1, b0, b1, g, s, pdl);
  }
}

}  // namespace cfc
