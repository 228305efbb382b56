// cfc_gemm_tc.cu -- the input projection of the forward pass on the 5th-generation tensor cores
// (tcgen05, accumulator in tensor memory), for B*K >= 8192 rows:
//
//   X[r][n] = sum_{k < n_x} u[r][k] * W[n][k] + b[n],   r < B*K, n < 4C
//
// X does not depend on h, so it leaves the serial recurrence as one parallel contraction over
// all steps; the epilogue adds the bias and hands X to the recurrence in place (gate ff1 in H,
// gates ff2 / ta / tb in the cache).
//
// Precision: X feeds the forward, whose tolerance is 1e-5 of max|H|.  Operands are fp32; each is
// split into three bf16 terms x = hi + mid + lo (all 24 significand bits) and the tile product
// keeps hi*hi + hi*mid + mid*hi + hi*lo + lo*hi + mid*mid (six tcgen05.mma per 16-row step, fp32
// accumulation in TMEM); the dropped terms are below 2^-24 of the product.
//
// A CTA computes a 128-row x n_tile block: warps 0-7 load fp32 operand rows (coalesced), split
// them and write the bf16 terms into 128-byte-swizzled K-major tiles (64 reduction entries per
// stage; n_x <= 512 is at most eight stages); warp 8 owns the TMEM accumulator and one lane
// issues the MMAs; after the last stage the tile goes through shared memory so each warp writes
// whole row segments.
#include <cuda_bf16.h>

#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kTcM = 128;          // rows of the output tile (UMMA M)
constexpr int kTcK = 64;           // reduction rows per stage (128 bytes of bf16)
constexpr int kConv = 256;         // converter / epilogue threads (warps 0-7)
constexpr int kTcThreads = kConv + 32;

struct TcParams {
  const float* d_pre;  // [BK][4C]
  const float* u;      // [BK][n_x]
  const float* H;      // [BK][C]
  const float* h0;     // [B][C]
  const float* W;      // [4C][n_in]
  float* out;          // dW partials [S][4C][n_in]  or  du [BK][n_x]
  const float* bias;   // projection: b [4C]
  float* xh;           // projection: X of gate ff1 -> H [BK][C]
  float* xcache;       // projection: X of gates ff2, ta, tb -> cache [BK][3][C]
  int* status;
  int B, BK, C, n_x, n_in;
  int rows, cols;      // output rows / columns of the GEMM (dW: 4C x n_in; du: BK x n_x)
  int red;             // length of the reduction index (dW: BK; du: 4C)
  int n_tile, m_tiles, kb_per_split, n_kb;
  int vec;             // operand rows can be read as float4 (n_x % 4 == 0 and C % 4 == 0)
};

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Split 8 fp32 values into three bf16 terms x = hi + mid + lo (8 significand bits each, so the
// three carry all 24 of fp32; each difference is exact in fp32) and store the three chunks.
__device__ __forceinline__ void store_split3_chunk(uint8_t* hi_tile, uint8_t* mid_tile,
                                                   uint8_t* lo_tile, int row, int kchunk,
                                                   const float (&v)[8]) {
  __nv_bfloat16 h[8], m[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __float2bfloat16_rn(v[i]);
    const float r1 = v[i] - __bfloat162float(h[i]);
    m[i] = __float2bfloat16_rn(r1);
    l[i] = __float2bfloat16_rn(r1 - __bfloat162float(m[i]));
  }
  const uint32_t off = sw128_offset(row, kchunk * 8);
  *reinterpret_cast<uint4*>(hi_tile + off) =
      make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                 pack_bf16x2(h[6], h[7]));
  *reinterpret_cast<uint4*>(mid_tile + off) =
      make_uint4(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]), pack_bf16x2(m[4], m[5]),
                 pack_bf16x2(m[6], m[7]));
  *reinterpret_cast<uint4*>(lo_tile + off) =
      make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]),
                 pack_bf16x2(l[6], l[7]));
}

// Input projection: A = u (rows r, reduction k < n_x: K-major as stored), B = W_u (rows n < 4C,
// the first n_x columns of W: K-major as stored).  The epilogue adds the bias and hands X to
// the recurrence in place: column n = g C + c of row r goes to H[r][c] (g = 0) or
// cache[r][g - 1][c].
//
// Precision: X feeds the forward, whose tolerance (1e-5 of max|H|) the two-term split's
// ~2^-17 per operand can exceed, so operands are split in three bf16 terms and the tile
// product keeps hi*hi + hi*mid + mid*hi + hi*lo + lo*hi + mid*mid (six MMAs per 16-step; the
// dropped terms are below 2^-24 of the product).  The reduction (n_x <= 512) is at most eight
// 64-entry blocks, and one stage of six tiles fits in shared memory.
struct ProjProblem {
  static constexpr int kTerms = 3, kStages = 1, kMT = 1;
  // The epilogue stages the tile in shared memory and writes whole row segments (store4)
  // when rows can be written as float4 (n_x and C multiples of 4).
  static constexpr bool kStagedOut = true;
  static __device__ __forceinline__ bool staged(const TcParams& p) { return p.vec != 0; }
  // Columns n .. n+3 of row r (n a multiple of 4; C a multiple of 4, so one gate holds all
  // four) plus the bias, into H or the cache.
  static __device__ __forceinline__ void store4(const TcParams& p, int, int r, int n, float4 x) {
    const int C = p.C;
    if (n >= 4 * C) return;
    const int g = n / C, c = n - g * C;
    const float4 b = __ldg(reinterpret_cast<const float4*>(p.bias + n));
    float* dst = (g == 0) ? p.xh + static_cast<size_t>(r) * C + c
                          : p.xcache + (static_cast<size_t>(r) * 3 + (g - 1)) * C + c;
    *reinterpret_cast<float4*>(dst) = make_float4(x.x + b.x, x.y + b.y, x.z + b.z, x.w + b.w);
  }
  // Entries k .. k+7 of a row of `width` valid values (zero beyond), as two float4 loads when
  // the row start is 16-byte aligned.
  static __device__ __forceinline__ void load8(const float* row, int k, int width, bool vec,
                                               float (&v)[8]) {
    if (vec && k + 8 <= width) {
      const float4 q0 = __ldg(reinterpret_cast<const float4*>(row + k));
      const float4 q1 = __ldg(reinterpret_cast<const float4*>(row + k + 4));
      v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
      v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (k + i < width) ? __ldg(row + k + i) : 0.f;
    }
  }
  // Tiles t = 0, 1, 2 (hi, mid, lo) of A start at a_hi + t kTcM 128, those of B at
  // b_hi + t n_tile 128 (a_lo / b_lo are the second ones).
  static __device__ __forceinline__ void convert(const TcParams& p, uint8_t* a_hi, uint8_t* a_lo,
                                                 uint8_t* b_hi, uint8_t* b_lo, int r0, int n0,
                                                 int k0, int tid) {
    const int M = 4 * p.C;
    // (row, 8-entry chunk) items, two per thread at a time with both loads issued first.
    for (int it = tid; it < kTcM * 8; it += 2 * kConv) {
      const int it1 = it + kConv;  // kTcM * 8 is a multiple of 2 * kConv
      float v0[8], v1[8];
      const int ra = r0 + (it >> 3), rb = r0 + (it1 >> 3);
      const int ka = k0 + 8 * (it & 7), kb = k0 + 8 * (it1 & 7);
      load8(p.u + static_cast<size_t>(ra < p.BK ? ra : 0) * p.n_x, ka, ra < p.BK ? p.n_x : 0,
            p.vec, v0);
      load8(p.u + static_cast<size_t>(rb < p.BK ? rb : 0) * p.n_x, kb, rb < p.BK ? p.n_x : 0,
            p.vec, v1);
      store_split3_chunk(a_hi, a_lo, a_lo + kTcM * 128, it >> 3, it & 7, v0);
      store_split3_chunk(a_hi, a_lo, a_lo + kTcM * 128, it1 >> 3, it1 & 7, v1);
    }
    for (int it = tid; it < p.n_tile * 8; it += 2 * kConv) {
      const int it1 = it + kConv;
      float v0[8], v1[8];
      const int na = n0 + (it >> 3), nb = n0 + (it1 >> 3);
      const int ka = k0 + 8 * (it & 7), kb = k0 + 8 * (it1 & 7);
      load8(p.W + static_cast<size_t>(na < M ? na : 0) * p.n_in, ka, na < M ? p.n_x : 0, p.vec,
            v0);
      if (it1 < p.n_tile * 8)
        load8(p.W + static_cast<size_t>(nb < M ? nb : 0) * p.n_in, kb, nb < M ? p.n_x : 0,
              p.vec, v1);
      store_split3_chunk(b_hi, b_lo, b_lo + p.n_tile * 128, it >> 3, it & 7, v0);
      if (it1 < p.n_tile * 8)
        store_split3_chunk(b_hi, b_lo, b_lo + p.n_tile * 128, it1 >> 3, it1 & 7, v1);
    }
  }
  static __device__ __forceinline__ void store16(const TcParams& p, int, int r, int n,
                                                 const float (&v)[16]) {
    const int M = 4 * p.C, C = p.C;
    if (p.vec && (C % 16) == 0 && n + 16 <= M) {
      // The 16 columns lie in one gate and one 16-byte aligned run of channels.
      const int g = n / C, c = n - g * C;
      float* dst = (g == 0) ? p.xh + static_cast<size_t>(r) * C + c
                            : p.xcache + (static_cast<size_t>(r) * 3 + (g - 1)) * C + c;
#pragma unroll
      for (int q = 0; q < 16; q += 4) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.bias + n + q));
        *reinterpret_cast<float4*>(dst + q) =
            make_float4(v[q] + b.x, v[q + 1] + b.y, v[q + 2] + b.z, v[q + 3] + b.w);
      }
      return;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int col = n + e;
      if (col >= M) continue;
      const int g = col / C, c = col - g * C;
      const float x = v[e] + __ldg(p.bias + col);
      if (g == 0) p.xh[static_cast<size_t>(r) * C + c] = x;
      else p.xcache[(static_cast<size_t>(r) * 3 + (g - 1)) * C + c] = x;
    }
  }
};

// One CTA's work: output tile `tile` (m-tile fastest) over reduction split `split`.
template <class Problem>
__device__ __forceinline__ void tc_gemm_body(const TcParams& p, int tile, int split) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned stage buffers (128-byte swizzle atoms), then the barriers.
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  constexpr int kStages = Problem::kStages, kTerms = Problem::kTerms;
  // Stage: kTerms A tiles [mt kTcM rows x 128 B], then kTerms B tiles [n_tile rows x 128 B].
  constexpr int kMT = Problem::kMT;
  constexpr int a_rows = kTcM * kMT;
  const int stage_bytes = kTerms * (a_rows + p.n_tile) * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * stage_bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);
  const uint32_t full0 = smem_addr(&bars[0]);             // full[s]  = full0 + 8 s
  const uint32_t empty0 = smem_addr(&bars[kStages]);      // empty[s] = empty0 + 8 s
  const uint32_t accb = smem_addr(&bars[2 * kStages]);    // accumulator ready

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int m0 = (tile % p.m_tiles) * a_rows;
  const int n0 = (tile / p.m_tiles) * p.n_tile;
  const int kb0 = split * p.kb_per_split;
  const int nk = min(p.kb_per_split, p.n_kb - kb0);
  // Accumulator j (rows m0 + 128 j ..) starts at tensor-memory column j * acc_cols, a power
  // of two (each accumulator where a single one would be allocated).
  uint32_t acc_cols = 32;
  while (acc_cols < static_cast<uint32_t>(p.n_tile)) acc_cols <<= 1;
  const uint32_t ncols = acc_cols * kMT;

  grid_dep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8u * s, kConv);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(accb, 1);
    fence_mbar_init_cluster();
  }
  // The operands come from the previous kernel; the tensor memory is taken only after it has
  // finished, so this kernel never waits for tensor memory a running predecessor holds.
  grid_dep_wait();
  if (warp == kConv / 32) {
    tmem_alloc(smem_addr(tmem_slot), ncols);
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < kConv / 32) {
    // ---- converters ----
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int s = i % kStages;
      if (i >= kStages)
        ok = mbar_wait_bounded_cta(empty0 + 8u * s, ((i - kStages) / kStages) & 1u, p.status);
      if (!ok) break;
      uint8_t* st = base + s * stage_bytes;
      Problem::convert(p, st, st + a_rows * 128, st + kTerms * a_rows * 128,
                       st + kTerms * a_rows * 128 + p.n_tile * 128, m0, n0, (kb0 + i) * kTcK, tid);
      fence_proxy_async_smem();
      mbar_arrive(full0 + 8u * s);
    }
    // ---- epilogue: TMEM row (32 * (warp % 4) + lane) -> output row; the two warpgroups take
    // alternate 16-column chunks ----
    if (ok) ok = mbar_wait_bounded_cta(accb, 0, p.status);
    tc_fence_after_sync();
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    bool done = false;
    // (Two-accumulator tiles store directly: staging their 200 KB measured slower.)
    if constexpr (Problem::kStagedOut && kMT == 1) {
      if (Problem::staged(p)) {
        // Every MMA has completed, so the stage buffer is free: the tile goes through it and
        // each warp then writes whole row segments (a row's n_tile columns are contiguous in
        // the destination).
        // [a_rows][n_tile + 4] floats: at most 128 x 260 x 4 bytes, inside the stage buffers.
        float* tile = reinterpret_cast<float*>(base);
        const int pitch = p.n_tile + 4;  // rows 16 bytes apart in bank order
        for (int j = 0; j < kMT; ++j) {
          const int r = kTcM * j + 32 * quarter + lane;
          for (int c0 = 16 * (warp >> 2); c0 < p.n_tile; c0 += 32) {
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + j * acc_cols + c0, v);
            float4* dst = reinterpret_cast<float4*>(tile + r * pitch + c0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConv) : "memory");  // warps 0-7 only
        for (int rr = warp; rr < a_rows; rr += kConv / 32) {
          const int m = m0 + rr;
          if (!ok || m >= p.rows) continue;
          for (int c = 4 * lane; c < p.n_tile; c += 128)
            Problem::store4(p, split, m, n0 + c,
                            *reinterpret_cast<const float4*>(tile + rr * pitch + c));
        }
        done = true;
      }
    }
    for (int j = 0; j < kMT && !done; ++j) {
      const int m = m0 + kTcM * j + 32 * quarter + lane;
      for (int c0 = 16 * (warp >> 2); c0 < p.n_tile; c0 += 32) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + j * acc_cols + c0, v);
        if (!ok || m >= p.rows) continue;
        Problem::store16(p, split, m, n0 + c0, v);
      }
    }
  } else if (lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = umma_idesc_bf16(kTcM, p.n_tile);
    uint32_t acc = 0;
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kStages;
      ok = mbar_wait_bounded_cta(full0 + 8u * s, (i / kStages) & 1u, p.status);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t st = smem_addr(base + s * stage_bytes);
      const uint32_t b_hi = st + kTerms * a_rows * 128, b_lo = b_hi + p.n_tile * 128;
#pragma unroll
      for (int mj = 0; mj < kMT; ++mj) {  // accumulator mj: A rows 128 mj .. 128 mj + 127
        const uint32_t d = tmem + mj * acc_cols;
        const uint32_t a_hi = st + mj * kTcM * 128, a_lo = a_hi + a_rows * 128;
#pragma unroll
        for (int j = 0; j < kTcK / 16; ++j) {
          const uint32_t koff = 32u * j;
          umma_bf16(d, umma_desc_sw128(a_hi + koff), umma_desc_sw128(b_hi + koff), idesc,
                    acc | static_cast<uint32_t>(j > 0));
          umma_bf16(d, umma_desc_sw128(a_hi + koff), umma_desc_sw128(b_lo + koff), idesc, 1);
          umma_bf16(d, umma_desc_sw128(a_lo + koff), umma_desc_sw128(b_hi + koff), idesc, 1);
          if constexpr (kTerms == 3) {  // a_lo / b_lo hold the mid terms; lo follows them
            const uint32_t a_l3 = a_lo + a_rows * 128, b_l3 = b_lo + p.n_tile * 128;
            umma_bf16(d, umma_desc_sw128(a_hi + koff), umma_desc_sw128(b_l3 + koff), idesc, 1);
            umma_bf16(d, umma_desc_sw128(a_l3 + koff), umma_desc_sw128(b_hi + koff), idesc, 1);
            umma_bf16(d, umma_desc_sw128(a_lo + koff), umma_desc_sw128(b_lo + koff), idesc, 1);
          }
        }
      }
      acc = 1;
      umma_commit(empty0 + 8u * s);  // stage reusable once these MMAs have read it
    }
    umma_commit(accb);  // accumulator complete (also after an early stop)
    // Whatever the converters did, the MMAs issued here finish before tensor memory is freed:
    // they depend on nothing outside this CTA, so this wait always completes.
    (void)mbar_wait_bounded_cta(accb, 0, p.status);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kConv / 32) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, ncols);
  }
}

template <class Problem>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const TcParams p) {
  tc_gemm_body<Problem>(p, blockIdx.x, blockIdx.y);
}

TcPlan tc_plan(int rows, int cols, int red, bool split, int terms = 2, int stages = 2,
               int mt = 1, int max_n_tile = 256) {
  TcPlan pl;
  pl.mt = mt;
  pl.n_tiles = (cols + max_n_tile - 1) / max_n_tile;
  pl.n_tile = (((cols + pl.n_tiles - 1) / pl.n_tiles) + 15) & ~15;
  pl.m_tiles = (rows + kTcM * mt - 1) / (kTcM * mt);
  pl.n_kb = (red + kTcK - 1) / kTcK;
  const int tiles = pl.m_tiles * pl.n_tiles;
  int s0 = 1;
  if (split) {
    // At most one wave of 148 CTAs (a fixed target, not the device's SM count: the split --
    // hence the summation order -- depends only on the sizes).
    s0 = tiles < 148 ? 148 / tiles : 1;
    if (s0 > pl.n_kb) s0 = pl.n_kb;
  }
  pl.kb_per_split = (pl.n_kb + s0 - 1) / s0;
  pl.splits = (pl.n_kb + pl.kb_per_split - 1) / pl.kb_per_split;
  pl.smem = static_cast<size_t>(stages) * terms * (kTcM * mt + pl.n_tile) * 128 + 1024 + 128;
  return pl;
}

}  // namespace

cudaError_t tc_prepare(int max_smem) {
  return cudaFuncSetAttribute(tc_gemm_kernel<ProjProblem>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

namespace {
TcParams make_params(const TcPlan& pl, const float* d_pre, int B, int K, int C, int n_x,
                     int* status) {
  TcParams p = {};
  p.d_pre = d_pre; p.status = status;
  p.B = B; p.BK = B * K; p.C = C; p.n_x = n_x; p.n_in = n_x + C;
  p.n_tile = pl.n_tile; p.m_tiles = pl.m_tiles; p.kb_per_split = pl.kb_per_split;
  p.n_kb = pl.n_kb;
  p.vec = (n_x % 4 == 0) && (C % 4 == 0);
  return p;
}
}  // namespace

TcPlan proj_tc_plan(int B, int K, int C, int n_x) {
  // Column tiles of at most 128: a 98 KB stage, so two CTAs share an SM and one's loads and
  // conversion overlap the other's MMAs and stores.
  return tc_plan(B * K, 4 * C, n_x, false, ProjProblem::kTerms, ProjProblem::kStages, 1, 128);
}

cudaError_t proj_tc_launch(const TcPlan& pl, const float* u, const float* W, const float* bias,
                           int B, int K, int C, int n_x, float* H, float* cache, int* status,
                           cudaStream_t s, bool pdl) {
  TcParams p = make_params(pl, nullptr, B, K, C, n_x, status);
  p.u = u; p.W = W; p.bias = bias; p.xh = H; p.xcache = cache;
  p.rows = B * K; p.cols = 4 * C; p.red = n_x;
  LaunchCfg c;
  c.grid = dim3(pl.m_tiles * pl.n_tiles, pl.splits, 1);
  c.block = dim3(kTcThreads, 1, 1);
  c.smem = pl.smem;
  c.stream = s;
  c.pdl = pdl;
  return launch(c, tc_gemm_kernel<ProjProblem>, p);
}

}  // namespace cfc
