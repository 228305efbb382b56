// cfc_reduce.cu -- reduce_axis0: out[n] = sum_{r < n_batch} per_batch[r][n], OVERWRITE.
//
// The K-loop parallelization spec (page "K-loop Parallelization -- Block-per-Batch Kernel
// Refactor", section "Architecture Choice", item 3) defines reduce_axis0(per_batch [B, N],
// n_batch, n_tail, out [N]): a block tree-reduce across the batch index with no atomicAdd,
// grid over the output tail dimension, output overwritten (never accumulated into).
//
// GB300 layout: grid = (column tiles, CZ) with a thread-block cluster of CZ CTAs along the
// batch axis, so a tall input (e.g. 262144 x 1024 bias partials) still spreads over up to
// 16 x (tiles) SMs.  Each CTA sums a fixed row range (8 row-lanes x 32 column-lanes, float4
// columns when aligned); lanes are merged in shared memory in lane order and the CZ CTA sums
// are merged through distributed shared memory in rank order.  The summation order depends only
// on (n_batch, n_tail), so the result is bitwise reproducible run to run.
#include "cfc_kernels.h"
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

constexpr int kRowLanes = 8;
constexpr int kColLanes = 32;

// Where sum n goes: out[n], or -- for a tail that is rows of `pitch` values (pitch > 0) --
// columns < ncol of row n / pitch to out[row * ncol + col], column ncol to out2[row], and the
// rest of the row (padding) nowhere.
struct OutMap {
  float* out;
  float* out2;
  int pitch, ncol;
};

__device__ __forceinline__ void put(const OutMap& o, int n, float v) {
  if (o.pitch == 0) {
    o.out[n] = v;
    return;
  }
  const int row = n / o.pitch, col = n - row * o.pitch;
  if (col < o.ncol) o.out[static_cast<size_t>(row) * o.ncol + col] = v;
  else if (col == o.ncol) o.out2[row] = v;
}

// One sum: n_tail columns of n_batch rows, each cluster CTA taking rows_per_cta rows.
struct Seg {
  const float* in;
  int n_batch, n_tail, rows_per_cta;
  OutMap o;
};

// Column tile `tile` of segment g (every CTA of the cluster along y works on the same tile).
template <int VEC>
__device__ __forceinline__ void reduce_tile(const Seg& g, int tile) {
  constexpr int TC = kColLanes * VEC;
  __shared__ __align__(16) float part[kRowLanes][TC];
  __shared__ __align__(16) float cta_sum[TC];
  const float* __restrict__ in = g.in;
  const int n_batch = g.n_batch, n_tail = g.n_tail, rows_per_cta = g.rows_per_cta;
  const OutMap& o = g.o;
  const int tid = threadIdx.x;
  const int cl = tid % kColLanes, rl = tid / kColLanes;
  const int col = tile * TC + cl * VEC;
  const int q = static_cast<int>(cluster_rank());
  const int CZ = static_cast<int>(gridDim.y);
  const int lo = q * rows_per_cta;
  const int hi = min(n_batch, lo + rows_per_cta);

  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
  if (col < n_tail) {
    if constexpr (VEC == 4) {
      const float* base = in + col;
      int r = lo + rl;
      for (; r + 3 * kRowLanes < hi; r += 4 * kRowLanes) {
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(r) * n_tail));
        const float4 v1 = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(r + kRowLanes) * n_tail));
        const float4 v2 = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(r + 2 * kRowLanes) * n_tail));
        const float4 v3 = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(r + 3 * kRowLanes) * n_tail));
        acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
        acc[0] += v1.x; acc[1] += v1.y; acc[2] += v1.z; acc[3] += v1.w;
        acc[0] += v2.x; acc[1] += v2.y; acc[2] += v2.z; acc[3] += v2.w;
        acc[0] += v3.x; acc[1] += v3.y; acc[2] += v3.z; acc[3] += v3.w;
      }
      for (; r < hi; r += kRowLanes) {
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(r) * n_tail));
        acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
      }
    } else {
      const float* base = in + col;
      int r = lo + rl;
      for (; r + 3 * kRowLanes < hi; r += 4 * kRowLanes) {
        const float v0 = __ldg(base + static_cast<size_t>(r) * n_tail);
        const float v1 = __ldg(base + static_cast<size_t>(r + kRowLanes) * n_tail);
        const float v2 = __ldg(base + static_cast<size_t>(r + 2 * kRowLanes) * n_tail);
        const float v3 = __ldg(base + static_cast<size_t>(r + 3 * kRowLanes) * n_tail);
        acc[0] += v0; acc[0] += v1; acc[0] += v2; acc[0] += v3;
      }
      for (; r < hi; r += kRowLanes) acc[0] += __ldg(base + static_cast<size_t>(r) * n_tail);
    }
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) part[rl][cl * VEC + v] = acc[v];
  __syncthreads();
  for (int c = tid; c < TC; c += kRowLanes * kColLanes) {
    float sacc = part[0][c];
#pragma unroll
    for (int l = 1; l < kRowLanes; ++l) sacc += part[l][c];
    cta_sum[c] = sacc;
  }
  if (CZ == 1) {
    __syncthreads();
    for (int c = tid; c < TC; c += kRowLanes * kColLanes) {
      const int n = tile * TC + c;
      if (n < n_tail) put(o, n, cta_sum[c]);
    }
    return;
  }
  cluster_sync_all();
  if (q == 0) {
    for (int c = tid; c < TC; c += kRowLanes * kColLanes) {
      const uint32_t a = smem_addr(&cta_sum[c]);
      float sacc = cta_sum[c];
      for (int qq = 1; qq < CZ; ++qq) sacc += ld_shared_cluster_f32(map_to_rank(a, qq));
      const int n = tile * TC + c;
      if (n < n_tail) put(o, n, sacc);
    }
  }
  cluster_sync_all();
}

template <int VEC>
__global__ void __launch_bounds__(kRowLanes * kColLanes) reduce_axis0_kernel(const Seg g) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  reduce_tile<VEC>(g, blockIdx.x);
}

// Two sums in one launch: column tiles [0, tiles_a) of segment a, the rest of segment b.
template <int VEC>
__global__ void __launch_bounds__(kRowLanes * kColLanes) reduce_axis0_pair_kernel(
    const Seg a, const Seg b, int tiles_a) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  if (static_cast<int>(blockIdx.x) < tiles_a) reduce_tile<VEC>(a, blockIdx.x);
  else reduce_tile<VEC>(b, blockIdx.x - tiles_a);
}

int choose_cz(int n_batch) {
  int cz = (n_batch + 127) / 128;
  if (cz < 1) cz = 1;
  if (cz > kMaxClusterSize) cz = kMaxClusterSize;
  return cz;
}

template <int VEC>
cudaError_t launch_vec(const float* in, int n_batch, int n_tail, const OutMap& o, cudaStream_t s,
                       bool pdl) {
  constexpr int TC = kColLanes * VEC;
  const int cz = choose_cz(n_batch);
  const Seg g{in, n_batch, n_tail, (n_batch + cz - 1) / cz, o};
  LaunchCfg c;
  c.grid = dim3((n_tail + TC - 1) / TC, cz, 1);
  c.block = dim3(kRowLanes * kColLanes, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(1, cz, 1);
  return launch(c, reduce_axis0_kernel<VEC>, g);
}

template <int VEC>
cudaError_t launch_pair_vec(const float* in, int n_batch, int n_tail, const OutMap& o,
                            const float* in_b, int n_batch_b, int n_tail_b, const OutMap& o_b,
                            cudaStream_t s, bool pdl) {
  constexpr int TC = kColLanes * VEC;
  // One cluster shape for both: the larger batch decides it; each segment spreads its own
  // rows over the cluster's CTAs (its summation order still depends only on its sizes and
  // the other segment's batch count).
  const int cz = choose_cz(n_batch > n_batch_b ? n_batch : n_batch_b);
  const Seg a{in, n_batch, n_tail, (n_batch + cz - 1) / cz, o};
  const Seg b{in_b, n_batch_b, n_tail_b, (n_batch_b + cz - 1) / cz, o_b};
  const int tiles_a = (n_tail + TC - 1) / TC;
  LaunchCfg c;
  c.grid = dim3(tiles_a + (n_tail_b + TC - 1) / TC, cz, 1);
  c.block = dim3(kRowLanes * kColLanes, 1, 1);
  c.stream = s;
  c.pdl = pdl;
  c.cluster = dim3(1, cz, 1);
  return launch(c, reduce_axis0_pair_kernel<VEC>, a, b, tiles_a);
}

}  // namespace

cudaError_t reduce_axis0_prepare() {
  cudaError_t e = cudaFuncSetAttribute(reduce_axis0_kernel<4>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(reduce_axis0_kernel<1>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(reduce_axis0_pair_kernel<4>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(reduce_axis0_pair_kernel<1>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t reduce_axis0_launch(const float* in, int n_batch, int n_tail, float* out,
                                cudaStream_t s, bool pdl) {
  return reduce_axis0_rows_launch(in, n_batch, n_tail, 0, 0, out, nullptr, s, pdl);
}

cudaError_t reduce_axis0_rows_launch(const float* in, int n_batch, int n_tail, int pitch,
                                     int ncol, float* out, float* out2, cudaStream_t s,
                                     bool pdl) {
  const OutMap o{out, out2, pitch, ncol};
  const bool vec = (n_tail % 4 == 0) && (reinterpret_cast<uintptr_t>(in) % 16 == 0);
  return vec ? launch_vec<4>(in, n_batch, n_tail, o, s, pdl)
             : launch_vec<1>(in, n_batch, n_tail, o, s, pdl);
}

cudaError_t reduce_axis0_pair_launch(const float* in, int n_batch, int n_tail, int pitch,
                                     int ncol, float* out, float* out2, const float* in_b,
                                     int n_batch_b, int n_tail_b, float* out_b, cudaStream_t s,
                                     bool pdl) {
  const OutMap o{out, out2, pitch, ncol};
  const OutMap o_b{out_b, nullptr, 0, 0};
  const bool vec = (n_tail % 4 == 0) && (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
                   (n_tail_b % 4 == 0) && (reinterpret_cast<uintptr_t>(in_b) % 16 == 0);
  return vec ? launch_pair_vec<4>(in, n_batch, n_tail, o, in_b, n_batch_b, n_tail_b, o_b, s, pdl)
             : launch_pair_vec<1>(in, n_batch, n_tail, o, in_b, n_batch_b, n_tail_b, o_b, s,
                                  pdl);
}

}  // namespace cfc
