// cfc_ptx.cuh -- thin inline-PTX helpers for sm_103a: thread-block-cluster ranks and
// distributed shared memory, mbarriers, asynchronous remote stores (st.async), and bounded
// waits that report a timeout instead of spinning forever.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace cfc {

// Device status word values (written by kernels into the library's status word).
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 1;

// A wait that has not completed after this many nanoseconds is abandoned (the kernel records
// kStatusTimeout and winds down).  Correct launches never come near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Programmatic dependent launch: wait until the previous kernel of the stream has completed
// and its writes are visible (a no-op when the kernel was launched without the attribute) ...
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ... and allow the next kernel of the stream to be scheduled before this one completes.
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bring the 128-byte line holding `p` into L2 (no register result, nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the other CTAs of the cluster.
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Upper bound (ns) a waiting thread may stay suspended inside one try_wait; the hardware
// resumes it as soon as the phase completes.  Suspended warps take no issue slots, so the
// warps still computing on the same SM run at full speed.
constexpr uint32_t kSuspendHintNs = 100000u;

// Probe of phase `parity` with cluster-scope acquire (remote st.async data written into this
// CTA's shared memory is visible once it returns true); may suspend the thread for the
// hardware's own time limit.  No suspend hint: in an exchange-only probe of the recurrences'
// step (GB300, 32 clusters) this took 0.234 us per step against 0.251 us with the hint.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of phase `parity` with cluster-scope acquire: returns at once.  For a
// warp whose lanes poll different barriers (a suspending probe would hold every lane).
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`; returns false (and records a timeout in *status) when
// the wait exceeds kWaitLimitNs.  The status word is only ever written here, never read: a
// flag left by an earlier launch (until cfc_device_status reads and clears it) cannot make a
// later launch give up.  Each wait measures its own limit, so after a failure the other waits
// of the same launch end within that limit too.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
      atomicExch(status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait_bounded_cta(uint32_t bar, uint32_t parity,
                                                      int* status) {
  if (mbar_try_wait_cta(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cta(bar, parity)) return true;
    if ((it & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
      atomicExch(status, kStatusTimeout);
      return false;
    }
  }
}

// Asynchronous 4-byte / 16-byte store into (possibly remote) shared memory of this cluster;
// completion is signalled as transaction bytes on the mbarrier `rbar` of the destination CTA.
__device__ __forceinline__ void st_async_b32(uint32_t raddr, float v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
      "r"(__float_as_uint(v)), "r"(rbar)
      : "memory");
}

// Predicated form: lanes with pred == false issue nothing (no divergent branch around it).
__device__ __forceinline__ void st_async_b32_if(bool pred, uint32_t raddr, float v,
                                                uint32_t rbar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t"
      "@p st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n\t}" ::"r"(
          raddr),
      "r"(__float_as_uint(v)), "r"(rbar), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

__device__ __forceinline__ void st_async_v4_if(bool pred, uint32_t raddr, float a, float b,
                                               float c, float d, uint32_t rbar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "@p st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];\n\t}" ::"r"(raddr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
      "r"(__float_as_uint(d)), "r"(rbar), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

__device__ __forceinline__ void st_async_v4(uint32_t raddr, float a, float b, float c, float d,
                                            uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(raddr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
      "r"(__float_as_uint(d)), "r"(rbar)
      : "memory");
}

// Full cluster barrier (every thread of every CTA in the cluster arrives).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t raddr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t raddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(raddr)
               : "memory");
  return v;
}

// 4-byte asynchronous global -> shared copy (completion tracked per thread by commit groups).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's most recent commit groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory).

// Allocate `ncols` (power of two >= 32) TMEM columns; the base address lands in *smem_dst.
// Executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory writes of this thread become visible to the async proxy (tensor cores / TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (`rbar` from map_to_rank), releasing at
// cluster scope what this thread has written or observed before.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Bulk copy global -> this CTA's shared memory, completing as transaction bytes on `bar`.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk copy this CTA's shared memory -> global, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(src), "r"(bytes)
               : "memory");
}

// Close this thread's current bulk group, then wait until all its bulk groups are complete
// (their global writes performed).
__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this thread's generic-proxy and async-proxy (bulk copy) accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Warp-collective load of 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart (tile base 1024-byte aligned; advance the start address by 32 B per 16-element step).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                    // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                  // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, fp32 accumulator, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of element (row, k) in a K-major 128-byte-swizzled bf16 tile with 64 columns.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 +
                               ((((k >> 3) ^ (row & 7)) & 7) << 4) + ((k & 7) << 1));
}

// Loads issued where they stand: prefetches into registers for the next step would otherwise
// be moved down to their use by the compiler, and their latency would land on the step's
// critical path.  (ld_early, ld_early_f4: read-only data; `p` a global address.)
__device__ __forceinline__ float4 ld_early_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
// Data another launch of this stream wrote (X from the projection): the L2 copy.
__device__ __forceinline__ float ld_early_cg(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// ---- packed conversions: one instruction converts two values, and a bf16 widens to fp32 by
// a 16-bit shift.  (Conversions share a narrow pipe with the exponentials and reciprocals.)
// Packed pairs hold the first value in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo_f32(uint32_t pk) { return __uint_as_float(pk << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t pk) {
  return __uint_as_float(pk & 0xFFFF0000u);
}
__device__ __forceinline__ uint32_t f16x2_rn(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Two terms of a pair: hi = bf16(x), lo = bf16(x - hi), packed; the same values as converting
// one at a time.
__device__ __forceinline__ void bf16_split2_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = bf16x2_rn(a, b);
  lo = bf16x2_rn(a - bf16_lo_f32(hi), b - bf16_hi_f32(hi));
}
// Two terms of a pair: hi = fp16(x), lo = fp16(x - hi), packed; the same values as converting
// one at a time.
__device__ __forceinline__ void f16_split2_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = f16x2_rn(a, b);
  const float2 w = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo = f16x2_rn(a - w.x, b - w.y);
}

// Single-precision sigmoid from the hardware exponential and reciprocal (__expf, __fdividef):
// a few ulp of relative error, far below the recurrence's fp32 accumulation error (the
// measured parity errors of H and the cache do not change against expf and a correctly
// rounded reciprocal), at about half the latency on the serial chain.  1 + e^-x overflowing
// to infinity gives 0, the correct limit.
__device__ __forceinline__ float sigmoid_fast(float x) {
  return __fdividef(1.0f, 1.0f + __expf(-x));
}

// Packed fp32 FMA (two independent lanes of fma.rn in one instruction on sm_100 and later):
// the recurrences' matrix-vector products pair consecutive inputs, halving their FMA issue.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

}  // namespace cfc
