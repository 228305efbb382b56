// cfc_ptx.cuh -- thin inline-PTX helpers for sm_103a: thread-block-cluster ranks and
// distributed shared memory, mbarriers, asynchronous remote stores (st.async), and bounded
// waits that report a timeout instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace cfc {

// Device status word values (written by kernels into the library's status word).
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 1;

// A wait that has not completed after this many nanoseconds is abandoned (the kernel records
// kStatusTimeout and winds down).  Correct launches never come near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

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
// CTA's shared memory is visible once it returns true); may suspend the thread meanwhile.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
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
// the wait exceeds kWaitLimitNs or another CTA has already recorded a failure.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (*reinterpret_cast<volatile int*>(status) != kStatusOk) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait_bounded_cta(uint32_t bar, uint32_t parity,
                                                      int* status) {
  if (mbar_try_wait_cta(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cta(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (*reinterpret_cast<volatile int*>(status) != kStatusOk) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicExch(status, kStatusTimeout);
        return false;
      }
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

// Accurate single-precision sigmoid: expf, then a correctly rounded reciprocal (the same value
// as the IEEE quotient 1 / (1 + e)); no approximate hardware exp / tanh variants.
__device__ __forceinline__ float sigmoid_acc(float x) { return __frcp_rn(1.0f + expf(-x)); }

}  // namespace cfc
