// cfc_selftest.cu -- an on-device check of the library's failure detection.
//
// Every wait in the library's kernels (mbarrier phases, cluster exchanges, tensor-core
// pipelines) is bounded: after kWaitLimitNs it records kStatusTimeout in the device status word
// and the kernel winds down instead of hanging.  This kernel makes that path run on purpose and
// harmlessly: one thread waits, through the same bounded wait, on a shared-memory mbarrier whose
// phase nothing completes.  No fault, no trap: the wait runs out, the status word is set, and the
// kernel returns, leaving the context usable.
#include "cfc_launch.cuh"
#include "cfc_ptx.cuh"

namespace cfc {
namespace {

__global__ void wait_self_test_kernel(int* status) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);  // one arrival would complete phase 0; none comes
  (void)mbar_wait_bounded_cta(b, 0, status);
}

}  // namespace

cudaError_t wait_self_test_launch(int* status, cudaStream_t s) {
  LaunchCfg c;
  c.grid = dim3(1, 1, 1);
  c.block = dim3(1, 1, 1);
  c.stream = s;
  return launch(c, wait_self_test_kernel, status);
}

}  // namespace cfc
