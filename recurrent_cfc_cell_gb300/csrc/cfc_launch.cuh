// cfc_launch.cuh -- one launch path for every kernel of the library: grid, block, dynamic
// shared memory, stream, optional thread-block-cluster shape and optional programmatic
// dependent launch.
//
// With `pdl` the kernel may be scheduled while the previous kernel of the stream is still
// running; it must then execute griddepcontrol.wait (grid_dep_wait) before it reads anything
// the previous kernel writes or writes anything at all in global memory.  The library sets
// `pdl` only between two kernels launched by the same entry point, so the work a caller
// queued before the entry point has always finished when any of its kernels starts.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace cfc {

struct LaunchCfg {
  dim3 grid;
  dim3 block;
  size_t smem = 0;
  cudaStream_t stream = nullptr;
  bool pdl = false;
  dim3 cluster = dim3(0, 0, 0);  // x == 0: no cluster attribute
};

template <typename... KArgs, typename... Args>
cudaError_t launch(const LaunchCfg& c, void (*kern)(KArgs...), Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = c.grid;
  cfg.blockDim = c.block;
  cfg.dynamicSmemBytes = c.smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (c.cluster.x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = c.cluster.x;
    attr[n].val.clusterDim.y = c.cluster.y;
    attr[n].val.clusterDim.z = c.cluster.z;
    ++n;
  }
  if (c.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace cfc
