// gg_launch.cuh — the launch helper that the permute and quantiser translation
// units share (host side).
#pragma once

#include <cuda_runtime.h>

namespace gg {

// Launch with programmatic stream serialisation: the kernel may start while
// the one ahead of it in the stream runs, and must call grid_dependency_wait()
// before it touches anything that kernel writes or reads.
template <typename... Params, typename... Args>
cudaError_t launch_early(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

}  // namespace gg
