// Kernel launch helper: cudaLaunchKernelEx with optional programmatic
// dependent launch (the kernel may start while its predecessor drains and
// must call griddepcontrol.wait before touching the predecessor's output).
#pragma once

#include <cuda_runtime.h>

namespace clover {

template <typename Arg>
cudaError_t launch_kernel(void (*kernel)(Arg), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

}  // namespace clover
