// gemm_launch.cuh — host-side launch of one gemm_kernel instantiation.
#pragma once

#include "internal.h"

namespace mxq {

template <int KIND, int EPI, int BT, bool PROMOTE>
cudaError_t launch_gemm_inst(const GemmMaps& maps, const GemmParams& p, int grid,
                             cudaStream_t stream) {
  using L = Layout<KIND, BT, EPI>;
  const int smem = L::TOTAL + 1024;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(gemm_kernel<KIND, EPI, BT, PROMOTE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_k(gemm_kernel<KIND, EPI, BT, PROMOTE>, dim3(grid), dim3(L::kThreads),
                  static_cast<size_t>(smem), stream, maps, p);
}

template <int KIND, int EPI, bool PROMOTE>
cudaError_t launch_gemm_bt(int bt, const GemmMaps& maps, const GemmParams& p, int grid,
                           cudaStream_t stream) {
  switch (bt) {
    case 32: return launch_gemm_inst<KIND, EPI, 32, PROMOTE>(maps, p, grid, stream);
    case 64: return launch_gemm_inst<KIND, EPI, 64, PROMOTE>(maps, p, grid, stream);
    case 128: return launch_gemm_inst<KIND, EPI, 128, PROMOTE>(maps, p, grid, stream);
    case 256:
      // 256 token columns: FP8 x FP8 only (the bf16 kinds do not fit shared memory)
      if constexpr (KIND == KIND_F8F8)
        return launch_gemm_inst<KIND, EPI, 256, PROMOTE>(maps, p, grid, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxq
