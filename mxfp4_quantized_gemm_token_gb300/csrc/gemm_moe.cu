// gemm_moe.cu — instantiations of the scaled-GEMM kernel for the two fused
// MoE stages (SiLU-and-mul epilogue, scatter-with-routing-weight epilogue).
#include "gemm_launch.cuh"

namespace mxq {

cudaError_t launch_gemm_moe(int kind, int epi, int bt, bool promote, const GemmMaps& maps,
                            const GemmParams& p, int grid, cudaStream_t stream) {
  (void)promote;
  if (kind == KIND_F8W) {
    // FP8 block weights: per-slice promotion with the block scale
    if (epi == EPI_SILU) return launch_gemm_bt<KIND_F8W, EPI_SILU, true>(bt, maps, p, grid, stream);
    if (epi == EPI_SCATTER)
      return launch_gemm_bt<KIND_F8W, EPI_SCATTER, true>(bt, maps, p, grid, stream);
  } else if (kind == KIND_F8H) {
    if (epi == EPI_SILU) return launch_gemm_bt<KIND_F8H, EPI_SILU, true>(bt, maps, p, grid, stream);
    if (epi == EPI_SCATTER)
      return launch_gemm_bt<KIND_F8H, EPI_SCATTER, true>(bt, maps, p, grid, stream);
  } else if (kind == KIND_MXH) {
    // MXFP4 decoded to f16 relative to each row's largest scale: whole-K
    if (epi == EPI_SILU) return launch_gemm_bt<KIND_MXH, EPI_SILU, false>(bt, maps, p, grid, stream);
    if (epi == EPI_SCATTER)
      return launch_gemm_bt<KIND_MXH, EPI_SCATTER, false>(bt, maps, p, grid, stream);
  } else if (kind == KIND_MXW) {
    // MXFP4: the ue8m0 scale is folded into the exact bf16 decode
    if (epi == EPI_SILU) return launch_gemm_bt<KIND_MXW, EPI_SILU, false>(bt, maps, p, grid, stream);
    if (epi == EPI_SCATTER)
      return launch_gemm_bt<KIND_MXW, EPI_SCATTER, false>(bt, maps, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mxq
