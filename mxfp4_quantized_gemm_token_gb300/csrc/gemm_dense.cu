// gemm_dense.cu — instantiations of the scaled-GEMM kernel for
// fp8_scaled_mm, and the launcher that dispatches every GEMM.
#include "gemm_launch.cuh"

namespace mxq {

cudaError_t launch_gemm_moe(int kind, int epi, int bt, bool promote, const GemmMaps& maps,
                            const GemmParams& p, int grid, cudaStream_t stream);

cudaError_t launch_gemm(int kind, int epi, int bt, bool promote, const GemmMaps& maps,
                        const GemmParams& p, int grid, cudaStream_t stream) {
  if (epi == EPI_NORMAL) {
    // tokens on the MMA M side: FP8 x FP8 with uniform weight-block scales
    if (kind == KIND_F8F8 && bt == 128)
      return launch_gemm_inst<KIND_F8F8, EPI_NORMAL, 128, true>(maps, p, grid, stream);
    if (kind == KIND_F8F8 && bt == 192)
      return launch_gemm_inst<KIND_F8F8, EPI_NORMAL, 192, true>(maps, p, grid, stream);
    if (kind == KIND_F8F8 && bt == 256)
      return launch_gemm_inst<KIND_F8F8, EPI_NORMAL, 256, true>(maps, p, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (epi == EPI_NORMAL_COLW) {
    // tokens on the MMA M side with a weight scale per column ([1, 128] blocks)
    if (kind == KIND_F8F8 && bt == 128)
      return launch_gemm_inst<KIND_F8F8, EPI_NORMAL_COLW, 128, true>(maps, p, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (epi != EPI_DENSE) return launch_gemm_moe(kind, epi, bt, promote, maps, p, grid, stream);
  if (kind == KIND_F8Q) {
    // decode-size W8A8 with the activation quantization inside the GEMM
    if (bt == 32) return launch_gemm_inst<KIND_F8Q, EPI_DENSE, 32, true>(maps, p, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (kind == KIND_F8F8) {
    // activation group scales always present: every slice is promoted
    return launch_gemm_bt<KIND_F8F8, EPI_DENSE, true>(bt, maps, p, grid, stream);
  }
  if (kind == KIND_F8W) {
    return promote ? launch_gemm_bt<KIND_F8W, EPI_DENSE, true>(bt, maps, p, grid, stream)
                   : launch_gemm_bt<KIND_F8W, EPI_DENSE, false>(bt, maps, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mxq
