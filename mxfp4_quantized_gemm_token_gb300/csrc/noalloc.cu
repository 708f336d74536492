// noalloc.cu — mxq_fp8_scaled_mm_noalloc: the scaled GEMM for callers that
// cannot allocate device memory.
//
// mxq_fp8_scaled_mm takes its split-K scratch from a caller-provided
// workspace.  Some callers have no way to provide one: code running inside a
// framework's memory pool that forbids raw cudaMalloc, plugins that receive
// only input/output buffers, or programs that must not allocate after start-up
// (pre-planned memory, real-time serving loops).  For them this entry point
// keeps the split-K partial sums in a fixed array that lives in the library
// itself, so a call needs nothing but its inputs and outputs.
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "mxq.h"

namespace {

// One scratch array per GPU that loads the library, held until the process
// exits.  MXQ_NOALLOC_SCRATCH_BYTES is its size.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MXQ_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" mxq_status mxq_fp8_scaled_mm_noalloc(
    const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda, const float* a_scale,
    int64_t sa0, int64_t sa1, const void* W, int64_t N, int64_t ldw, const float* w_scale,
    int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1, const void* bias,
    int32_t bias_dtype, void* out, int32_t out_dtype, int64_t ldo, mxq_stream_t stream) {
  // the arguments first, so a bad call reports its real error
  const mxq_status vst =
      mxq::validate_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, w_scale, block_n,
                       block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo);
  if (vst != MXQ_OK) return vst;
  if (M == 0 || N == 0) return MXQ_OK;
  // the split-K partials of the plan the call will run on this device
  size_t need = 0;
  const mxq_status st = mxq::mm_workspace_bytes(M, N, K, a_dtype, block_n, block_k, &need);
  if (st != MXQ_OK) return st;
  if (need > static_cast<size_t>(MXQ_NOALLOC_SCRATCH_BYTES)) {
    mxq::set_last_error("mxq_fp8_scaled_mm_noalloc: this shape needs " + std::to_string(need) +
                        " bytes of split-K scratch, more than the built-in " +
                        std::to_string(static_cast<long long>(MXQ_NOALLOC_SCRATCH_BYTES)) +
                        " bytes; use mxq_fp8_scaled_mm with a workspace");
    return MXQ_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  if (need > 0) {
    // The array's name in host code is only a stand-in; its device address
    // on the current device is looked up on every call (a cheap host-side
    // query), so a reset device or a different context never sees a stale
    // address.
    const cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess) {
      mxq::set_last_error(std::string("mxq_fp8_scaled_mm_noalloc: cudaGetSymbolAddress: ") +
                          cudaGetErrorString(e));
      return MXQ_ERR_CUDA;
    }
  }
  // The partials are fully rewritten by every split, so nothing needs clearing.
  return mxq_fp8_scaled_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, w_scale, block_n,
                           block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo, scratch,
                           need > 0 ? static_cast<size_t>(MXQ_NOALLOC_SCRATCH_BYTES) : 0, stream);
}
