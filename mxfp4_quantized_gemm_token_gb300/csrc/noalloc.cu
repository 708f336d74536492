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

#include <mutex>
#include <string>

#include "internal.h"
#include "mxq.h"

namespace {

// One scratch array per GPU that loads the library, held until the process
// exits.  MXQ_NOALLOC_SCRATCH_BYTES is its size.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MXQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

}  // namespace

extern "C" mxq_status mxq_fp8_scaled_mm_noalloc(
    const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda, const float* a_scale,
    int64_t sa0, int64_t sa1, const void* W, int64_t N, int64_t ldw, const float* w_scale,
    int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1, const void* bias,
    int32_t bias_dtype, void* out, int32_t out_dtype, int64_t ldo, mxq_stream_t stream) {
  if (M < 0 || N < 0 || K <= 0) return mxq_fp8_scaled_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1,
                                                         W, N, ldw, w_scale, block_n, block_k, sw0,
                                                         sw1, bias, bias_dtype, out, out_dtype,
                                                         ldo, nullptr, 0, stream);
  if (M == 0 || N == 0) return MXQ_OK;
  // the split-K partials this shape needs on this device
  size_t need = 0;
  mxq_status st = mxq_fp8_scaled_mm_workspace_size(M, N, K, a_dtype, &need);
  if (st != MXQ_OK) return st;
  if (need > static_cast<size_t>(MXQ_NOALLOC_SCRATCH_BYTES)) {
    mxq::set_last_error("mxq_fp8_scaled_mm_noalloc: this shape needs " + std::to_string(need) +
                        " bytes of split-K scratch, more than the built-in " +
                        std::to_string(static_cast<long long>(MXQ_NOALLOC_SCRATCH_BYTES)) +
                        " bytes; use mxq_fp8_scaled_mm with a workspace");
    return MXQ_ERR_UNSUPPORTED;
  }
  // set-up once per device, with that device current: the device address of
  // the array (its host-side name is only a stand-in)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    mxq::set_last_error("mxq_fp8_scaled_mm_noalloc: no current CUDA device");
    return MXQ_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) {
        mxq::set_last_error(std::string("mxq_fp8_scaled_mm_noalloc: cudaGetSymbolAddress: ") +
                            cudaGetErrorString(e));
        return MXQ_ERR_CUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  // The partials are fully rewritten by every split, so nothing needs clearing.
  return mxq_fp8_scaled_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, w_scale, block_n,
                           block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo, scratch,
                           static_cast<size_t>(MXQ_NOALLOC_SCRATCH_BYTES), stream);
}
