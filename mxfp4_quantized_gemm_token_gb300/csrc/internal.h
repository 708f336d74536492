// internal.h — host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "gemm_kernel.cuh"
#include "mxq.h"

namespace mxq {

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;   // device status word (static __device__ variable)
};

// Per-device facts, checked once per device (compute capability 10.3).
bool device_info(DeviceInfo* info, std::string* err);

// Sets the message mxq_last_error() returns on this thread.
void set_last_error(const std::string& msg);

// Process-wide options (see MXQ_OPT_*).
int64_t option(int32_t which);

// Host-side argument checks of mxq_fp8_scaled_mm: MXQ_OK or the first
// problem's status (with mxq_last_error set).
mxq_status validate_mm(const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
                       const float* a_scale, int64_t sa0, int64_t sa1, const void* W, int64_t N,
                       int64_t ldw, const float* w_scale, int32_t block_n, int32_t block_k,
                       int64_t sw0, int64_t sw1, const void* bias, int32_t bias_dtype,
                       const void* out, int32_t out_dtype, int64_t ldo);

// Split-K scratch bytes of the plan mxq_fp8_scaled_mm runs for these sizes
// on the current device (0: no split).
mxq_status mm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t a_dtype, int32_t block_n,
                              int32_t block_k, size_t* bytes);

// tensor-map encode through the driver entry point (no libcuda link)
bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle, std::string* err);

// Launch kernel<<<grid, block, smem, stream>>>(args...), with programmatic
// stream serialization (the kernel may launch while the previous one on
// the stream finishes; it waits for it in pdl_wait()) unless MXQ_OPT_PDL
// is 0.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (option(MXQ_OPT_PDL) != 0) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  // consume a launch error here (as cudaGetLastError after <<<>>> would), so
  // that it is reported once, through this library's status
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

cudaError_t launch_gemm(int kind, int epi, int bt, bool promote, const GemmMaps& maps,
                        const GemmParams& p, int grid, cudaStream_t stream);

cudaError_t launch_group_quant(const void* x, int64_t M, int64_t K, int64_t ldx, int group,
                               float eps, void* q, float* scales, int num_sms, cudaStream_t stream);

cudaError_t launch_mxfp4_quant(const void* x, bool bf16, int64_t R, int64_t C, int64_t ldx,
                               void* packed, void* scales, int num_sms, cudaStream_t stream);

cudaError_t launch_moe_align(const int32_t* topk_ids, int64_t S, int32_t E, int32_t block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* offsets,
                             int32_t* num_blocks, int64_t cap, int* status, cudaStream_t stream);

cudaError_t launch_gather_rows(const void* hidden, int64_t ldh, int64_t K, int32_t topk,
                               const int32_t* sorted_ids, const int32_t* offsets,
                               const int32_t* num_blocks, int32_t block_m, int64_t cap, void* xs,
                               int* zero, int64_t nzero, const float* tscale, float* rscale,
                               cudaStream_t stream);

cudaError_t launch_mx_row_emax(const void* s1, int64_t rows1, int64_t ncols1, int64_t ld1, void* e1,
                               const void* s2, int64_t rows2, int64_t ncols2, int64_t ld2, void* e2,
                               const int32_t* expert_ids, const int32_t* num_blocks, int E,
                               int64_t cap, cudaStream_t stream);

cudaError_t launch_rows_to_f16(const void* src, int64_t rows, int64_t K, int64_t ld,
                               const int32_t* count, void* dst, float* rscale,
                               cudaStream_t stream);

cudaError_t launch_combine(const float* y, int64_t T, int32_t topk, int64_t K, void* out,
                           int64_t ldo, cudaStream_t stream);

cudaError_t launch_splitk_reduce(const float* partial, int splits, int64_t M, int64_t N,
                                 const void* bias, int bias_dtype, void* out, int out_dtype,
                                 int64_t ldo, cudaStream_t stream);

cudaError_t launch_unsort_rows(const void* ic1, int64_t N, const int32_t* sorted_ids,
                               const int32_t* offsets, const int32_t* num_blocks, int32_t block_m,
                               int64_t cap, void* act_out, cudaStream_t stream);

}  // namespace mxq
