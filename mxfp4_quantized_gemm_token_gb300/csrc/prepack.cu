// prepack.cu — load-time weight prepack for fp8_scaled_mm.
//
// The pages prepare weights once after loading: "[CPU] fp8_per_tensor_scaled_mm_cpu"
// (implementation breakdown) transposes and packs the FP8 weight into the
// layout its AMX kernel reads, and "[XPU] block-FP8 linear via torch
// scaled_mm" (process_weights_after_loading_block_quant) stores the block
// scales transposed-contiguous.  The GPU counterpart:
//   - each 128-row x 128-byte weight tile (one MMA operand slice) is stored
//     as one contiguous 16 KB block holding exactly the 128-byte-swizzled
//     shared-memory image the tensor core reads, tiles of a row block
//     consecutive along K; the GEMM then streams a tile with one plain bulk
//     copy (contiguous DRAM bursts, no tensor map) instead of 128 rows of
//     128 bytes at the matrix row stride;
//   - the block scales are stored K-block-major, [ceil(K/128), ceil(N/bn)]
//     contiguous, so the 128 row scales a weight tile needs per K slice are
//     one contiguous run.
// Rows past N and columns past K are zero in the packed tiles.
#include <cuda_runtime.h>

#include <algorithm>
#include <string>

#include "internal.h"
#include "mxq.h"

namespace mxq {

namespace {

// One CTA per packed tile (row block tn, K slice kb): 1024 16-byte chunks,
// chunk c of row r goes to r * 128 + ((c ^ (r & 7)) << 4).
__global__ void __launch_bounds__(256) prepack_tiles_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                            int64_t K, int64_t ldw, int nkb,
                                                            uint8_t* __restrict__ Wp) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t tile = blockIdx.x;
  const int64_t tn = tile / nkb, kb = tile - tn * nkb;
  uint8_t* dst = Wp + tile * 16384;
  for (int i = threadIdx.x; i < 1024; i += 256) {
    const int r = i >> 3, c = i & 7;
    const int64_t n = tn * 128 + r, k0 = kb * 128 + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) {
      const uint8_t* src = W + n * ldw + k0;
      if (k0 + 16 <= K) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else if (k0 < K) {
        uint8_t b[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) b[j] = (k0 + j < K) ? __ldg(src + j) : 0;
        v = *reinterpret_cast<const uint4*>(b);
      }
    }
    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
}

// ws_p[kb * nbn + nb] = w_scale[nb * sw0 + kb * sw1]
__global__ void prepack_scales_kernel(const float* __restrict__ ws, int64_t nbn, int64_t nkb,
                                      int64_t sw0, int64_t sw1, float* __restrict__ ws_p) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t total = nbn * nkb;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t kb = i / nbn, nb = i - kb * nbn;
    ws_p[i] = __ldg(ws + nb * sw0 + kb * sw1);
  }
}

bool block_args(int32_t block_n, int32_t block_k, bool* per_tensor) {
  *per_tensor = block_n == 0 && block_k == 0;
  return *per_tensor || (block_k == 128 && (block_n == 1 || block_n == 128));
}

}  // namespace

}  // namespace mxq

using namespace mxq;

extern "C" mxq_status mxq_prepacked_weight_size(int64_t N, int64_t K, int32_t block_n,
                                                int32_t block_k, size_t* w_bytes,
                                                size_t* s_bytes) {
  bool pt = false;
  if (!w_bytes || !s_bytes || N < 0 || K <= 0) {
    set_last_error("prepacked_weight_size: need N >= 0, K > 0 and non-NULL results");
    return MXQ_ERR_INVALID_ARG;
  }
  if (!block_args(block_n, block_k, &pt)) {
    set_last_error("weight block size must be [128, 128], [1, 128] or per-tensor [0, 0]");
    return MXQ_ERR_UNSUPPORTED;
  }
  const int64_t tiles = (N + 127) / 128 * ((K + 127) / 128);
  *w_bytes = static_cast<size_t>(tiles) * 16384;
  *s_bytes = pt ? sizeof(float)
                : static_cast<size_t>((N + block_n - 1) / block_n) * ((K + 127) / 128) * sizeof(float);
  return MXQ_OK;
}

extern "C" mxq_status mxq_prepack_weight(const void* W, int64_t N, int64_t K, int64_t ldw,
                                         const float* w_scale, int32_t block_n, int32_t block_k,
                                         int64_t sw0, int64_t sw1, void* Wp, float* ws_p,
                                         mxq_stream_t stream) {
  bool pt = false;
  if (N < 0 || K <= 0) {
    set_last_error("prepack_weight: need N >= 0 and K > 0");
    return MXQ_ERR_INVALID_ARG;
  }
  if (!block_args(block_n, block_k, &pt)) {
    set_last_error("weight block size must be [128, 128], [1, 128] or per-tensor [0, 0]");
    return MXQ_ERR_UNSUPPORTED;
  }
  if (N == 0) return MXQ_OK;
  if (!W || !w_scale || !Wp || !ws_p) {
    set_last_error("prepack_weight: W, w_scale, Wp and ws_p must be non-NULL");
    return MXQ_ERR_INVALID_ARG;
  }
  if (ldw < K || ldw % 16 != 0 || (reinterpret_cast<uintptr_t>(W) & 15) != 0) {
    set_last_error("prepack_weight: W needs a 16-byte aligned base and ldw >= K, a multiple of 16");
    return MXQ_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(Wp) & 255) != 0 || (reinterpret_cast<uintptr_t>(ws_p) & 15) != 0) {
    set_last_error("prepack_weight: Wp must be 256-byte and ws_p 16-byte aligned");
    return MXQ_ERR_INVALID_ARG;
  }
  if (N > (1 << 30) || K > (1 << 30)) {
    set_last_error("prepack_weight: dimensions above 2^30");
    return MXQ_ERR_UNSUPPORTED;
  }
  if (!pt && (sw0 < 0 || sw1 < 0)) {
    set_last_error("prepack_weight: negative scale strides");
    return MXQ_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) {
    set_last_error(err);
    return MXQ_ERR_UNSUPPORTED;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nkb = (K + 127) / 128, tiles = (N + 127) / 128 * nkb;
  cudaError_t e = launch_k(prepack_tiles_kernel, dim3(static_cast<unsigned>(tiles)), dim3(256), 0,
                           st, reinterpret_cast<const uint8_t*>(W), N, K, ldw,
                           static_cast<int>(nkb), reinterpret_cast<uint8_t*>(Wp));
  if (e == cudaSuccess) {
    const int64_t nbn = pt ? 1 : (N + block_n - 1) / block_n;
    const int64_t kbs = pt ? 1 : nkb;
    const int64_t blocks = std::min<int64_t>((nbn * kbs + 255) / 256, 4096);
    e = launch_k(prepack_scales_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                 w_scale, nbn, kbs, pt ? 0 : sw0, pt ? 0 : sw1, ws_p);
  }
  if (e != cudaSuccess) {
    set_last_error(std::string("prepack launch: ") + cudaGetErrorString(e));
    return MXQ_ERR_CUDA;
  }
  return MXQ_OK;
}
