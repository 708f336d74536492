// api.cu — the extern "C" entry points of libmxq (declared in mxq.h):
// host-side validation, tensor-map encoding, work planning and launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "mxq.h"

namespace mxq {

// One status word per device, read and cleared by mxq_sync_status.
__device__ int g_status_word;

namespace {

thread_local std::string g_err;

mxq_status fail(mxq_status st, const std::string& msg) {
  g_err = msg;
  return st;
}

mxq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MXQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

std::atomic<int64_t> g_opts[13] = {0, 4, 0, 2000000000LL, 0, 0, 0, 0, 0, 1, 0, 3, 0};

std::mutex g_dev_mu;
DeviceInfo g_devs[64];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

void set_last_error(const std::string& msg) { g_err = msg; }

int64_t option(int32_t which) {
  if (which < 0 || which >= static_cast<int32_t>(sizeof(g_opts) / sizeof(g_opts[0]))) return 0;
  return g_opts[which].load();
}

bool device_info(DeviceInfo* info, std::string* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return false;
  }
  if (dev < 0 || dev >= 64) {
    *err = "device index out of range";
    return false;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_devs[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    if ((e = cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&n.num_sms, cudaDevAttrMultiProcessorCount, dev))) {
      *err = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
      return false;
    }
    if (n.cc_major != 10 || n.cc_minor != 3) {
      *err = "libmxq is built for sm_103a (GB300); this device is compute capability " +
             std::to_string(n.cc_major) + "." + std::to_string(n.cc_minor);
      return false;
    }
    d = n;
  }
  *info = d;
  // The status word's device address is looked up on every call (a cheap
  // host-side query) rather than cached, so a reset device or another
  // context on it never receives a stale address.
  void* p = nullptr;
  if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) {
    *err = std::string("cudaGetSymbolAddress(status): ") + cudaGetErrorString(e);
    return false;
  }
  info->status = reinterpret_cast<int*>(p);
  return true;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle, std::string* err) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    *err = "cuTensorMapEncodeTiled is unavailable";
    return false;
  }
  std::memset(map, 0, sizeof(*map));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (code " + std::to_string(static_cast<int>(r)) + ")";
    return false;
  }
  return true;
}

}  // namespace mxq

using namespace mxq;

// ------------------------------------------------------------------- misc

extern "C" const char* mxq_last_error(void) { return g_err.c_str(); }

extern "C" const char* mxq_version(void) { return "mxq 0.1 (sm_103a, tcgen05)"; }

extern "C" mxq_status mxq_set_option(int32_t opt, int64_t value) {
  if (opt < MXQ_OPT_SMALL_M_MAX || opt > MXQ_OPT_FUSE_QUANT)
    return fail(MXQ_ERR_INVALID_ARG, "unknown option " + std::to_string(opt));
  if (opt == MXQ_OPT_NORMAL_TILE && value != 0 && value != 128 && value != 192 && value != 256)
    return fail(MXQ_ERR_INVALID_ARG, "NORMAL_TILE is 0 (auto), 128, 192 or 256");
  if (opt == MXQ_OPT_TILE_N && value != 0 && value != 32 && value != 64 && value != 128 &&
      value != 256)
    return fail(MXQ_ERR_INVALID_ARG, "TILE_N is 0 (auto), 32, 64, 128 or 256");
  if (value < 0) return fail(MXQ_ERR_INVALID_ARG, "option values are non-negative");
  if ((opt == MXQ_OPT_PDL || opt == MXQ_OPT_FUSE_COMBINE || opt == MXQ_OPT_FUSE_QUANT) &&
      value != 0 && value != 1)
    return fail(MXQ_ERR_INVALID_ARG, "PDL, FUSE_COMBINE and FUSE_QUANT are 0 (off) or 1 (on)");
  if (opt == MXQ_OPT_MOE_F16 && value > 3)
    return fail(MXQ_ERR_INVALID_ARG, "MOE_F16 is 0, 1, 2 or 3");
  if (opt == MXQ_OPT_FORCE_PATH && value > 3)
    return fail(MXQ_ERR_INVALID_ARG,
                "FORCE_PATH is 0 (per block), 1 (narrow), 2 (full width) or 3 (one path per layer)");
  g_opts[opt].store(value);
  return MXQ_OK;
}

extern "C" mxq_status mxq_get_option(int32_t opt, int64_t* value) {
  if (opt < MXQ_OPT_SMALL_M_MAX || opt > MXQ_OPT_FUSE_QUANT || value == nullptr)
    return fail(MXQ_ERR_INVALID_ARG, "unknown option or NULL value");
  *value = g_opts[opt].load();
  return MXQ_OK;
}

extern "C" mxq_status mxq_sync_status(mxq_stream_t stream) {
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  if ((e = cudaMemcpy(&word, d.status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the status word");
  if (word != 0) {
    const int zero = 0;
    if ((e = cudaMemcpy(d.status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clearing the status word");
  }
  if (word & kStatusTimeout)
    return fail(MXQ_ERR_TIMEOUT, "a bounded device wait expired; the kernel stopped early");
  if (word & kStatusBadIndex) return fail(MXQ_ERR_DEVICE, "an expert id outside [0, E) was skipped");
  return MXQ_OK;
}

// ------------------------------------------------------------- group quant

extern "C" mxq_status mxq_per_token_group_quant_fp8(const void* x, int64_t M, int64_t K,
                                                    int64_t ldx, int32_t group, float eps, void* q,
                                                    float* scales, mxq_stream_t stream) {
  if (M < 0 || K <= 0) return fail(MXQ_ERR_INVALID_ARG, "need M >= 0 and K > 0");
  if (M == 0) return MXQ_OK;
  if (!x || !q || !scales) return fail(MXQ_ERR_INVALID_ARG, "x, q and scales must be non-NULL");
  if (ldx < K) return fail(MXQ_ERR_INVALID_ARG, "ldx must be >= K");
  if (group < 8 || group > 1024 || group % 8 != 0)
    return fail(MXQ_ERR_UNSUPPORTED, "group must be a multiple of 8 in [8, 1024]");
  if (!(eps > 0.f) || !(eps < 3.4e38f))
    return fail(MXQ_ERR_INVALID_ARG, "eps must be positive and finite");
  if ((reinterpret_cast<uintptr_t>(x) & 1) != 0)
    return fail(MXQ_ERR_INVALID_ARG, "x must be 2-byte aligned");
  if ((reinterpret_cast<uintptr_t>(scales) & 3) != 0)
    return fail(MXQ_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  cudaError_t e = launch_group_quant(x, M, K, ldx, group, eps, q, scales, d.num_sms,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "group quant launch");
  return MXQ_OK;
}

// ---------------------------------------------------------- MXFP4 encode

extern "C" mxq_status mxq_quantize_mxfp4(const void* x, int32_t x_dtype, int64_t R, int64_t C,
                                         int64_t ldx, void* packed, void* scales,
                                         mxq_stream_t stream) {
  if (R < 0 || C <= 0) return fail(MXQ_ERR_INVALID_ARG, "need R >= 0 and C > 0");
  if (C % 32 != 0) return fail(MXQ_ERR_UNSUPPORTED, "C must be a multiple of 32");
  if (x_dtype != MXQ_BF16 && x_dtype != MXQ_F32)
    return fail(MXQ_ERR_UNSUPPORTED, "x_dtype must be MXQ_BF16 or MXQ_F32");
  if (R == 0) return MXQ_OK;
  if (!x || !packed || !scales) return fail(MXQ_ERR_INVALID_ARG, "NULL tensor argument");
  if (ldx < C) return fail(MXQ_ERR_INVALID_ARG, "ldx must be >= C");
  const int es = x_dtype == MXQ_BF16 ? 2 : 4;
  if (!aligned16(x) || (ldx * es) % 16 != 0 || !aligned16(packed))
    return fail(MXQ_ERR_UNSUPPORTED,
                "x and packed need 16-byte aligned bases and x rows a multiple of 16 bytes");
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  cudaError_t e = launch_mxfp4_quant(x, x_dtype == MXQ_BF16, R, C, ldx, packed, scales, d.num_sms,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MXFP4 quantization launch");
  return MXQ_OK;
}

// ------------------------------------------------------------ scaled mm

namespace {

struct MmPlan {
  int bt, kind, tiles_n, tiles_m, nkb, splits, kb_per_split;
  bool promote;
  bool normal;   // tokens on the MMA M side (EPI_NORMAL)
};

MmPlan plan_mm(int64_t M, int64_t N, int64_t K, int32_t a_dtype, bool block, bool has_ascale,
               int num_sms, bool uniform_wscale = true) {
  MmPlan pl;
  pl.kind = a_dtype == MXQ_E4M3 ? KIND_F8F8 : KIND_F8W;
  pl.bt = M <= 32 ? 32 : (M <= 64 ? 64 : 128);
  const int64_t tile = option(MXQ_OPT_TILE_N);
  if (tile > 0) pl.bt = (tile == 256 && pl.kind != KIND_F8F8) ? 128 : static_cast<int>(tile);
  // Large M: put the tokens on the MMA M side (each TMEM lane's token scale
  // is one scalar per slice; [1, 128] weight scales become a per-column
  // vector the scale warp stages)
  pl.normal = pl.kind == KIND_F8F8 && has_ascale && M > 128 && tile == 0;
  if (pl.normal) {
    const int64_t nt = option(MXQ_OPT_NORMAL_TILE);
    // 128-wide weight tiles: four TMEM accumulator buffers (one per slice in
    // flight) and two epilogue warpgroups of 64 columns; measured faster than
    // 192 (two buffers) and 256 (the epilogue spills) at M = 1024 and 4096
    pl.bt = (nt > 0 && uniform_wscale) ? static_cast<int>(nt) : 128;
  }
  pl.promote = block || has_ascale;
  pl.tiles_n = static_cast<int>(cdiv(N, pl.normal ? pl.bt : 128));
  pl.tiles_m = static_cast<int>(cdiv(M, pl.normal ? 128 : pl.bt));
  pl.nkb = static_cast<int>(cdiv(K, 128));
  const int64_t units = static_cast<int64_t>(pl.tiles_n) * pl.tiles_m;
  int splits = static_cast<int>(option(MXQ_OPT_SPLIT_K));
  if (splits <= 0) {
    splits = 1;
    if (units * 2 <= num_sms)
      splits = static_cast<int>(std::min<int64_t>(pl.nkb, num_sms / units));
    // keep at least 4 slices per split
    while (splits > 1 && cdiv(pl.nkb, splits) < 4) --splits;
  }
  splits = std::max(1, std::min(splits, pl.nkb));
  pl.kb_per_split = static_cast<int>(cdiv(pl.nkb, splits));
  pl.splits = static_cast<int>(cdiv(pl.nkb, pl.kb_per_split));
  return pl;
}

int sms_for_grid(const DeviceInfo& d) {
  const int64_t cap = option(MXQ_OPT_NUM_SMS);
  return (cap > 0 && cap < d.num_sms) ? static_cast<int>(cap) : d.num_sms;
}

}  // namespace

namespace mxq {

// Host-side argument checks of mxq_fp8_scaled_mm (and its no-alloc variant):
// MXQ_OK, or the status and message of the first problem found.  Sizes with
// M == 0 or N == 0 pass (the call is then a no-op).
mxq_status validate_mm(const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
                       const float* a_scale, int64_t sa0, int64_t sa1, const void* W, int64_t N,
                       int64_t ldw, const float* w_scale, int32_t block_n, int32_t block_k,
                       int64_t sw0, int64_t sw1, const void* bias, int32_t bias_dtype,
                       const void* out, int32_t out_dtype, int64_t ldo) {
  if (M < 0 || N < 0 || K <= 0) return fail(MXQ_ERR_INVALID_ARG, "need M, N >= 0 and K > 0");
  if (M == 0 || N == 0) return MXQ_OK;
  if (!A || !W || !out || !w_scale)
    return fail(MXQ_ERR_INVALID_ARG, "A, W, w_scale and out must be non-NULL");
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30))
    return fail(MXQ_ERR_UNSUPPORTED, "dimensions above 2^30");
  if (a_dtype != MXQ_E4M3 && a_dtype != MXQ_BF16)
    return fail(MXQ_ERR_UNSUPPORTED, "a_dtype must be MXQ_E4M3 (W8A8) or MXQ_BF16 (W8A16)");
  const bool per_tensor = block_n == 0 && block_k == 0;
  const bool block = block_k == 128 && (block_n == 1 || block_n == 128);
  if (!per_tensor && !block)
    return fail(MXQ_ERR_UNSUPPORTED,
                "weight block size must be [128, 128], [1, 128] or per-tensor [0, 0]; got [" +
                    std::to_string(block_n) + ", " + std::to_string(block_k) + "]");
  if (a_dtype == MXQ_E4M3 && !a_scale)
    return fail(MXQ_ERR_INVALID_ARG, "W8A8 needs the activation group scales a_scale");
  if (a_dtype == MXQ_BF16 && a_scale)
    return fail(MXQ_ERR_INVALID_ARG, "bf16 activations take no activation scale");
  if (out_dtype != MXQ_BF16 && out_dtype != MXQ_F32)
    return fail(MXQ_ERR_UNSUPPORTED, "out_dtype must be MXQ_BF16 or MXQ_F32");
  if (bias && bias_dtype != MXQ_F32 && bias_dtype != MXQ_BF16)
    return fail(MXQ_ERR_UNSUPPORTED, "bias_dtype must be MXQ_F32 or MXQ_BF16");
  if (lda < K || ldw < K || ldo < N)
    return fail(MXQ_ERR_INVALID_ARG, "row strides below the row length");
  const int aes = a_dtype == MXQ_E4M3 ? 1 : 2;
  if (!aligned16(A) || (lda * aes) % 16 != 0 || !aligned16(W) || ldw % 16 != 0)
    return fail(MXQ_ERR_UNSUPPORTED,
                "A and W need 16-byte aligned bases and row strides that are multiples of 16 bytes");
  if (block && (sw0 < 0 || sw1 < 0 || (a_scale && (sa0 < 0 || sa1 < 0))))
    return fail(MXQ_ERR_INVALID_ARG, "negative scale strides");
  return MXQ_OK;
}

}  // namespace mxq

namespace {

// The plan mxq_fp8_scaled_mm runs for a validated argument set.  The
// workspace query and the no-alloc entry point use the same function, so the
// size they report is the size of the split the call actually makes.
MmPlan plan_for_call(int64_t M, int64_t N, int64_t K, int32_t a_dtype, int32_t block_n,
                     int32_t block_k, int sms) {
  const bool block = !(block_n == 0 && block_k == 0);
  return plan_mm(M, N, K, a_dtype, block, a_dtype == MXQ_E4M3, sms, block_n != 1);
}

size_t plan_workspace_bytes(const MmPlan& pl, int64_t M, int64_t N) {
  return pl.splits > 1 ? static_cast<size_t>(pl.splits) * M * N * sizeof(float) : 0;
}

}  // namespace

namespace mxq {

mxq_status mm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t a_dtype, int32_t block_n,
                              int32_t block_k, size_t* bytes) {
  *bytes = 0;
  if (M == 0 || N == 0) return MXQ_OK;
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  *bytes = plan_workspace_bytes(plan_for_call(M, N, K, a_dtype, block_n, block_k, sms_for_grid(d)),
                                M, N);
  return MXQ_OK;
}

}  // namespace mxq

extern "C" mxq_status mxq_fp8_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K,
                                                       int32_t a_dtype, int32_t block_n,
                                                       int32_t block_k, size_t* bytes) {
  if (!bytes || M < 0 || N < 0 || K <= 0)
    return fail(MXQ_ERR_INVALID_ARG, "bad sizes or NULL result pointer");
  if (a_dtype != MXQ_E4M3 && a_dtype != MXQ_BF16)
    return fail(MXQ_ERR_UNSUPPORTED, "a_dtype must be MXQ_E4M3 (W8A8) or MXQ_BF16 (W8A16)");
  if (!(block_n == 0 && block_k == 0) && !(block_k == 128 && (block_n == 1 || block_n == 128)))
    return fail(MXQ_ERR_UNSUPPORTED,
                "weight block size must be [128, 128], [1, 128] or per-tensor [0, 0]");
  return mm_workspace_bytes(M, N, K, a_dtype, block_n, block_k, bytes);
}

namespace {

// The scaled GEMM for validated arguments with M, N > 0.  W is the weight
// matrix (row stride ldw) or, when wpacked is set, unused: the weights are
// then the prepacked tiles of mxq_prepack_weight.
mxq_status scaled_mm_run(const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
                         const float* a_scale, int64_t sa0, int64_t sa1, const void* W, int64_t N,
                         int64_t ldw, const uint8_t* wpacked, const float* w_scale,
                         int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
                         const void* bias, int32_t bias_dtype, void* out, int32_t out_dtype,
                         int64_t ldo, void* workspace, size_t ws_bytes, mxq_stream_t stream) {
  const bool per_tensor = block_n == 0 && block_k == 0;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 15) != 0)
    return fail(MXQ_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  const int sms = sms_for_grid(d);
  MmPlan pl = plan_for_call(M, N, K, a_dtype, block_n, block_k, sms);
  const size_t need = plan_workspace_bytes(pl, M, N);
  if (need > 0) {
    if (workspace == nullptr) {
      // no workspace: the same GEMM without split-K
      pl.splits = 1;
      pl.kb_per_split = pl.nkb;
    } else if (ws_bytes < need) {
      return fail(MXQ_ERR_INVALID_ARG,
                  "workspace of " + std::to_string(ws_bytes) + " bytes is smaller than the " +
                      std::to_string(need) +
                      " this shape's split-K plan needs (mxq_fp8_scaled_mm_workspace_size)");
    }
  }

  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const int bv = pl.bt == 32 ? 1 : (pl.bt == 64 ? 2 : (pl.bt == 128 ? 3 : 4));
  if (pl.normal) {
    // MMA A = tokens (128-row boxes), MMA B = weights (bt-row boxes)
    if (!make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, lda, 128, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B, &err) ||
        (wpacked == nullptr &&
         !make_map_2d(&maps.b[bv], CU_TENSOR_MAP_DATA_TYPE_UINT8, W, K, N, ldw, 128, pl.bt,
                      CU_TENSOR_MAP_SWIZZLE_128B, &err)))
      return fail(MXQ_ERR_CUDA, err);
  } else if (wpacked == nullptr &&
             !make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, K, N, ldw, 128, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B, &err)) {
    return fail(MXQ_ERR_CUDA, err);
  }
  if (pl.normal) {
  } else if (a_dtype == MXQ_E4M3) {
    if (!make_map_2d(&maps.b[bv], CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, lda, 128, pl.bt,
                     CU_TENSOR_MAP_SWIZZLE_128B, &err))
      return fail(MXQ_ERR_CUDA, err);
  } else {
    if (!make_map_2d(&maps.b[bv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, pl.bt,
                     CU_TENSOR_MAP_SWIZZLE_128B, &err))
      return fail(MXQ_ERR_CUDA, err);
  }

  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = pl.nkb;
  p.tiles_n = pl.tiles_n;
  p.tiles_m = pl.tiles_m;
  p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split;
  p.a_scale = a_scale;
  p.sa0 = sa0;
  p.sa1 = sa1;
  p.w_scale = w_scale;
  p.sw0 = sw0;
  p.sw1 = sw1;
  p.block_n = per_tensor ? 0 : block_n;
  p.bias = bias;
  p.bias_dtype = bias ? bias_dtype : 0;
  p.out = out;
  p.out_dtype = out_dtype;
  p.ldo = ldo;
  p.partial = pl.splits > 1 ? reinterpret_cast<float*>(workspace) : nullptr;
  p.wpacked = wpacked;
  p.npad = static_cast<int>(cdiv(N, 128) * 128);
  p.status = d.status;
  p.budget_ns = static_cast<unsigned long long>(option(MXQ_OPT_WAIT_BUDGET_NS));
  p.inject_stall = static_cast<int>(option(MXQ_OPT_INJECT_STALL));
  const uintptr_t ob = reinterpret_cast<uintptr_t>(out);
  if (pl.normal)   // 16-byte row chunks of 8 outputs
    p.vec_ok = (out_dtype == MXQ_BF16) ? (ldo % 8 == 0 && (ob & 15) == 0)
                                        : (ldo % 4 == 0 && (ob & 15) == 0);
  else
    p.vec_ok = (ldo % 4 == 0) && ((out_dtype == MXQ_BF16) ? (ob & 7) == 0 : (ob & 15) == 0);

  const int64_t units = static_cast<int64_t>(pl.tiles_n) * pl.tiles_m * pl.splits;
  const int grid = static_cast<int>(std::min<int64_t>(units, sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int epi = !pl.normal ? EPI_DENSE : (block_n == 1 ? EPI_NORMAL_COLW : EPI_NORMAL);
  cudaError_t e = launch_gemm(pl.kind, epi, pl.bt, pl.promote,
                              maps, p, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "scaled-mm launch");
  if (pl.splits > 1) {
    e = launch_splitk_reduce(p.partial, pl.splits, M, N, bias, p.bias_dtype, out, out_dtype, ldo,
                             st);
    if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  }
  return MXQ_OK;
}

}  // namespace

extern "C" mxq_status mxq_fp8_scaled_mm(const void* A, int32_t a_dtype, int64_t M, int64_t K,
                                        int64_t lda, const float* a_scale, int64_t sa0,
                                        int64_t sa1, const void* W, int64_t N, int64_t ldw,
                                        const float* w_scale, int32_t block_n, int32_t block_k,
                                        int64_t sw0, int64_t sw1, const void* bias,
                                        int32_t bias_dtype, void* out, int32_t out_dtype,
                                        int64_t ldo, void* workspace, size_t ws_bytes,
                                        mxq_stream_t stream) {
  const mxq_status vst = validate_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, w_scale,
                                     block_n, block_k, sw0, sw1, bias, bias_dtype, out, out_dtype,
                                     ldo);
  if (vst != MXQ_OK) return vst;
  if (M == 0 || N == 0) return MXQ_OK;
  return scaled_mm_run(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, nullptr, w_scale,
                       block_n, block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo,
                       workspace, ws_bytes, stream);
}

extern "C" mxq_status mxq_fp8_scaled_mm_prepacked(
    const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda, const float* a_scale,
    int64_t sa0, int64_t sa1, const void* Wp, int64_t N, const float* ws_p, int32_t block_n,
    int32_t block_k, const void* bias, int32_t bias_dtype, void* out, int32_t out_dtype,
    int64_t ldo, void* workspace, size_t ws_bytes, mxq_stream_t stream) {
  // the packed scales are K-block-major: Ws[nb, kb] = ws_p[kb * ceil(N / bn) + nb]
  const bool per_tensor = block_n == 0 && block_k == 0;
  const int64_t nbn = per_tensor || block_n <= 0 ? 1 : cdiv(N, block_n);
  const mxq_status vst =
      validate_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, Wp, N, cdiv(K, 16) * 16, ws_p,
                  block_n, block_k, 1, nbn, bias, bias_dtype, out, out_dtype, ldo);
  if (vst != MXQ_OK) return vst;
  if (M == 0 || N == 0) return MXQ_OK;
  if ((reinterpret_cast<uintptr_t>(Wp) & 255) != 0)
    return fail(MXQ_ERR_INVALID_ARG, "prepacked weights must be 256-byte aligned");
  return scaled_mm_run(A, a_dtype, M, K, lda, a_scale, sa0, sa1, nullptr, N, 0,
                       reinterpret_cast<const uint8_t*>(Wp), ws_p, block_n, block_k, 1, nbn, bias,
                       bias_dtype, out, out_dtype, ldo, workspace, ws_bytes, stream);
}

extern "C" mxq_status mxq_fp8_scaled_bmm(
    int64_t batch, const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
    int64_t a_bstride, const float* a_scale, int64_t sa0, int64_t sa1, int64_t sa_bstride,
    const void* W, int64_t N, int64_t ldw, int64_t w_bstride, const float* w_scale,
    int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1, int64_t sw_bstride,
    const void* bias, int32_t bias_dtype, int64_t bias_bstride, void* out, int32_t out_dtype,
    int64_t ldo, int64_t out_bstride, mxq_stream_t stream) {
  if (batch < 0) return fail(MXQ_ERR_INVALID_ARG, "batch must be >= 0");
  if (batch == 0) return MXQ_OK;
  const mxq_status vst = validate_mm(A, a_dtype, M, K, lda, a_scale, sa0, sa1, W, N, ldw, w_scale,
                                     block_n, block_k, sw0, sw1, bias, bias_dtype, out, out_dtype,
                                     ldo);
  if (vst != MXQ_OK) return vst;
  if (M == 0 || N == 0) return MXQ_OK;
  if (a_bstride != M * lda || w_bstride != N * ldw)
    return fail(MXQ_ERR_UNSUPPORTED,
                "A and W batches must be stacked contiguously (a_bstride = M*lda, w_bstride = N*ldw)");
  if (sa_bstride < 0 || sw_bstride < 0 || bias_bstride < 0 || out_bstride < 0)
    return fail(MXQ_ERR_INVALID_ARG, "negative batch strides");
  if (batch * M >= (1LL << 31) || batch * N >= (1LL << 31))
    return fail(MXQ_ERR_UNSUPPORTED, "batch * M and batch * N must stay below 2^31");
  const bool per_tensor = block_n == 0 && block_k == 0;
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  const int sms = sms_for_grid(d);
  // weight-major tiles (tokens on the MMA N side), no split-K: the batch
  // itself provides the parallelism of the small per-head problems
  MmPlan pl = plan_for_call(M, N, K, a_dtype, block_n, block_k, sms);
  if (pl.normal) {
    pl.normal = false;
    pl.bt = M <= 32 ? 32 : (M <= 64 ? 64 : 128);
    pl.tiles_n = static_cast<int>(cdiv(N, 128));
    pl.tiles_m = static_cast<int>(cdiv(M, pl.bt));
  }
  pl.splits = 1;
  pl.kb_per_split = pl.nkb;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const int bv = pl.bt == 32 ? 1 : (pl.bt == 64 ? 2 : (pl.bt == 128 ? 3 : 4));
  if (!make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, K, batch * N, ldw, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B, &err))
    return fail(MXQ_ERR_CUDA, err);
  if (a_dtype == MXQ_E4M3) {
    if (!make_map_2d(&maps.b[bv], CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, batch * M, lda, 128, pl.bt,
                     CU_TENSOR_MAP_SWIZZLE_128B, &err))
      return fail(MXQ_ERR_CUDA, err);
  } else if (!make_map_2d(&maps.b[bv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, batch * M, lda * 2,
                          64, pl.bt, CU_TENSOR_MAP_SWIZZLE_128B, &err)) {
    return fail(MXQ_ERR_CUDA, err);
  }
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = pl.nkb;
  p.tiles_n = pl.tiles_n;
  p.tiles_m = pl.tiles_m;
  p.splits = 1;
  p.kb_per_split = pl.nkb;
  p.batch = static_cast<int>(batch);
  p.a_scale = a_scale;
  p.sa0 = sa0;
  p.sa1 = sa1;
  p.sa_e = sa_bstride;
  p.w_scale = w_scale;
  p.sw0 = sw0;
  p.sw1 = sw1;
  p.sw_e = sw_bstride;
  p.block_n = per_tensor ? 0 : block_n;
  p.bias = bias;
  p.bias_dtype = bias ? bias_dtype : 0;
  p.bias_e = bias_bstride;
  p.out = out;
  p.out_dtype = out_dtype;
  p.ldo = ldo;
  p.out_e = out_bstride;
  p.npad = static_cast<int>(cdiv(N, 128) * 128);
  p.status = d.status;
  p.budget_ns = static_cast<unsigned long long>(option(MXQ_OPT_WAIT_BUDGET_NS));
  p.inject_stall = static_cast<int>(option(MXQ_OPT_INJECT_STALL));
  const uintptr_t ob = reinterpret_cast<uintptr_t>(out);
  p.vec_ok = (ldo % 4 == 0) && (out_bstride % 4 == 0) &&
             ((out_dtype == MXQ_BF16) ? (ob & 7) == 0 : (ob & 15) == 0);
  const int64_t units = static_cast<int64_t>(pl.tiles_n) * pl.tiles_m * batch;
  if (units >= (1LL << 31)) return fail(MXQ_ERR_UNSUPPORTED, "too many tiles");
  const int grid = static_cast<int>(std::min<int64_t>(units, sms));
  cudaError_t e = launch_gemm(pl.kind, EPI_DENSE, pl.bt, pl.promote, maps, p, grid,
                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scaled-bmm launch");
  return MXQ_OK;
}

// ------------------------------------------------ block-FP8 linear (bf16 in)

namespace {

// token rows up to which the linear quantizes inside the GEMM (one 32-wide
// token tile; every weight tile re-quantizes the tokens it needs)
constexpr int64_t kFusedQuantMaxM = 32;

struct LinearWs {
  size_t q, s, part, total;
  bool fused;
};

mxq_status linear_ws(int64_t M, int64_t N, int64_t K, int32_t block_n, int sms, LinearWs* w) {
  const MmPlan pl = plan_for_call(M, N, K, MXQ_E4M3, block_n, 128, sms);
  w->fused = M <= kFusedQuantMaxM && option(MXQ_OPT_FUSE_QUANT) != 0 && !pl.normal && pl.bt == 32;
  size_t o = 0;
  w->q = w->s = 0;
  if (!w->fused) {
    w->q = o;
    o = round_up(o + static_cast<size_t>(M) * K, 256);
    w->s = o;
    o = round_up(o + static_cast<size_t>(M) * cdiv(K, 128) * sizeof(float), 256);
  }
  w->part = o;
  o = round_up(o + plan_workspace_bytes(pl, M, N), 256);
  w->total = o;
  return MXQ_OK;
}

}  // namespace

extern "C" mxq_status mxq_w8a8_block_fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K,
                                                               int32_t block_n, size_t* bytes) {
  if (!bytes || M < 0 || N < 0 || K <= 0)
    return fail(MXQ_ERR_INVALID_ARG, "bad sizes or NULL result pointer");
  if (block_n != 1 && block_n != 128)
    return fail(MXQ_ERR_UNSUPPORTED, "block_n must be 1 or 128");
  *bytes = 0;
  if (M == 0 || N == 0) return MXQ_OK;
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  LinearWs w;
  linear_ws(M, N, K, block_n, sms_for_grid(d), &w);
  *bytes = w.total;
  return MXQ_OK;
}

extern "C" mxq_status mxq_w8a8_block_fp8_linear(
    const void* x, int64_t M, int64_t K, int64_t ldx, const void* W, int64_t N, int64_t ldw,
    const float* w_scale, int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
    const void* bias, int32_t bias_dtype, void* out, int32_t out_dtype, int64_t ldo,
    void* workspace, size_t ws_bytes, mxq_stream_t stream) {
  if (M < 0 || N < 0 || K <= 0) return fail(MXQ_ERR_INVALID_ARG, "need M, N >= 0 and K > 0");
  if (!(block_k == 128 && (block_n == 1 || block_n == 128)))
    return fail(MXQ_ERR_UNSUPPORTED,
                "weight block size must be [128, 128] or [1, 128]; got [" +
                    std::to_string(block_n) + ", " + std::to_string(block_k) + "]");
  if (M == 0 || N == 0) return MXQ_OK;
  if (!x) return fail(MXQ_ERR_INVALID_ARG, "x must be non-NULL");
  if (ldx < K) return fail(MXQ_ERR_INVALID_ARG, "ldx must be >= K");
  if (!aligned16(x) || (ldx * 2) % 16 != 0)
    return fail(MXQ_ERR_UNSUPPORTED, "x needs a 16-byte aligned base and rows a multiple of 16 bytes");
  // the rest of the checks are those of the W8A8 GEMM (a stand-in pointer for
  // the quantized activations and their scales)
  const mxq_status vst =
      validate_mm(x, MXQ_E4M3, M, K, cdiv(K, 16) * 16, w_scale, 1, 1, W, N, ldw, w_scale, block_n,
                  block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo);
  if (vst != MXQ_OK) return vst;
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  LinearWs w;
  linear_ws(M, N, K, block_n, sms_for_grid(d), &w);
  if (w.total > 0 && (workspace == nullptr || ws_bytes < w.total ||
                      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
    return fail(MXQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned and hold " +
                                         std::to_string(w.total) +
                                         " bytes (mxq_w8a8_block_fp8_linear_workspace_size)");
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!w.fused) {
    // separate per-token-group quantization, then the W8A8 GEMM
    if (K % 16 != 0)
      return fail(MXQ_ERR_UNSUPPORTED,
                  "above the fused-quantization size, K must be a multiple of 16");
    void* q = ws + w.q;
    float* sc = reinterpret_cast<float*>(ws + w.s);
    cudaError_t e = launch_group_quant(x, M, K, ldx, 128, 1e-10f, q, sc, d.num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "group quant launch");
    return scaled_mm_run(q, MXQ_E4M3, M, K, K, sc, cdiv(K, 128), 1, W, N, ldw, nullptr, w_scale,
                         block_n, block_k, sw0, sw1, bias, bias_dtype, out, out_dtype, ldo,
                         w.total > w.part ? ws + w.part : nullptr, w.total - w.part, stream);
  }
  // fused: bf16 tokens are quantized per 1 x 128 group inside the GEMM
  const int sms = sms_for_grid(d);
  MmPlan pl = plan_for_call(M, N, K, MXQ_E4M3, block_n, block_k, sms);
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, K, N, ldw, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B, &err) ||
      !make_map_2d(&maps.b[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B, &err))
    return fail(MXQ_ERR_CUDA, err);
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = pl.nkb;
  p.tiles_n = pl.tiles_n;
  p.tiles_m = pl.tiles_m;
  p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split;
  p.a_scale = nullptr;   // the group scales come from the quantizer warps
  p.w_scale = w_scale;
  p.sw0 = sw0;
  p.sw1 = sw1;
  p.block_n = block_n;
  p.bias = bias;
  p.bias_dtype = bias ? bias_dtype : 0;
  p.out = out;
  p.out_dtype = out_dtype;
  p.ldo = ldo;
  p.partial = pl.splits > 1 ? reinterpret_cast<float*>(ws + w.part) : nullptr;
  p.npad = static_cast<int>(cdiv(N, 128) * 128);
  p.q_eps = 1e-10f;
  p.status = d.status;
  p.budget_ns = static_cast<unsigned long long>(option(MXQ_OPT_WAIT_BUDGET_NS));
  p.inject_stall = static_cast<int>(option(MXQ_OPT_INJECT_STALL));
  const uintptr_t ob = reinterpret_cast<uintptr_t>(out);
  p.vec_ok = (ldo % 4 == 0) && ((out_dtype == MXQ_BF16) ? (ob & 7) == 0 : (ob & 15) == 0);
  const int64_t units = static_cast<int64_t>(pl.tiles_n) * pl.tiles_m * pl.splits;
  const int grid = static_cast<int>(std::min<int64_t>(units, sms));
  cudaError_t e = launch_gemm(KIND_F8Q, EPI_DENSE, 32, true, maps, p, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "fused linear launch");
  if (pl.splits > 1) {
    e = launch_splitk_reduce(p.partial, pl.splits, M, N, bias, p.bias_dtype, out, out_dtype, ldo,
                             st);
    if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  }
  return MXQ_OK;
}

// ------------------------------------------------------------- moe_align

extern "C" mxq_status mxq_moe_align_block(const int32_t* topk_ids, int64_t T, int32_t topk,
                                          int32_t E, int32_t block_m, int32_t* sorted_ids,
                                          int32_t* expert_ids, int32_t* offsets,
                                          int32_t* num_blocks, int64_t cap, void* workspace,
                                          size_t ws_bytes, mxq_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  if (T < 0 || topk <= 0) return fail(MXQ_ERR_INVALID_ARG, "need T >= 0 and topk > 0");
  if (E < 1 || E > 1024) return fail(MXQ_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128)
    return fail(MXQ_ERR_UNSUPPORTED, "block_m must be 16, 32, 64 or 128");
  if (!sorted_ids || !expert_ids || !offsets || !num_blocks || (T > 0 && !topk_ids))
    return fail(MXQ_ERR_INVALID_ARG, "NULL output or id array");
  const int64_t S = T * topk;
  if (S >= (1LL << 30)) return fail(MXQ_ERR_UNSUPPORTED, "too many slots");
  const int64_t need = cdiv(S, block_m) + std::min<int64_t>(E, S);
  if (cap < need)
    return fail(MXQ_ERR_INVALID_ARG,
                "cap must be >= ceil(S/block_m) + min(E, S) = " + std::to_string(need));
  if (cap * block_m >= (1LL << 31)) return fail(MXQ_ERR_UNSUPPORTED, "cap too large");
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  cudaError_t e = launch_moe_align(topk_ids, S, E, block_m, sorted_ids, expert_ids, offsets,
                                   num_blocks, cap, d.status, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_align launch");
  return MXQ_OK;
}

// ------------------------------------------------------------ fused MoE

namespace {

struct MoeWs {
  size_t sorted, experts, offsets, nblocks, xs, ic1, y, cnt, hf16, tscale, rs1, ic1h, rs2, emax,
      total;
  int64_t S, cap, ncnt;
};

// block_m 0: the library's choice.  Expert blocks of 32 slots let the
// weight-decode warps of the FP8-block GEMM run as two groups (the registers
// of a 64-wide tile do not allow it); when experts average more than 16
// slots, 32-slot blocks would split experts and stream their weights twice,
// so 64.  (MXFP4 runs two decode groups at either width.)
int32_t resolve_block_m(int32_t block_m, int64_t S, int32_t E) {
  if (block_m != 0) return block_m;
  return S <= 16 * static_cast<int64_t>(E) ? 32 : 64;
}

MoeWs moe_ws(int64_t T, int64_t K, int32_t E, int64_t N, int32_t topk, int32_t block_m) {
  MoeWs w;
  w.S = T * topk;
  w.cap = cdiv(w.S, block_m) + std::min<int64_t>(E, w.S);
  size_t o = 0;
  w.sorted = o;
  o = round_up(o + static_cast<size_t>(w.cap) * block_m * 4, 256);
  w.experts = o;
  o = round_up(o + static_cast<size_t>(w.cap) * 4, 256);
  w.offsets = o;
  o = round_up(o + static_cast<size_t>(w.cap + 1) * 4, 256);
  w.nblocks = o;
  o = round_up(o + 4, 256);
  w.xs = o;
  o = round_up(o + static_cast<size_t>(w.S) * K * 2, 256);
  w.ic1 = o;
  o = round_up(o + static_cast<size_t>(w.S) * N * 2, 256);
  w.y = o;
  o = round_up(o + static_cast<size_t>(w.S) * K * 4, 256);
  // fused combine: one counter per (token, 128-row tile of the K outputs)
  w.cnt = o;
  w.ncnt = T * cdiv(K, 128);
  o = round_up(o + static_cast<size_t>(w.ncnt) * 4, 256);
  // f16 operands: the token rows, their scales, the compact rows' scales, the
  // stage-2 input and its row scales
  w.hf16 = o;
  o = round_up(o + static_cast<size_t>(T) * K * 2, 256);
  w.tscale = o;
  o = round_up(o + static_cast<size_t>(T) * 4, 256);
  w.rs1 = o;
  o = round_up(o + static_cast<size_t>(w.S) * 4, 256);
  w.ic1h = o;
  o = round_up(o + static_cast<size_t>(w.S) * N * 2, 256);
  w.rs2 = o;
  o = round_up(o + static_cast<size_t>(w.S) * 4, 256);
  // MXFP4 with f16 operands: the largest scale exponent of every expert row
  // (W1 rows, then W2 rows)
  w.emax = o;
  o = round_up(o + static_cast<size_t>(E) * (2 * N + K), 256);
  w.total = o;
  return w;
}

mxq_status fused_experts_impl(const void* hidden, int64_t T, int64_t K, int64_t ldh, int32_t wtype,
                              int32_t E, int64_t N, const void* w1, const void* w1_scale,
                              const float* w1_bias, const void* w2, const void* w2_scale,
                              const float* w2_bias, const float* topk_weights,
                              const int32_t* topk_ids, int32_t topk, int32_t block_m, void* out,
                              int64_t ldo, void* workspace, size_t ws_bytes, void* act_out,
                              float* y_out, float* h_out, int32_t activation, float alpha,
                              float limit, cudaStream_t st) {
  if (T < 0 || K <= 0 || N <= 0 || topk <= 0)
    return fail(MXQ_ERR_INVALID_ARG, "need T >= 0, K > 0, N > 0, topk > 0");
  if (T == 0) return MXQ_OK;
  if (!hidden || !w1 || !w1_scale || !w2 || !w2_scale || !topk_weights || !topk_ids || !out)
    return fail(MXQ_ERR_INVALID_ARG, "NULL tensor argument");
  if (E < 1 || E > 1024) return fail(MXQ_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  if (topk > E) return fail(MXQ_ERR_INVALID_ARG, "topk must be <= E");
  if (activation != MXQ_ACT_SILU && activation != MXQ_ACT_SWIGLU_CLAMP)
    return fail(MXQ_ERR_UNSUPPORTED, "activation must be MXQ_ACT_SILU or MXQ_ACT_SWIGLU_CLAMP");
  if (activation == MXQ_ACT_SWIGLU_CLAMP && !(limit > 0.f && alpha > 0.f && alpha < 3.4e38f))
    return fail(MXQ_ERR_INVALID_ARG, "clamped SwiGLU needs alpha > 0 and limit > 0");
  block_m = resolve_block_m(block_m, T * topk, E);
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128)
    return fail(MXQ_ERR_UNSUPPORTED, "block_m must be 0 (library choice), 16, 32, 64 or 128");
  if (wtype != MXQ_W_FP8_BLOCK128 && wtype != MXQ_W_MXFP4)
    return fail(MXQ_ERR_UNSUPPORTED, "wtype must be MXQ_W_FP8_BLOCK128 or MXQ_W_MXFP4");
  if (ldh < K || ldo < K) return fail(MXQ_ERR_INVALID_ARG, "row strides below K");
  if (wtype == MXQ_W_FP8_BLOCK128 && (K % 16 != 0 || N % 16 != 0))
    return fail(MXQ_ERR_UNSUPPORTED, "FP8 expert weights need K and N multiples of 16");
  if (wtype == MXQ_W_MXFP4 && (K % 32 != 0 || N % 32 != 0))
    return fail(MXQ_ERR_UNSUPPORTED, "MXFP4 expert weights need K and N multiples of 32");
  if (!aligned16(hidden) || (ldh * 2) % 16 != 0 || !aligned16(w1) || !aligned16(w2))
    return fail(MXQ_ERR_UNSUPPORTED,
                "hidden, w1, w2 need 16-byte alignment (and ldh*2 % 16 == 0)");
  if (static_cast<int64_t>(E) * 2 * N >= (1LL << 31) || static_cast<int64_t>(E) * K >= (1LL << 31))
    return fail(MXQ_ERR_UNSUPPORTED, "expert weight row count above 2^31");
  const MoeWs w = moe_ws(T, K, E, N, topk, block_m);
  if (w.S >= (1LL << 30)) return fail(MXQ_ERR_UNSUPPORTED, "too many slots");
  if (!workspace || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(MXQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned and hold " +
                                         std::to_string(w.total) + " bytes");
  DeviceInfo d;
  std::string err;
  if (!device_info(&d, &err)) return fail(MXQ_ERR_UNSUPPORTED, err);
  const int sms = sms_for_grid(d);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(ws + w.sorted);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(ws + w.experts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + w.offsets);
  int32_t* nblocks = reinterpret_cast<int32_t*>(ws + w.nblocks);
  void* xs = ws + w.xs;
  void* ic1 = ws + w.ic1;
  float* y = reinterpret_cast<float*>(ws + w.y);
  const bool fuse_combine = option(MXQ_OPT_FUSE_COMBINE) != 0;
  int* cnt = reinterpret_cast<int*>(ws + w.cnt);
  const int64_t f16_opt = option(MXQ_OPT_MOE_F16);
  // f16 operands: 2 both formats, 1 FP8 only, 3 (default) FP8 always and
  // MXFP4 above 16 routed slots (below, its three extra launches cost more
  // than the cheaper decode saves)
  const bool f16 = f16_opt == 2 || (f16_opt == 1 && wtype == MXQ_W_FP8_BLOCK128) ||
                   (f16_opt == 3 && (wtype == MXQ_W_FP8_BLOCK128 || w.S > 16));
  void* hf16 = ws + w.hf16;
  float* tscale = reinterpret_cast<float*>(ws + w.tscale);
  float* rs1 = reinterpret_cast<float*>(ws + w.rs1);
  void* ic1h = ws + w.ic1h;
  float* rs2 = reinterpret_cast<float*>(ws + w.rs2);
  uint8_t* emax = ws + w.emax;

  cudaError_t e = launch_moe_align(topk_ids, w.S, E, block_m, sorted_ids, expert_ids, offsets,
                                   nblocks, w.cap, d.status, st);
  if (e != cudaSuccess) return cuda_fail(e, "moe_align launch");
  if (f16) {
    e = launch_rows_to_f16(hidden, T, K, ldh, nullptr, hf16, tscale, st);
    if (e != cudaSuccess) return cuda_fail(e, "token conversion launch");
  }
  if (f16 && wtype == MXQ_W_MXFP4) {
    // the f16 decode's per-row reference exponents of both expert matrices
    e = launch_mx_row_emax(w1_scale, 2 * N, K / 32, K / 32, emax, w2_scale, K, N / 32, N / 32,
                           emax + E * 2 * N, expert_ids, nblocks, E, w.cap, st);
    if (e != cudaSuccess) return cuda_fail(e, "MXFP4 row exponent launch");
  }
  e = launch_gather_rows(f16 ? hf16 : hidden, f16 ? K : ldh, K, topk, sorted_ids, offsets, nblocks,
                         block_m, w.cap, xs, fuse_combine ? cnt : nullptr, w.ncnt,
                         f16 ? tscale : nullptr, f16 ? rs1 : nullptr, st);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");

  const bool fp8 = wtype == MXQ_W_FP8_BLOCK128;
  const int kind = fp8 ? (f16 ? KIND_F8H : KIND_F8W) : (f16 ? KIND_MXH : KIND_MXW);
  const int bt = std::max(32, static_cast<int>(block_m));
  const int64_t force = option(MXQ_OPT_FORCE_PATH);
  const int64_t small_m = std::min<int64_t>(option(MXQ_OPT_SMALL_M_MAX), 1 << 30);
  int narrow_max = static_cast<int>(small_m);          // per expert block (the default)
  if (force == 1) narrow_max = 1 << 30;
  if (force == 2) narrow_max = 0;
  if (force == 3) {
    // one path for the whole layer, chosen from the average slots per
    // expert, max(1, S / E) (the global crossover the per-block choice is
    // measured against)
    const int64_t avg_m = std::max<int64_t>(1, w.S / E);
    narrow_max = avg_m <= small_m ? (1 << 30) : 0;
  }

  for (int stage = 0; stage < 2; ++stage) {
    // stage 0: act = silu-mul(xs . W1^T);  stage 1: y = w * (act . W2^T + b2)
    const int64_t rows = stage == 0 ? 2 * N : K;   // rows of one expert matrix
    const int64_t red = stage == 0 ? K : N;        // reduction length
    const void* wt = stage == 0 ? w1 : w2;
    const void* wsc = stage == 0 ? w1_scale : w2_scale;
    if (stage == 1 && f16) {
      // stage-2 tokens: the act rows (bf16) as f16 with their row scales
      e = launch_rows_to_f16(ic1, w.S, N, N, nullptr, ic1h, rs2, st);
      if (e != cudaSuccess) return cuda_fail(e, "act conversion launch");
    }
    const void* src = stage == 0 ? xs : (f16 ? ic1h : ic1);
    GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const uint32_t arows = stage == 0 ? 64 : 128;
    if (fp8) {
      if (!make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt, red, E * rows, red, 128, arows,
                       CU_TENSOR_MAP_SWIZZLE_128B, &err))
        return fail(MXQ_ERR_CUDA, err);
    } else {
      // boxes of 128-byte rows (two K slices of e2m1) with the 128-byte
      // swizzle: the decode threads (one per weight row) read 16-byte chunks
      // without bank conflicts
      if (!make_map_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt, red / 2, E * rows, red / 2, 128,
                       arows, CU_TENSOR_MAP_SWIZZLE_128B, &err))
        return fail(MXQ_ERR_CUDA, err);
    }
    // token boxes of 16 / 32 / 64 / 128 rows, and (b[4]) 8 rows for expert
    // blocks of at most 8 slots
    for (int v = 0; v < 5; ++v) {
      const uint32_t br = v == 4 ? 8u : 16u << v;
      if (v < 4 && static_cast<int>(br) > bt) continue;
      if (!make_map_2d(&maps.b[v],
                       f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src,
                       red, w.S, red * 2, 64, br, CU_TENSOR_MAP_SWIZZLE_128B, &err))
        return fail(MXQ_ERR_CUDA, err);
    }
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int>(w.S);
    p.N = static_cast<int>(rows);
    p.K = static_cast<int>(red);
    p.nkb = static_cast<int>(cdiv(red, 128));
    p.tiles_n = static_cast<int>(stage == 0 ? cdiv(N, 64) : cdiv(K, 128));
    p.tiles_m = 1;
    p.splits = 1;
    p.kb_per_split = p.nkb;
    p.grouped = 1;
    p.num_blocks = nblocks;
    p.expert_ids = expert_ids;
    p.offsets = offsets;
    p.sorted_ids = sorted_ids;
    p.block_m = block_m;
    p.narrow_max = narrow_max;
    p.n_half = static_cast<int>(N);
    p.act = activation == MXQ_ACT_SWIGLU_CLAMP ? 1 : 0;
    p.act_alpha = alpha;
    p.act_limit = limit;
    if (fp8) {
      p.w_scale = reinterpret_cast<const float*>(wsc);
      p.sw0 = cdiv(red, 128);
      p.sw1 = 1;
      p.sw_e = cdiv(rows, 128) * cdiv(red, 128);
      p.block_n = 128;
    } else {
      p.mx_scale = reinterpret_cast<const uint8_t*>(wsc);
      p.mx_ld = red / 32;
      p.mx_cols = static_cast<int>(red / 32);
      p.mx_rows_total = static_cast<int64_t>(E) * rows;
      {
        const uintptr_t sb = reinterpret_cast<uintptr_t>(wsc);
        p.mx_align = ((p.mx_ld % 4) == 0 && (sb % 4) == 0) ? 4 : (((p.mx_ld % 2) == 0 && (sb % 2) == 0) ? 2 : 1);
      }
      p.block_n = 0;
    }
    if (f16) {
      // column scales: the inverse power of two of each compact token row
      p.a_scale = stage == 0 ? rs1 : rs2;
      p.sa0 = 1;
      p.sa1 = 0;
    }
    if (kind == KIND_MXH) p.mx_emax = emax + (stage == 0 ? 0 : E * 2 * N);
    p.bias = stage == 0 ? w1_bias : w2_bias;
    p.bias_dtype = MXQ_F32;
    p.bias_e = rows;
    p.route_w = topk_weights;
    p.h_out = stage == 0 ? h_out : nullptr;
    if (stage == 1 && fuse_combine) {
      p.combine_cnt = cnt;
      p.combine_out = out;
      p.combine_ldo = ldo;
      p.topk = topk;
    }
    p.out = stage == 0 ? ic1 : static_cast<void*>(y);
    p.out_dtype = stage == 0 ? MXQ_BF16 : MXQ_F32;
    p.ldo = stage == 0 ? N : K;
    // scatter: 16-byte y rows (the workspace is 256-byte aligned)
    p.vec_ok = stage == 1 && K % 4 == 0;
    p.status = d.status;
    p.budget_ns = static_cast<unsigned long long>(option(MXQ_OPT_WAIT_BUDGET_NS));
    p.inject_stall = static_cast<int>(option(MXQ_OPT_INJECT_STALL));
    const int64_t units = w.cap * p.tiles_n;
    const int grid = static_cast<int>(std::min<int64_t>(units, sms));
    e = launch_gemm(kind, stage == 0 ? EPI_SILU : EPI_SCATTER, bt, fp8, maps, p, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, stage == 0 ? "stage-1 launch" : "stage-2 launch");
  }
  if (!fuse_combine) {
    e = launch_combine(y, T, topk, K, out, ldo, st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  if (act_out) {
    e = launch_unsort_rows(ic1, N, sorted_ids, offsets, nblocks, block_m, w.cap, act_out, st);
    if (e != cudaSuccess) return cuda_fail(e, "unsort launch");
  }
  if (y_out) {
    e = cudaMemcpyAsync(y_out, y, static_cast<size_t>(w.S) * K * 4, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "y copy");
  }
  return MXQ_OK;
}

}  // namespace

extern "C" mxq_status mxq_fused_experts_workspace_size(int64_t T, int64_t K, int32_t E, int64_t N,
                                                       int32_t topk, int32_t block_m,
                                                       int32_t wtype, size_t* bytes) {
  (void)wtype;
  if (!bytes || T < 0 || K <= 0 || N <= 0 || topk <= 0 || E < 1 || block_m < 0)
    return fail(MXQ_ERR_INVALID_ARG, "bad sizes or NULL result pointer");
  *bytes = moe_ws(T, K, E, N, topk, resolve_block_m(block_m, T * topk, E)).total;
  return MXQ_OK;
}

extern "C" mxq_status mxq_fused_experts(const void* hidden, int64_t T, int64_t K, int64_t ldh,
                                        int32_t wtype, int32_t E, int64_t N, const void* w1,
                                        const void* w1_scale, const float* w1_bias, const void* w2,
                                        const void* w2_scale, const float* w2_bias,
                                        const float* topk_weights, const int32_t* topk_ids,
                                        int32_t topk, int32_t block_m, void* out, int64_t ldo,
                                        void* workspace, size_t ws_bytes, mxq_stream_t stream) {
  return fused_experts_impl(hidden, T, K, ldh, wtype, E, N, w1, w1_scale, w1_bias, w2, w2_scale,
                            w2_bias, topk_weights, topk_ids, topk, block_m, out, ldo, workspace,
                            ws_bytes, nullptr, nullptr, nullptr, MXQ_ACT_SILU, 0.f, 0.f,
                            reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxq_status mxq_fused_experts_debug(
    const void* hidden, int64_t T, int64_t K, int64_t ldh, int32_t wtype, int32_t E, int64_t N,
    const void* w1, const void* w1_scale, const float* w1_bias, const void* w2,
    const void* w2_scale, const float* w2_bias, const float* topk_weights, const int32_t* topk_ids,
    int32_t topk, int32_t block_m, void* out, int64_t ldo, void* workspace, size_t ws_bytes,
    void* act_out, float* y_out, float* h_out, mxq_stream_t stream) {
  return fused_experts_impl(hidden, T, K, ldh, wtype, E, N, w1, w1_scale, w1_bias, w2, w2_scale,
                            w2_bias, topk_weights, topk_ids, topk, block_m, out, ldo, workspace,
                            ws_bytes, act_out, y_out, h_out, MXQ_ACT_SILU, 0.f, 0.f,
                            reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxq_status mxq_fused_experts_ex(
    const void* hidden, int64_t T, int64_t K, int64_t ldh, int32_t wtype, int32_t E, int64_t N,
    const void* w1, const void* w1_scale, const float* w1_bias, const void* w2,
    const void* w2_scale, const float* w2_bias, const float* topk_weights, const int32_t* topk_ids,
    int32_t topk, int32_t block_m, int32_t activation, float alpha, float limit, void* out,
    int64_t ldo, void* workspace, size_t ws_bytes, void* act_out, float* y_out, float* h_out,
    mxq_stream_t stream) {
  return fused_experts_impl(hidden, T, K, ldh, wtype, E, N, w1, w1_scale, w1_bias, w2, w2_scale,
                            w2_bias, topk_weights, topk_ids, topk, block_m, out, ldo, workspace,
                            ws_bytes, act_out, y_out, h_out, activation, alpha, limit,
                            reinterpret_cast<cudaStream_t>(stream));
}
