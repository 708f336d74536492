// quant.cu — per-token-group FP8 quantization of bf16 activations.
//
// "[XPU] block-FP8 linear via torch scaled_mm", key code excerpts: when no
// input scale is given, the activation is quantized per 1 x block_k group
// (per_token_group_quant_fp8) into e4m3 with one fp32 scale per group,
// shape [M, K/128].  For each group: s = max(amax, eps) / 448, and every
// element is q = e4m3(clamp(x / s, -448, 448)), round to nearest even, with
// IEEE fp32 division (no reciprocal) so the codes are reproducible.
//
// Memory-bound: 2 bytes in, 1 + 4/128 bytes out per element.  The fast path
// gives each 128-element group to a half warp (8 contiguous bf16 = one 16-byte
// load per lane), reduces amax with shuffles, and writes 8 codes per lane;
// each half warp handles four groups at a time to keep loads in flight.
#include <cuda_bf16.h>

#include "internal.h"

namespace mxq {


// group == 128, K % 128 == 0, 16-byte aligned rows.  A warp takes 8 groups
// per iteration (each half warp 4): all 4 loads of a lane are issued before
// any of them is used, so 64 bytes per lane are in flight.
__global__ void group_quant128_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K,
                                      int64_t ldx, float eps, uint8_t* __restrict__ q,
                                      float* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int U = 4;
  // the launcher uses this kernel only while M * K/128 < 2^31, so the group
  // index fits 32 bits: one 32-bit division per iteration locates the row
  // of the warp's first group, and the others follow by steps (64-bit
  // division is a long instruction sequence on the GPU)
  const uint32_t G = static_cast<uint32_t>(K / 128);
  const uint32_t total = static_cast<uint32_t>(M) * G;
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;
  const int hw = lane >> 4;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; 2 * U * w < total;
       w += nwarps) {
    uint4 raw[U];
    int64_t mm[U], gg[U];
    bool ok[U];
    const uint32_t base = 2 * U * w;
    const uint32_t m0 = base / G;
    const uint32_t r0 = base - m0 * G;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t item = base + 2 * u + hw;
      ok[u] = item < total;
      uint32_t m = m0, r = r0 + 2 * u + hw;
      while (r >= G) {   // at most once when G >= 8
        r -= G;
        ++m;
      }
      mm[u] = ok[u] ? m : 0;
      gg[u] = ok[u] ? r : 0;
      raw[u] = ok[u] ? __ldg(reinterpret_cast<const uint4*>(x + mm[u] * ldx + gg[u] * 128 + hl * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float v[8];
      const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(wv[i] << 16);
        v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = fabsf(v[i]);
        amax = (a > amax) ? a : amax;
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, amax, off);
        amax = (o > amax) ? o : amax;
      }
      if (ok[u]) {
        const float s = __fdiv_rn((amax > eps) ? amax : eps, 448.f);
        uint32_t pk[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float* vv = v + 4 * h;
          const uint16_t a =
              e4m3x2_rn(clamp448(__fdiv_rn(vv[0], s)), clamp448(__fdiv_rn(vv[1], s)));
          const uint16_t b =
              e4m3x2_rn(clamp448(__fdiv_rn(vv[2], s)), clamp448(__fdiv_rn(vv[3], s)));
          pk[h] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
        }
        *reinterpret_cast<uint2*>(q + mm[u] * K + gg[u] * 128 + hl * 8) = make_uint2(pk[0], pk[1]);
        if (hl == 0) scales[mm[u] * G + gg[u]] = s;
      }
    }
  }
}

// any group (multiple of 8, <= 1024), ragged K, any row stride: one warp per group
__global__ void group_quant_generic_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                           int64_t K, int64_t ldx, int group, float eps,
                                           uint8_t* __restrict__ q, float* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t G = (K + group - 1) / group;
  const int64_t total = M * G;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total;
       w += nwarps) {
    const int64_t m = w / G, g = w - (w / G) * G;
    const int64_t k0 = g * group;
    const int64_t k1 = (k0 + group < K) ? k0 + group : K;
    float amax = 0.f;
    for (int64_t k = k0 + lane; k < k1; k += 32) {
      const float a = fabsf(__bfloat162float(x[m * ldx + k]));
      amax = (a > amax) ? a : amax;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, amax, off);
      amax = (o > amax) ? o : amax;
    }
    const float s = __fdiv_rn((amax > eps) ? amax : eps, 448.f);
    for (int64_t k = k0 + lane; k < k1; k += 32) {
      const float t = clamp448(__fdiv_rn(__bfloat162float(x[m * ldx + k]), s));
      q[m * K + k] = static_cast<uint8_t>(e4m3x2_rn(t, 0.f) & 0xFF);
    }
    if (lane == 0) scales[m * G + g] = s;
  }
}

cudaError_t launch_group_quant(const void* x, int64_t M, int64_t K, int64_t ldx, int group,
                               float eps, void* q, float* scales, int num_sms,
                               cudaStream_t stream) {
  const bool fast = group == 128 && K % 128 == 0 && ldx % 8 == 0 &&
                    M * (K / 128) < (int64_t(1) << 31) &&
                    (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(q) & 7) == 0;
  const int threads = 256;
  const int64_t G = (K + group - 1) / group;
  const int64_t items = fast ? (M * G + 7) / 8 : M * G;       // warps of work
  int64_t blocks = (items + (threads / 32) - 1) / (threads / 32);
  // a persistent grid of the blocks that fit at once (no ragged last wave)
  static int resident[2] = {0, 0};
  int& res = resident[fast ? 1 : 0];
  if (res == 0) {
    int r = 0;
    cudaError_t e = fast ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, group_quant128_kernel,
                                                                       threads, 0)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                               &r, group_quant_generic_kernel, threads, 0);
    if (e != cudaSuccess) return e;
    res = r > 0 ? r : 1;
  }
  const int64_t cap = static_cast<int64_t>(num_sms) * res;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (fast)
    return launch_k(group_quant128_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                    stream, reinterpret_cast<const __nv_bfloat16*>(x), M, K, ldx, eps,
                    reinterpret_cast<uint8_t*>(q), scales);
  return launch_k(group_quant_generic_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                  stream, reinterpret_cast<const __nv_bfloat16*>(x), M, K, ldx, group, eps,
                  reinterpret_cast<uint8_t*>(q), scales);
}

}  // namespace mxq

// ------------------------------------------------------------ MXFP4 encode
// Weight quantization to MXFP4 by the OCP Microscaling (MX) v1.0 rule, the
// format of the MXFP4 expert weights ("[CPU] routed FP8/MXFP4 MoE", related
// PR 49347: online MXFP4 quantization).  Per block of 32 consecutive values:
// shared exponent E = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 for
// an all-zero block), ue8m0 byte E + 127, elements = E2M1 round-to-nearest-
// even of v * 2^-E with saturation at 6 (the conversion instruction's rule),
// sign kept.  One thread per block: 64 (bf16) or 128 (fp32) contiguous bytes
// in, 16 bytes of codes and one scale byte out.
namespace mxq {

__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool BF16IN>
__global__ void mxfp4_quant_kernel(const void* __restrict__ x, int64_t R, int64_t C, int64_t ldx,
                                   uint8_t* __restrict__ packed, uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t G = C / 32;
  const int64_t total = R * G;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / G, g = i - r * G;
    float v[32];
    if (BF16IN) {
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(x) + r * ldx + g * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = __ldg(src + j);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          v[8 * j + 2 * t] = __uint_as_float(wv[t] << 16);
          v[8 * j + 2 * t + 1] = __uint_as_float(wv[t] & 0xFFFF0000u);
        }
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) +
                                                          r * ldx + g * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 w = __ldg(src + j);
        v[4 * j] = w.x;
        v[4 * j + 1] = w.y;
        v[4 * j + 2] = w.z;
        v[4 * j + 3] = w.w;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
    int E = -127;
    if (amax > 0.f) E = max(-127, min(127, ilogbf(amax) - 2));
    const float inv = ldexpf(1.0f, -E);   // 2^-E: exact (2^127 down to 2^-127)
    uint32_t words[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
        w |= e2m1x2_rn(v[8 * j + 2 * t] * inv, v[8 * j + 2 * t + 1] * inv) << (8 * t);
      words[j] = w;
    }
    *reinterpret_cast<uint4*>(packed + r * (C / 2) + g * 16) =
        make_uint4(words[0], words[1], words[2], words[3]);
    scales[r * G + g] = static_cast<uint8_t>(E + 127);
  }
}

cudaError_t launch_mxfp4_quant(const void* x, bool bf16, int64_t R, int64_t C, int64_t ldx,
                               void* packed, void* scales, int num_sms, cudaStream_t stream) {
  const int64_t total = R * (C / 32);
  int64_t blocks = (total + 127) / 128;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (bf16)
    return launch_k(mxfp4_quant_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(128), 0,
                    stream, x, R, C, ldx, reinterpret_cast<uint8_t*>(packed),
                    reinterpret_cast<uint8_t*>(scales));
  return launch_k(mxfp4_quant_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(128), 0,
                  stream, x, R, C, ldx, reinterpret_cast<uint8_t*>(packed),
                  reinterpret_cast<uint8_t*>(scales));
}

}  // namespace mxq
