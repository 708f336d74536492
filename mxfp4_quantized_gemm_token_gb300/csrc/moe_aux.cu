// moe_aux.cu — the non-GEMM steps of the routed MoE path: expert-block
// alignment, the token-row gather that feeds stage 1, the top-k combine, and
// the small helpers (split-K reduction of fp8_scaled_mm, debug unsort).
#include <cuda_bf16.h>
#include <algorithm>
#include <cuda_fp16.h>

#include "internal.h"

namespace mxq {

// ------------------------------------------------------------ moe_align
// "[CPU] routed FP8/MXFP4 MoE" consumes, per expert block mb: expert_ids[mb],
// the block's token slots sorted_ids[mb*block_m + m] and the compact row
// offsets[mb]; this kernel produces them.  One CTA of 1024 threads:
//   1. histogram of slots per expert (shared-memory atomics);
//   2. exclusive scans of the per-expert block and slot counts: warp
//      shuffles, then a scan of the 32 warp totals, 1024 experts per pass;
//   3. the block table (expert_ids, offsets);
//   4. a stable ranking of the slots, 1024 at a time in slot order: inside a
//      warp, lanes with the same expert find each other with match.any and
//      rank by lane; per-warp counts in shared memory are turned into
//      per-warp starting positions by one pass per expert over the 32 warps,
//      which also carries the running count per expert to the next chunk.
// The result is unique (stable order), so it is compared bit for bit.
__global__ void __launch_bounds__(1024) moe_align_kernel(const int32_t* __restrict__ ids, int S,
                                                         int E, int BM, int cap,
                                                         int32_t* __restrict__ sorted_ids,
                                                         int32_t* __restrict__ expert_ids,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ num_blocks,
                                                         int* status) {
  extern __shared__ int sm[];
  int* cnt = sm;
  int* blk_start = cnt + E;
  int* pos_start = blk_start + E;
  int* run = pos_start + E;
  int* wcnt = run + E;   // [32][E]
  __shared__ int wsum_b[32], wsum_p[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_launch_dependents();

  for (int i = tid; i < E; i += 1024) {
    cnt[i] = 0;
    run[i] = 0;
  }
  for (int i = tid; i < 32 * E; i += 1024) wcnt[i] = 0;
  for (int64_t i = tid; i < static_cast<int64_t>(cap) * BM; i += 1024) sorted_ids[i] = S;
  for (int i = tid; i < cap; i += 1024) expert_ids[i] = -1;
  for (int i = tid; i <= cap; i += 1024) offsets[i] = S;
  __syncthreads();

  bool bad = false;
  for (int s = tid; s < S; s += 1024) {
    const int e = __ldg(ids + s);
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(status, kStatusBadIndex);
  __syncthreads();

  // exclusive scans: first block and first compact row of each expert
  int carry_b = 0, carry_p = 0;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + tid;
    const int c = (e < E) ? cnt[e] : 0;
    const int ob = (c + BM - 1) / BM, op = c;
    int vb = ob, vp = op;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int tb = __shfl_up_sync(0xffffffffu, vb, d);
      const int tp = __shfl_up_sync(0xffffffffu, vp, d);
      if (lane >= d) {
        vb += tb;
        vp += tp;
      }
    }
    if (lane == 31) {
      wsum_b[warp] = vb;
      wsum_p[warp] = vp;
    }
    __syncthreads();
    if (warp == 0) {
      const int xb = wsum_b[lane], xp = wsum_p[lane];
      int ib = xb, ip = xp;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int tb = __shfl_up_sync(0xffffffffu, ib, d);
        const int tp = __shfl_up_sync(0xffffffffu, ip, d);
        if (lane >= d) {
          ib += tb;
          ip += tp;
        }
      }
      wsum_b[lane] = ib - xb;   // exclusive over warps
      wsum_p[lane] = ip - xp;
    }
    __syncthreads();
    if (e < E) {
      blk_start[e] = carry_b + wsum_b[warp] + vb - ob;
      pos_start[e] = carry_p + wsum_p[warp] + vp - op;
    }
    // this pass's totals: the last expert's inclusive values
    const int tot_b = __shfl_sync(0xffffffffu, vb, 31) + wsum_b[warp];
    const int tot_p = __shfl_sync(0xffffffffu, vp, 31) + wsum_p[warp];
    __syncthreads();
    if (tid == 1023) {
      wsum_b[0] = tot_b;
      wsum_p[0] = tot_p;
    }
    __syncthreads();
    carry_b += wsum_b[0];
    carry_p += wsum_p[0];
    __syncthreads();
  }
  if (tid == 0) {
    *num_blocks = carry_b;
    offsets[carry_b] = carry_p;
  }
  for (int e = tid; e < E; e += 1024) {
    const int nb = (cnt[e] + BM - 1) / BM;
    for (int j = 0; j < nb; ++j) {
      expert_ids[blk_start[e] + j] = e;
      offsets[blk_start[e] + j] = pos_start[e] + j * BM;
    }
  }

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < S; base += 1024) {
    const int s = base + tid;
    int e = (s < S) ? __ldg(ids + s) : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    const bool leader = (__ffs(peers) - 1) == lane;
    if (valid && leader) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    // per expert: counts of the 32 warps -> each warp's first position
    for (int ee = tid; ee < E; ee += 1024) {
      int acc = run[ee];
#pragma unroll 8
      for (int w = 0; w < 32; ++w) {
        const int t = wcnt[w * E + ee];
        wcnt[w * E + ee] = acc;
        acc += t;
      }
      run[ee] = acc;
    }
    __syncthreads();
    if (valid)
      sorted_ids[static_cast<int64_t>(blk_start[e]) * BM + wcnt[warp * E + e] + rank] = s;
    __syncthreads();
    if (base + 1024 < S) {
      for (int i = tid; i < 32 * E; i += 1024) wcnt[i] = 0;
      __syncthreads();
    }
  }
}

cudaError_t launch_moe_align(const int32_t* topk_ids, int64_t S, int32_t E, int32_t block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* offsets,
                             int32_t* num_blocks, int64_t cap, int* status, cudaStream_t stream) {
  const int smem = static_cast<int>((4 + 32) * E * sizeof(int));
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(moe_align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return launch_k(moe_align_kernel, dim3(1), dim3(1024), static_cast<size_t>(smem), stream,
                  topk_ids, static_cast<int>(S), E, block_m, static_cast<int>(cap), sorted_ids,
                  expert_ids, offsets, num_blocks, status);
}

// --------------------------------------------------------- rows to f16
// The f16 MMA operand of the fused MoE: each bf16 row x (K values) becomes
// x * 2^p in f16 with p = 14 - floor(log2(max |x|)) (the row maximum lands in
// [2^14, 2^15), below the f16 maximum), and rscale = 2^-p undoes it in the
// epilogue.  Power-of-two scaling is exact, and so is the f16 value of every
// element not more than ~2^31 below its row maximum (bf16's 8 significant
// bits then stay inside f16's range); an all-zero row keeps p = 0.  One warp
// per row; `rows` may be read on the device (count != NULL).
__global__ void rows_to_f16_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int64_t K,
                                   int64_t ld, const int32_t* __restrict__ count,
                                   __half* __restrict__ dst, float* __restrict__ rscale, int vec) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t nrows = count != nullptr ? static_cast<int64_t>(__ldg(count)) : rows;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < nrows;
       r += nwarps) {
    const __nv_bfloat16* s = src + r * ld;
    float m = 0.f;
    if (vec) {
      for (int64_t k = lane * 8; k < K; k += 256) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(s + k));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          m = fmaxf(m, fabsf(__uint_as_float(wv[i] << 16)));
          m = fmaxf(m, fabsf(__uint_as_float(wv[i] & 0xFFFF0000u)));
        }
      }
    } else {
      for (int64_t k = lane; k < K; k += 32) m = fmaxf(m, fabsf(__bfloat162float(s[k])));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    int pw = 0;
    if (m > 0.f) pw = max(-126, min(126, 14 - ilogbf(m)));
    const float up = ldexpf(1.0f, pw);
    if (lane == 0) rscale[r] = ldexpf(1.0f, -pw);
    __half* d = dst + r * K;
    if (vec) {
      for (int64_t k = lane * 8; k < K; k += 256) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(s + k));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __half2 h = __floats2half2_rn(__uint_as_float(wv[i] << 16) * up,
                                        __uint_as_float(wv[i] & 0xFFFF0000u) * up);
          o[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(d + k) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    } else {
      for (int64_t k = lane; k < K; k += 32) d[k] = __float2half_rn(__bfloat162float(s[k]) * up);
    }
  }
}

cudaError_t launch_rows_to_f16(const void* src, int64_t rows, int64_t K, int64_t ld,
                               const int32_t* count, void* dst, float* rscale,
                               cudaStream_t stream) {
  const int vec = (K % 8 == 0) && (ld % 8 == 0) && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  return launch_k(rows_to_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                  reinterpret_cast<const __nv_bfloat16*>(src), rows, K, ld, count,
                  reinterpret_cast<__half*>(dst), rscale, vec);
}

// ------------------------------------------------ MXFP4 row exponents
// The f16 decode of MXFP4 expert weights scales every 32-group relative to
// the largest ue8m0 exponent of its weight row: emax[e * rows + r] = max over
// k of scales[(e * rows + r) * ld + k], for both expert matrices in one
// launch.  Only the experts of the block table are visited (a block whose
// expert repeats the previous block's is skipped).  CTA (block b, chunk c):
// chunks [0, ch1) cover the rows of matrix 1 and [ch1, ch1 + ch2) those of
// matrix 2, 256 rows each; one thread per row reads the row with the widest
// loads its alignment allows (align: 4, 2 or 1 bytes for both matrices).
namespace {

__device__ __forceinline__ unsigned row_max_u8(const uint8_t* row, int ncols, int align) {
  unsigned m = 0;
  int c = 0;
  if (align >= 4) {
    for (; c + 4 <= ncols; c += 4) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(row + c));
      m = max(m, max(max(v & 0xFFu, (v >> 8) & 0xFFu), max((v >> 16) & 0xFFu, v >> 24)));
    }
  } else if (align >= 2) {
    for (; c + 2 <= ncols; c += 2) {
      const uint32_t v = __ldg(reinterpret_cast<const uint16_t*>(row + c));
      m = max(m, max(v & 0xFFu, v >> 8));
    }
  }
  for (; c < ncols; ++c) m = max(m, static_cast<unsigned>(__ldg(row + c)));
  return m;
}

// rows of at most EMAX_STAGE_COLS bytes, stored back to back (ld == ncols)
// and 16-byte aligned per chunk: a chunk of 256 rows is one contiguous range,
// read with coalesced 16-byte loads into shared memory, and each thread then
// takes its row's maximum there (a thread reading its own row from global
// memory touches a separate line per lane)
constexpr int EMAX_STAGE_COLS = 160;

__global__ void __launch_bounds__(256) mx_row_emax_kernel(
    const uint8_t* __restrict__ s1, int64_t rows1, int ncols1, int64_t ld1, uint8_t* __restrict__ e1,
    const uint8_t* __restrict__ s2, int64_t rows2, int ncols2, int64_t ld2, uint8_t* __restrict__ e2,
    int align, int staged, const int32_t* __restrict__ expert_ids,
    const int32_t* __restrict__ num_blocks, int E, int64_t ch1, int64_t ch2) {
  __shared__ __align__(16) uint8_t sbuf[256 * EMAX_STAGE_COLS];
  pdl_wait();
  pdl_launch_dependents();
  // every exit below depends on the block index only, so the whole CTA
  // leaves together and the barriers of the staged path are uniform
  const int b = blockIdx.x;
  if (b >= __ldg(num_blocks)) return;
  const int e = __ldg(expert_ids + b);
  if (e < 0 || e >= E || (b > 0 && __ldg(expert_ids + b - 1) == e)) return;
  for (int64_t c = blockIdx.y; c < ch1 + ch2; c += gridDim.y) {
    const bool second = c >= ch1;
    const int64_t rows = second ? rows2 : rows1;
    const int64_t r0 = (second ? c - ch1 : c) * 256;
    const uint8_t* base = second ? s2 : s1;
    const int64_t ld = second ? ld2 : ld1;
    const int ncols = second ? ncols2 : ncols1;
    uint8_t* out = (second ? e2 : e1) + static_cast<int64_t>(e) * rows + r0;
    if (staged) {
      const int nr = static_cast<int>(rows - r0 < 256 ? rows - r0 : 256);
      const int nbytes = nr * ncols;
      const uint8_t* src = base + (static_cast<int64_t>(e) * rows + r0) * ld;
      __syncthreads();   // the previous chunk's rows have been read
      for (int i = threadIdx.x; i < nbytes / 16; i += 256)
        reinterpret_cast<uint4*>(sbuf)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
      for (int i = (nbytes / 16) * 16 + threadIdx.x; i < nbytes; i += 256) sbuf[i] = __ldg(src + i);
      __syncthreads();
      if (static_cast<int>(threadIdx.x) < nr) {
        const uint8_t* row = sbuf + threadIdx.x * ncols;
        unsigned m = 0;
#pragma unroll 8
        for (int j = 0; j < ncols; ++j) m = max(m, static_cast<unsigned>(row[j]));
        out[threadIdx.x] = static_cast<uint8_t>(m);
      }
    } else {
      const int64_t r = r0 + threadIdx.x;
      if (r >= rows) continue;
      out[threadIdx.x] = static_cast<uint8_t>(
          row_max_u8(base + (static_cast<int64_t>(e) * rows + r) * ld, ncols, align));
    }
  }
}

}  // namespace

cudaError_t launch_mx_row_emax(const void* s1, int64_t rows1, int64_t ncols1, int64_t ld1, void* e1,
                               const void* s2, int64_t rows2, int64_t ncols2, int64_t ld2, void* e2,
                               const int32_t* expert_ids, const int32_t* num_blocks, int E,
                               int64_t cap, cudaStream_t stream) {
  if (cap <= 0) return cudaSuccess;
  const uintptr_t a = reinterpret_cast<uintptr_t>(s1) | reinterpret_cast<uintptr_t>(s2) |
                      static_cast<uintptr_t>(ld1) | static_cast<uintptr_t>(ld2);
  const int align = (a & 3) == 0 ? 4 : ((a & 1) == 0 ? 2 : 1);
  // staged: rows back to back, short enough for the shared buffer, and every
  // chunk of 256 rows of every expert starting on a 16-byte boundary
  const int staged = ld1 == ncols1 && ld2 == ncols2 && ncols1 <= EMAX_STAGE_COLS &&
                     ncols2 <= EMAX_STAGE_COLS &&
                     ((reinterpret_cast<uintptr_t>(s1) | reinterpret_cast<uintptr_t>(s2)) & 15) == 0 &&
                     (rows1 * ld1) % 16 == 0 && (rows2 * ld2) % 16 == 0;
  const int64_t ch1 = (rows1 + 255) / 256, ch2 = (rows2 + 255) / 256;
  const unsigned gy = static_cast<unsigned>(std::min<int64_t>(ch1 + ch2, 65535));
  return launch_k(mx_row_emax_kernel, dim3(static_cast<unsigned>(cap), gy), dim3(256), 0, stream,
                  reinterpret_cast<const uint8_t*>(s1), rows1, static_cast<int>(ncols1), ld1,
                  reinterpret_cast<uint8_t*>(e1), reinterpret_cast<const uint8_t*>(s2), rows2,
                  static_cast<int>(ncols2), ld2, reinterpret_cast<uint8_t*>(e2), align, staged,
                  expert_ids, num_blocks, E, ch1, ch2);
}

// ------------------------------------------------------------ row gather
// Stage-1 operand: compact row r = offsets[b] + m holds hidden[slot / topk],
// slot = sorted_ids[b*block_m + m] (the page copies the same rows per block
// before its first N tile).  One warp per (block, row) position.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ hidden, int64_t ldh, int64_t K,
                                   int topk, const int32_t* __restrict__ sorted_ids,
                                   const int32_t* __restrict__ offsets,
                                   const int32_t* __restrict__ num_blocks, int BM,
                                   __nv_bfloat16* __restrict__ xs, int vec, int* __restrict__ zero,
                                   int64_t nzero, const float* __restrict__ tscale,
                                   float* __restrict__ rscale) {
  pdl_wait();
  pdl_launch_dependents();
  // also clears the fused combine's counters for this call
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nzero;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    zero[i] = 0;
  const int nb = __ldg(num_blocks);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = static_cast<int64_t>(nb) * BM;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total;
       w += nwarps) {
    const int b = static_cast<int>(w / BM), m = static_cast<int>(w % BM);
    const int r0 = __ldg(offsets + b);
    if (m >= __ldg(offsets + b + 1) - r0) continue;
    const int slot = __ldg(sorted_ids + w);
    const __nv_bfloat16* src = hidden + static_cast<int64_t>(slot / topk) * ldh;
    __nv_bfloat16* dst = xs + static_cast<int64_t>(r0 + m) * K;
    if (rscale != nullptr && lane == 0) rscale[r0 + m] = __ldg(tscale + slot / topk);
    if (vec) {
      for (int64_t k = lane * 8; k < K; k += 256)
        *reinterpret_cast<uint4*>(dst + k) = __ldg(reinterpret_cast<const uint4*>(src + k));
    } else {
      for (int64_t k = lane; k < K; k += 32) dst[k] = src[k];
    }
  }
}

cudaError_t launch_gather_rows(const void* hidden, int64_t ldh, int64_t K, int32_t topk,
                               const int32_t* sorted_ids, const int32_t* offsets,
                               const int32_t* num_blocks, int32_t block_m, int64_t cap, void* xs,
                               int* zero, int64_t nzero, const float* tscale, float* rscale,
                               cudaStream_t stream) {
  const int vec = (K % 8 == 0) && (ldh % 8 == 0) &&
                  (reinterpret_cast<uintptr_t>(hidden) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(xs) & 15) == 0;
  const int64_t warps = cap * block_m;
  int64_t blocks = (warps + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  return launch_k(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                  reinterpret_cast<const __nv_bfloat16*>(hidden), ldh, K, topk, sorted_ids,
                  offsets, num_blocks, block_m, reinterpret_cast<__nv_bfloat16*>(xs), vec, zero,
                  zero != nullptr ? nzero : 0, tscale, rscale);
}

// ------------------------------------------------------------ combine
// out[t] = bf16( sum_{k=0..topk-1} y[t*topk + k] ), ascending k, fp32 sum;
// y already carries the routing weight.
__global__ void combine_kernel(const float* __restrict__ y, int64_t T, int topk, int64_t K,
                               __nv_bfloat16* __restrict__ out, int64_t ldo, int vec) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (vec) {
    const int64_t K4 = K / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < T * K4;
         i += stride) {
      const int64_t t = i / K4, k = (i - t * K4) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < topk; ++j) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(y + (t * topk + j) * K + k));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + t * ldo + k) = pk;
    }
  } else {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < T * K;
         i += stride) {
      const int64_t t = i / K, k = i - t * K;
      float acc = 0.f;
      for (int j = 0; j < topk; ++j) acc += y[(t * topk + j) * K + k];
      out[t * ldo + k] = __float2bfloat16_rn(acc);
    }
  }
}

cudaError_t launch_combine(const float* y, int64_t T, int32_t topk, int64_t K, void* out,
                           int64_t ldo, cudaStream_t stream) {
  const int vec = (K % 4 == 0) && (ldo % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 7) == 0 &&
                  (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  const int64_t n = vec ? T * (K / 4) : T * K;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  if (blocks < 1) blocks = 1;
  return launch_k(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, y, T,
                  topk, K, reinterpret_cast<__nv_bfloat16*>(out), ldo, vec);
}

// ------------------------------------------------------ split-K reduction
// out[m, n] = round( sum_s partial[s, m, n] + bias[n] ), ascending s.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int64_t M,
                                     int64_t N, const void* bias, int bias_dtype, void* out,
                                     int out_dtype, int64_t ldo) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M * N;
       i += stride) {
    const int64_t m = i / N, n = i - m * N;
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[s * M * N + i];
    if (bias != nullptr)
      acc += (bias_dtype == DT_BF16)
                 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(bias)[n])
                 : reinterpret_cast<const float*>(bias)[n];
    if (out_dtype == DT_BF16)
      reinterpret_cast<__nv_bfloat16*>(out)[m * ldo + n] = __float2bfloat16_rn(acc);
    else
      reinterpret_cast<float*>(out)[m * ldo + n] = acc;
  }
}

cudaError_t launch_splitk_reduce(const float* partial, int splits, int64_t M, int64_t N,
                                 const void* bias, int bias_dtype, void* out, int out_dtype,
                                 int64_t ldo, cudaStream_t stream) {
  int64_t blocks = (M * N + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  if (blocks < 1) blocks = 1;
  return launch_k(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                  partial, splits, M, N, bias, bias_dtype, out, out_dtype, ldo);
}

// ------------------------------------------------------------ debug unsort
// act_out[slot] = ic1[offsets[b] + m] for slot = sorted_ids[b*block_m + m].
__global__ void unsort_rows_kernel(const __nv_bfloat16* __restrict__ ic1, int64_t N,
                                   const int32_t* __restrict__ sorted_ids,
                                   const int32_t* __restrict__ offsets,
                                   const int32_t* __restrict__ num_blocks, int BM,
                                   __nv_bfloat16* __restrict__ act_out) {
  pdl_wait();
  pdl_launch_dependents();
  const int nb = __ldg(num_blocks);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       w < static_cast<int64_t>(nb) * BM; w += nwarps) {
    const int b = static_cast<int>(w / BM), m = static_cast<int>(w % BM);
    const int r0 = __ldg(offsets + b);
    if (m >= __ldg(offsets + b + 1) - r0) continue;
    const int slot = __ldg(sorted_ids + w);
    for (int64_t k = lane; k < N; k += 32)
      act_out[static_cast<int64_t>(slot) * N + k] = ic1[static_cast<int64_t>(r0 + m) * N + k];
  }
}

cudaError_t launch_unsort_rows(const void* ic1, int64_t N, const int32_t* sorted_ids,
                               const int32_t* offsets, const int32_t* num_blocks, int32_t block_m,
                               int64_t cap, void* act_out, cudaStream_t stream) {
  int64_t blocks = (cap * block_m + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  return launch_k(unsort_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                  reinterpret_cast<const __nv_bfloat16*>(ic1), N, sorted_ids, offsets, num_blocks,
                  block_m, reinterpret_cast<__nv_bfloat16*>(act_out));
}

}  // namespace mxq
