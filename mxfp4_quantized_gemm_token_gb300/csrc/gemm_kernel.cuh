// gemm_kernel.cuh — the tcgen05 scaled-GEMM kernel behind fp8_scaled_mm and
// both fused-MoE stages.
//
// Two orientations.  Weight-major ("swap-AB", EPI_DENSE / SILU / SCATTER):
// the weight matrix W [rows, K] is the MMA's M side (128 rows per tile, one
// TMEM lane per weight row) and the tokens are the N side (16 - 128 columns),
// so decode-size token counts cost a narrow instruction instead of a
// mostly-empty 128-row tile.  Token-major (EPI_NORMAL, large M with uniform
// weight-block scales): 128 tokens on M / the TMEM lanes and 128 / 192 / 256
// weight rows on N, so each lane's slice scale is one scalar.
//
// Warp roles (one CTA per SM, persistent over work units):
//   warp 0        TMA producer: lane 0 loads the A operand ring (for FP8 x
//                 FP8 also the B operand of the same slice, onto the same
//                 barrier); for the bf16 kinds lane 1 loads the B operand
//                 (bf16 tokens) into its own ring
//   warps 1, 2    tcgen05.mma issuers (one elected lane each; warp 1 also
//                 owns the TMEM allocation).  One thread blocks ~100 cycles
//                 per instruction, so two issuers take alternate K slices:
//                 with per-slice promotion every slice has its own TMEM
//                 buffer; whole-K kinds give each unit a pair of
//                 accumulators that the epilogue adds
//   warp 3        scale loader, four slices ahead into a shared ring: the
//                 column scales As(m, kb) (times Ws(kb) when uniform over the
//                 tile) and, when not, the per-row Ws(n, kb); token-major:
//                 As of the 128 token rows and Ws of the tile's weight
//                 blocks; MXFP4: the slice's ue8m0 bytes.  The epilogue
//                 never waits on a global load
//   warps 4..     epilogue, one to four warpgroups splitting the columns:
//                 TMEM -> registers, scale promotion (packed FMA), output
//   last 8 / 16   (bf16 kinds only) weight decode, one thread per weight
//                 row: e4m3 -> bf16 or e2m1 x 2^(e-127) -> bf16 from the
//                 shared tile into a 4-slot TMEM ring that the MMA reads as
//                 its A operand (no bf16 copy of the weights in shared
//                 memory)
//
// Block scales ("[XPU] block-FP8 linear via torch scaled_mm": activations
// BlockWise1x128, weights BlockWise128x128 or 1x128) are not powers of two, so
// they cannot ride the hardware block-scaled MMA.  Instead each 128-wide K
// slice is accumulated into its own TMEM buffer (a ring of two to four) and
// the epilogue folds it into fp32 registers with the slice's scale product:
//   acc[n, m] += Ws(n, kb) * As(m, kb) * partial_kb[n, m]
// which is the definition of the scaled product evaluated slice by slice.
// Per-tensor W8A16 scaling and MXFP4 (exact bf16 decode) accumulate in TMEM
// across all of K and scale once.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mxq {

// KIND_F8W / KIND_MXW: e4m3 / e2m1 weights decoded to bf16, bf16 tokens.
// KIND_F8H / KIND_MXH (the fused MoE): the same weights decoded to f16, one
// conversion instruction per pair; the tokens are f16 rows pre-scaled by a
// power of two whose inverse is the column scale.  MXH decodes each 32-group
// as e2m1 * 2^(e - emax) with emax the largest ue8m0 exponent of the whole
// weight row (mx_emax), accumulates over all of K, and the epilogue applies
// 2^(emax - 127) per row and the token scale per column once.
// KIND_F8Q: FP8 weights x bf16 activations quantized inside the kernel per
// 1 x 128 group (each group is one K slice of a token row) to e4m3, then the
// FP8 x FP8 product of KIND_F8F8 (decode-size W8A8 with the quantization fused).
enum { KIND_F8F8 = 0, KIND_F8W = 1, KIND_MXW = 2, KIND_F8H = 3, KIND_MXH = 4, KIND_F8Q = 5 };
__host__ __device__ constexpr bool kind_f8mma(int k) { return k == KIND_F8F8 || k == KIND_F8Q; }
__host__ __device__ constexpr bool kind_mx(int k) { return k == KIND_MXW || k == KIND_MXH; }
__host__ __device__ constexpr bool kind_f8w(int k) { return k == KIND_F8W || k == KIND_F8H; }
__host__ __device__ constexpr bool kind_f16(int k) { return k == KIND_F8H || k == KIND_MXH; }
// EPI_DENSE: weights on the MMA M side (swap-AB; decode and [1,128] blocks)
// EPI_NORMAL: tokens on the MMA M side, weights on N (large M with uniform
//             [128,128] / per-tensor weight scales: the slice scale is one
//             scalar per TMEM lane, As(m, kb) * Ws(kb))
// EPI_NORMAL_COLW: the token-major orientation with one weight scale per
//             column ([1, 128] weight blocks), staged per slice by the scale warp
enum { EPI_DENSE = 0, EPI_SILU = 1, EPI_SCATTER = 2, EPI_NORMAL = 3, EPI_NORMAL_COLW = 4 };
__host__ __device__ constexpr bool epi_normal(int e) { return e == EPI_NORMAL || e == EPI_NORMAL_COLW; }
enum { DT_BF16 = 1, DT_F32 = 2 };

struct GemmMaps {
  CUtensorMap a;      // weights; fp8 box [128 B x 128 (64 for SiLU) rows], e2m1x2 box [64 B x rows]
  CUtensorMap b[5];   // tokens; box rows 16 / 32 / 64 / 128 / 256 (grouped: b[4] 8 rows)
};

struct GemmParams {
  int M;              // dense: tokens; grouped: compact rows S
  int N;              // dense: weight rows; grouped: rows of one expert matrix (2N or K)
  int K;
  int nkb;            // ceil(K / 128)
  int tiles_n;
  int tiles_m;
  int splits;
  int kb_per_split;
  // batched dense GEMM (weight-major only): `batch` independent problems of
  // M x N x K; A and W are stacked along their rows (batch b's rows at
  // b*M / b*N), scales, bias and output advance by sa_e / sw_e / bias_e /
  // out_e per batch (the batch index takes the place of the expert)
  int batch;
  int64_t sa_e, out_e;
  // grouped (MoE) work description, produced on the device by moe_align
  int grouped;
  const int* num_blocks;
  const int* expert_ids;
  const int* offsets;
  const int* sorted_ids;
  int block_m;
  int narrow_max;     // blocks with m_size <= narrow_max use the narrowest legal MMA N
  int n_half;         // SiLU stage: intermediate size N (gate rows = [0, N))
  int act;            // SiLU stage activation: 0 SiLU-and-mul, 1 clamped SwiGLU
  float act_alpha, act_limit;
  // scales
  const float* a_scale;
  int64_t sa0, sa1;
  const float* w_scale;
  int64_t sw0, sw1, sw_e;
  int block_n;        // 0 = per-tensor (w_scale[0]); 1 or 128 = block rows
  const uint8_t* mx_scale;
  const uint8_t* mx_emax;   // MXH: largest ue8m0 exponent of each weight row [rows_total]
  int64_t mx_ld;
  int mx_cols;
  int64_t mx_rows_total;
  int mx_align;       // 4, 2 or 1: alignment of every row of the ue8m0 scales
  const void* bias;
  int bias_dtype;
  int64_t bias_e;
  const float* route_w;
  // scatter stage, fused top-k combine (or NULL): one counter per (token,
  // weight tile), zero at entry; the warp that completes a token's tile sums
  // its topk rows of y in ascending k into combine_out (bf16, row stride
  // combine_ldo)
  int* combine_cnt;
  void* combine_out;
  int64_t combine_ldo;
  int topk;
  float* h_out;       // SiLU stage, debug: the fp32 accumulator (before bias) in slot order, or NULL
  void* out;
  int out_dtype;
  int64_t ldo;
  float* partial;
  // prepacked weights (dense GEMM only), or NULL: 128 x 128-byte tiles, tile
  // (row block, K slice) at ((row / 128) * nkb + kb) * 16384, each the
  // 128-byte-swizzled shared-memory image; rows up to npad exist
  const uint8_t* wpacked;
  int npad;
  float q_eps;         // F8Q: the group-scale floor (s = max(amax, q_eps) / 448)
  int* status;
  unsigned long long budget_ns;
  int inject_stall;
  int vec_ok;
};

template <int KIND, int BT, int EPI>
struct Layout {
  // epilogue warpgroups: one for up to 64 columns, two for 128; FP8 x FP8
  // tiles of 192 / 256 columns use three / four (64 columns each)
  static constexpr int EW = (kind_f8mma(KIND) && BT >= 192) ? BT / 64 : (BT >= 128 ? 2 : 1);
  static constexpr int COLS = BT / EW;                     // token columns per epilogue WG
  static constexpr int CONV_WARP0 = 4 + 4 * EW;
  // weight-decode warps, in groups of eight (one thread per weight row and
  // K half).  Two groups that take alternate K slices where the registers
  // allow it (MXFP4 tiles of up to 64 token columns, FP8-block tiles of 32):
  // one group's decode is latency-bound (its integer ALU work leaves the
  // pipe half idle)
  static constexpr int NDG =
      ((KIND == KIND_MXW && BT <= 64) || (KIND == KIND_MXH && BT <= 32) ||
       (kind_f8w(KIND) && BT <= 32))
          ? 2
          : 1;
  // bf16 kinds: weight-decode warps; F8Q: one warpgroup quantizing the tokens
  static constexpr int NCV = (KIND == KIND_F8F8) ? 0 : (KIND == KIND_F8Q ? 4 : 8 * NDG);
  static constexpr int kThreads = 128 * (1 + EW) + 32 * NCV;
  // MXFP4: one A stage holds two consecutive K slices of a unit, loaded as
  // 128-byte rows (K 256); the TMA streams 128-byte rows about 1.5x faster
  // than 64-byte ones.  A unit with an odd slice count ends on a stage with
  // one slice (the box's other half is the zero fill past K).
  static constexpr int A_PER = kind_mx(KIND) ? 2 : 1;      // K slices per A stage
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = BT * 128 * (kind_f8mma(KIND) ? 1 : 2);
  // F8Q: the raw bf16 token slice of each stage (two 64-column halves)
  static constexpr int X_BYTES = (KIND == KIND_F8Q) ? BT * 256 : 0;
  static constexpr int STG = EW >= 4 ? 8 : 16;             // token columns staged per pass
  // TMEM columns loaded per wait (bounded by registers: acc + one group
  // live).  The token-major epilogue at 512 threads reads its 64 columns with
  // one wait, so the accumulator buffer goes back to the MMA before any FMA.
  static constexpr int GRP = (epi_normal(EPI) && kThreads == 512)
                                 ? 64
                                 : (kThreads >= 640 ? 16 : ((kThreads >= 512 || COLS > 64) ? 32 : COLS));
  // output staging of the weight-major epilogue (the token-major one stores directly)
  static constexpr int OUT_BYTES = epi_normal(EPI) ? 0 : EW * STG * 128 * 4;
  static constexpr int SSLOTS = 8;                         // scale ring depth
  static constexpr int MISC_BYTES = 16384;
  static constexpr int BUDGET = 225 * 1024 - 1024;   // minus alignment slack
  static constexpr int FIXED = OUT_BYTES + MISC_BYTES;
  // F8F8: A and B stages in lock step; bf16 kinds: the B ring 4 deep when it fits
  static constexpr int BS_PREF =
      kind_f8mma(KIND) ? 0 : (B_BYTES * 4 + 4 * A_BYTES + FIXED <= BUDGET ? 4 : 2);
  static constexpr int AS_RAW =
      kind_f8mma(KIND) ? (BUDGET - FIXED) / (A_BYTES + B_BYTES + X_BYTES)
                          : (BUDGET - FIXED - BS_PREF * B_BYTES) / A_BYTES;
  static constexpr int AS = AS_RAW > 12 ? 12 : AS_RAW;
  static constexpr int BS = kind_f8mma(KIND) ? AS : BS_PREF;
  static constexpr int TOTAL = AS * A_BYTES + BS * B_BYTES + AS * X_BYTES + OUT_BYTES + MISC_BYTES;
  // TMEM accumulator buffers (the bf16 kinds keep columns 256.. for the
  // decoded-weight ring)
  static constexpr int NBUF = (BT > 128 || (KIND != KIND_F8F8 && BT == 128)) ? 2 : 4;
  // each accumulator starts at a power-of-two column offset (192-wide tiles
  // take 256-column slots); the allocation is a power of two
  static constexpr int BSTRIDE = BT > 128 ? 256 : BT;
  // bf16 kinds: decoded weight slices (128 rows x 128 K bf16 = 64 TMEM
  // columns each) live in a TMEM ring after the accumulators and feed the
  // MMA's A operand directly: MXFP4 six slots when the accumulators leave
  // room (tiles of up to 32 tokens), else four; an even count, so that each
  // slot is filled by one decode group and read by one MMA issuer
  static constexpr int C_TCOL = kind_f8mma(KIND) ? 256 : (NBUF * BSTRIDE < 128 ? 128 : NBUF * BSTRIDE);
  static constexpr int CS_RAW = (512 - C_TCOL) / 64;
  static constexpr int CS = kind_f8mma(KIND) ? 0 : ((kind_mx(KIND) && CS_RAW >= 6) ? 6 : 4);
  static constexpr int TMEM_COLS = kind_f8mma(KIND) ? NBUF * BSTRIDE : 512;
  static_assert(kind_f8mma(KIND) || (NBUF * BSTRIDE <= C_TCOL && C_TCOL + CS * 64 <= 512 && CS <= 8 &&
                                     CS % 2 == 0),
                "accumulators overlap the decode ring");
  static_assert(AS >= 2 && BS >= 2, "pipeline too shallow");
  // two consumers take alternate slices of the A ring (decode groups, or the
  // MMA issuers of FP8 x FP8): with three stages one of them can pass a
  // parity wait a lap early (found by the CPU model of the ring protocol)
  static_assert(AS >= 4 || (A_PER == 1 && NDG == 1 && !kind_f8mma(KIND)), "A ring too shallow");
  static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory over budget");
  static_assert(COLS % 32 == 0 && COLS <= 128, "epilogue column split");
  static_assert(SSLOTS * BT * 4 <= 8192, "scale ring size");
};

struct Unit {
  int n0;       // first weight row of the tile inside its matrix (scales, bias, output)
  int m0;       // first token row (dense) / compact row (grouped)
  int rows;     // valid token columns
  int kb0, kb1;
  int e;        // expert (grouped) or 0
  int blk;      // expert block (grouped)
  int split;
  int tn;
  int wrow0, wrow1;   // TMA row coordinates of the MMA-A box(es)
  int brow;           // TMA row coordinate of the MMA-B box
  int n_inst;   // MMA instruction N
  int bvar;     // MMA-B box variant (maps.b[bvar])
  int brows;    // rows of that box (the B tile's rows in shared memory)
  int lvar;     // box variant the tokens are loaded with (maps.b[lvar])
  int lrows;    // rows it loads (<= brows; rows past it are never stored)
};

__device__ __forceinline__ int box_variant(int n) {
  return n <= 16 ? 0 : (n <= 32 ? 1 : (n <= 64 ? 2 : (n <= 128 ? 3 : 4)));
}

template <int EPI, int BT>
__device__ __forceinline__ Unit get_unit(const GemmParams& p, int u) {
  Unit U;
  if (!p.grouped) {
    const int per = p.tiles_m * p.splits;
    const int per_b = p.tiles_n * per;
    U.e = (p.batch > 1) ? u / per_b : 0;
    const int ub = u - U.e * per_b;
    U.tn = ub / per;
    const int r = ub - U.tn * per;
    const int tm = r / p.splits;
    U.split = r - tm * p.splits;
    U.kb0 = U.split * p.kb_per_split;
    U.kb1 = min(p.nkb, U.kb0 + p.kb_per_split);
    U.blk = 0;
    U.n_inst = BT;
    U.bvar = box_variant(BT);
    U.brows = BT;
    U.lvar = U.bvar;
    U.lrows = BT;
    if (epi_normal(EPI)) {
      // 128 tokens (A, TMEM lanes) x BT weight rows (B, TMEM columns)
      U.n0 = U.tn * BT;
      U.m0 = tm * 128;
      U.rows = min(128, p.M - U.m0);
      U.wrow0 = U.m0;
      U.wrow1 = U.m0;
      U.brow = U.n0;
    } else {
      U.n0 = U.tn * 128;
      U.m0 = tm * BT;
      U.rows = min(BT, p.M - U.m0);
      U.wrow0 = U.e * p.N + U.n0;
      U.wrow1 = U.wrow0;
      U.brow = U.e * p.M + U.m0;
    }
  } else {
    U.blk = u / p.tiles_n;
    U.tn = u - U.blk * p.tiles_n;
    U.split = 0;
    U.e = __ldg(p.expert_ids + U.blk);
    U.m0 = __ldg(p.offsets + U.blk);
    U.rows = __ldg(p.offsets + U.blk + 1) - U.m0;
    U.kb0 = 0;
    U.kb1 = p.nkb;
    const int64_t base = static_cast<int64_t>(U.e) * p.N;
    if (EPI == EPI_SILU) {
      U.n0 = U.tn * 64;
      U.wrow0 = static_cast<int>(base + U.n0);
      U.wrow1 = static_cast<int>(base + p.n_half + U.n0);
    } else {
      U.n0 = U.tn * 128;
      U.wrow0 = static_cast<int>(base + U.n0);
      U.wrow1 = U.wrow0;
    }
    // per-block instruction shape: the narrowest legal N (multiple of 16)
    // that covers the block, or the full tile width
    const int fit = ((U.rows + 15) / 16) * 16;
    U.n_inst = (U.rows <= p.narrow_max) ? min(fit, BT) : BT;
    U.bvar = box_variant(U.n_inst);
    U.brows = 16 << U.bvar;
    // a block of at most 8 slots loads 8 token rows: the MMA's other 8 rows
    // of B hold stale data that only feeds accumulator columns past the
    // block, which are never stored (token tiles share the TMA engine with
    // the weight stream)
    U.lvar = (U.n_inst == 16 && U.rows <= 8) ? 4 : U.bvar;
    U.lrows = (U.n_inst == 16 && U.rows <= 8) ? 8 : U.brows;
    U.brow = U.m0;
  }
  return U;
}

// weight row (inside its matrix) held by TMEM lane `lane` of the tile
template <int EPI>
__device__ __forceinline__ int lane_row(const GemmParams& p, const Unit& U, int lane) {
  if (EPI == EPI_SILU) return lane < 64 ? U.n0 + lane : p.n_half + U.n0 + (lane - 64);
  return U.n0 + lane;
}

template <int EPI>
__device__ __forceinline__ bool lane_row_valid(const GemmParams& p, const Unit& U, int lane) {
  if (EPI == EPI_SILU) return U.n0 + (lane & 63) < p.n_half;
  return U.n0 + lane < p.N;
}

__device__ __forceinline__ float load_bias(const GemmParams& p, int64_t idx) {
  if (p.bias == nullptr) return 0.f;
  if (p.bias_dtype == DT_BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.bias)[idx]);
  return reinterpret_cast<const float*>(p.bias)[idx];
}

// ------------------------------------------------------------ weight decode
// Weight decode, exact.  Every e4m3 value and every e2m1 value is a normal f16
// (or zero), so the pair is first widened to f16; those bits shifted right by
// 3 form a bf16 with the same mantissa and a biased exponent 112 short, and
// one bf16 multiply by 2^112 (or, for MXFP4, by 2^(e - 127 + 112), the
// group's ue8m0 scale folded in) restores the value.  The 32-bit source word
// is split into byte / half registers by a vector move, so no extraction
// instructions are spent (the decode is bound by the integer ALU pipe).
__device__ __forceinline__ uint32_t f16x2_bits_to_bf16x2(uint32_t h, uint32_t k2) {
  uint32_t t = ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&t);
  v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&k2));
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t word, uint32_t& lo, uint32_t& hi) {
  uint32_t h0, h1;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b; }"
      : "=r"(h0), "=r"(h1) : "r"(word));
  lo = f16x2_bits_to_bf16x2(h0, 0x77807780u);
  hi = f16x2_bits_to_bf16x2(h1, 0x77807780u);
}
__device__ __forceinline__ void e2m1x8_to_bf16x8(uint32_t word, uint32_t k2, uint32_t* o) {
  uint32_t h0, h1, h2, h3;
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(word));
  o[0] = f16x2_bits_to_bf16x2(h0, k2);
  o[1] = f16x2_bits_to_bf16x2(h1, k2);
  o[2] = f16x2_bits_to_bf16x2(h2, k2);
  o[3] = f16x2_bits_to_bf16x2(h3, k2);
}

// f16 decode (KIND_F8H / KIND_MXH): e4m3 and e2m1 values are exact f16, so
// the conversion instruction's result is the operand; MXFP4 multiplies each
// pair by the group's f16 factor 2^(e - emax) (exact while e - emax >= -23).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t word, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b; }"
      : "=r"(lo), "=r"(hi) : "r"(word));
}
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t word, uint32_t f2, uint32_t* o) {
  uint32_t h[4];
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(word));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h[i]), *reinterpret_cast<const __half2*>(&f2));
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
}
// f16 bits of 2^d for d <= 0 (subnormal below 2^-14, zero below 2^-24)
__device__ __forceinline__ uint32_t f16_pow2(int d) {
  return d >= -14 ? static_cast<uint32_t>(d + 15) << 10 : (d >= -24 ? 1u << (d + 24) : 0u);
}

// MXFP4: the two ue8m0 bytes (low byte first) of 32-groups 2*half and
// 2*half + 1 of slice kb in the scale row srow; 2^0 past the unit's slices
// and past K (the weights there are zero)
__device__ __forceinline__ uint32_t mx_scale2(const GemmParams& p, const uint8_t* srow, int kb,
                                              int kb1, int half) {
  const int col = kb * 4 + 2 * half;
  if (kb >= kb1 || col >= p.mx_cols) return 0x7F7Fu;
  if (p.mx_align >= 2 && col + 2 <= p.mx_cols)
    return __ldg(reinterpret_cast<const uint16_t*>(srow + col));
  const uint32_t b0 = __ldg(srow + col);
  const uint32_t b1 = (col + 1 < p.mx_cols) ? __ldg(srow + col + 1) : 127u;
  return b0 | (b1 << 8);
}

// Barrier of the 128 epilogue threads on an mbarrier, so that it is bounded
// like every other wait (a plain bar.sync would hang if one warp gave up).
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, const WaitCtx& w) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase, w);
  phase ^= 1;
  return ok;
}

// ------------------------------------------------------------------ kernel
template <int KIND, int EPI, int BT, bool PROMOTE>
__global__ void __launch_bounds__(Layout<KIND, BT, EPI>::kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  using L = Layout<KIND, BT, EPI>;
  static_assert(!kind_f8mma(KIND) || PROMOTE, "FP8 x FP8 slices are always promoted (two issuers rely on it)");
  static_assert(PROMOTE || L::STG == 16, "whole-K epilogue reads 16-column chunks");
  constexpr int AS = L::AS, BS = L::BS, CS = L::CS, EW = L::EW, COLS = L::COLS;
  constexpr int SSL = L::SSLOTS, STG = L::STG, GRP = L::GRP, NB = L::NBUF;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // align by offsetting the shared array itself (an integer round-trip would
  // turn every shared access below into a generic one)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + AS * L::A_BYTES;
  uint8_t* sX = sB + BS * L::B_BYTES;    // F8Q raw token slices
  float* sOut = reinterpret_cast<float*>(sX + AS * L::X_BYTES);
  uint8_t* misc = reinterpret_cast<uint8_t*>(sOut) + L::OUT_BYTES;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* a_empty = a_full + 12;
  uint64_t* b_full = a_empty + 12;
  uint64_t* b_empty = b_full + 12;
  uint64_t* c_full = b_empty + 12;
  uint64_t* c_empty = c_full + 8;
  uint64_t* t_full = c_empty + 8;
  uint64_t* t_empty = t_full + 4;
  uint64_t* s_full = t_empty + 4;
  uint64_t* s_empty = s_full + SSL;
  uint64_t* drain = s_empty + SSL;   // one per MMA issuer
  uint64_t* epi_bar = drain + 2;     // bounded barriers, one per epilogue warpgroup
  // F8Q: q_full[stage] (quantized B operand ready, on b_full), and the ring of
  // token-group scales per slice, qs_full / qs_empty [8]
  uint64_t* q_full = b_full;
  uint64_t* qs_full = epi_bar + 4;
  uint64_t* qs_empty = qs_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qs_empty + 8);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float* sAsc = reinterpret_cast<float*>(misc + 1024);            // [SSL][BT] column scales
  float* sWr = reinterpret_cast<float*>(misc + 1024 + 8192);      // [SSL][128] row scales
  // F8Q: [8][BT] token-group scales As(m, kb), slot = slice % 8
  float* sQs = reinterpret_cast<float*>(misc + 1024 + 4096);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WaitCtx wc{p.status, abort_flag, p.budget_ns};
  // a row scale per TMEM lane is needed when Ws is not uniform over the tile
  const bool lane_ws = PROMOTE && (p.block_n == 1 || EPI == EPI_SILU);

  if (threadIdx.x == 0) {
    for (int i = 0; i < AS; ++i) {
      mbar_init(&a_full[i], 1);
      // the MMA (FP8-MMA kinds) or the eight warps of the decode group of
      // each slice of the stage (twice over for a stage with one slice)
      mbar_init(&a_empty[i], kind_f8mma(KIND) ? 1 : 8 * L::A_PER);
    }
    for (int i = 0; i < BS; ++i) {
      mbar_init(&b_full[i], KIND == KIND_F8Q ? 4 : 1);   // F8Q: q_full, the 4 quantizer warps
      mbar_init(&b_empty[i], 1);
    }
    if (KIND == KIND_F8Q) {
      for (int i = 0; i < 8; ++i) {
        mbar_init(&qs_full[i], 4);
        mbar_init(&qs_empty[i], 4 * EW);
      }
    }
    for (int i = 0; i < CS; ++i) {
      mbar_init(&c_full[i], 8);
      mbar_init(&c_empty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4 * EW);
    }
    for (int i = 0; i < SSL; ++i) {
      mbar_init(&s_full[i], 1);
      // MXFP4 slots feed one decode group (bf16) or a decode group and the
      // epilogue (f16, per-slice promotion)
      mbar_init(&s_empty[i], kind_mx(KIND) ? 8 : 4 * EW);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int g = 0; g < EW; ++g) mbar_init(&epi_bar[g], 128);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // (maps.a holds the weights in the weight-major orientation; prepacked
  // weights are read without a tensor map)
  if (warp == 0 && lane == 0 && (epi_normal(EPI) || p.wpacked == nullptr))
    tma_prefetch_desc(&maps.a);
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above touches no global memory; from here on the previous
  // kernel's results (tokens, scales, the expert-block table) are read
  pdl_wait();
  pdl_launch_dependents();

  const int total = p.grouped ? __ldg(p.num_blocks) * p.tiles_n
                              : p.tiles_n * p.tiles_m * p.splits * max(1, p.batch);

  if (warp == 0) {
    // ------------------------------------------------ operand producer
    if (lane == 0 && !p.inject_stall) {
      // weights on the A side are streamed once: evict them first; tokens on
      // the A side (token-major path) are reused by every weight tile
      const uint64_t pol = epi_normal(EPI) ? policy_evict_last() : policy_evict_first();
      // the copies of slice kb of unit U (MXFP4: slices kb and kb + 1) into
      // A stage s (with the tokens too for the FP8-MMA kinds, which fill
      // both operands on one barrier)
      auto issue_a = [&](int s, const Unit& U, int kb) {
        const int kc = kind_mx(KIND) ? kb * 64 : kb * 128;
        uint8_t* dst = sA + s * L::A_BYTES;
        if (epi_normal(EPI) && p.wpacked != nullptr) {
          // token-major with prepacked weights: the B operand (BT weight
          // rows of slice kb) is BT / 64 contiguous 8 KB halves of packed
          // tiles; halves past the padded row count are not loaded (their
          // accumulator columns are never stored)
          uint32_t bytes = L::A_BYTES;
#pragma unroll
          for (int c = 0; c < BT / 64; ++c)
            if (U.brow + 64 * c < p.npad) bytes += 8192;
          mbar_expect_tx(&a_full[s], bytes);
#pragma unroll
          for (int c = 0; c < BT / 64; ++c) {
            const int row = U.brow + 64 * c;
            if (row < p.npad)
              bulk_load(sB + s * L::B_BYTES + c * 8192,
                        p.wpacked + (static_cast<int64_t>(row >> 7) * p.nkb + kb) * 16384 +
                            ((row >> 6) & 1) * 8192,
                        8192, &a_full[s]);
          }
        } else if (KIND == KIND_F8F8) {
          // FP8 x FP8: both operands of the slice land on one barrier
          mbar_expect_tx(&a_full[s], L::A_BYTES + U.brows * 128);
          tma_load_2d(sB + s * L::B_BYTES, &maps.b[U.bvar], &a_full[s], kb * 128, U.brow);
        } else if (KIND == KIND_F8Q) {
          // weights and the bf16 token slice (two 64-column halves) on one
          // barrier; the quantizer warps turn the tokens into the e4m3 B
          mbar_expect_tx(&a_full[s], L::A_BYTES + U.brows * 256);
          uint8_t* xd = sX + s * L::X_BYTES;
          tma_load_2d(xd, &maps.b[U.bvar], &a_full[s], kb * 128, U.brow);
          tma_load_2d(xd + U.brows * 128, &maps.b[U.bvar], &a_full[s], kb * 128 + 64, U.brow);
        } else {
          mbar_expect_tx(&a_full[s], L::A_BYTES);
        }
        if (!epi_normal(EPI) && EPI != EPI_SILU && p.wpacked != nullptr) {
          // weight-major with prepacked weights: one contiguous 16 KB tile
          bulk_load_hint(dst, p.wpacked + (static_cast<int64_t>(U.wrow0 >> 7) * p.nkb + kb) * 16384,
                         16384, &a_full[s], pol);
        } else if (EPI == EPI_SILU) {
          tma_load_2d_hint(dst, &maps.a, &a_full[s], kc, U.wrow0, pol);
          tma_load_2d_hint(dst + L::A_BYTES / 2, &maps.a, &a_full[s], kc, U.wrow1, pol);
        } else {
          tma_load_2d_hint(dst, &maps.a, &a_full[s], kc, U.wrow0, pol);
        }
      };
      // (lane 1 fills the token ring of the bf16 / f16 kinds)
      uint32_t it = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        for (int kb = U.kb0; kb < U.kb1; kb += L::A_PER, ++it) {
          const int s = it % AS;
          if (!mbar_wait(&a_empty[s], ((it / AS) & 1) ^ 1, wc)) goto prod_done;
          issue_a(s, U, kb);
        }
      }
    prod_done:
      if (*abort_flag) {
        // let every copy already issued land before the CTA goes away
        volatile int zero = 0;
        WaitCtx dw{p.status, &zero, 1000000000ull};
        const uint32_t first = it > static_cast<uint32_t>(AS) ? it - AS : 0;
        for (uint32_t i = first; i < it; ++i) mbar_wait(&a_full[i % AS], (i / AS) & 1, dw);
      }
    } else if (lane == 1 && !kind_f8mma(KIND) && !p.inject_stall) {
      // bf16 kinds: the B operand (bf16 / f16 tokens, two 64-column halves)
      // of every slice, in slice order, into its own ring released by the MMA
      uint32_t itb = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++itb) {
          const int sb = itb % BS;
          if (!mbar_wait(&b_empty[sb], ((itb / BS) & 1) ^ 1, wc)) goto prod_b_done;
          uint8_t* dst = sB + sb * L::B_BYTES;
          mbar_expect_tx(&b_full[sb], U.lrows * 256);
          tma_load_2d(dst, &maps.b[U.lvar], &b_full[sb], kb * 128, U.brow);
          tma_load_2d(dst + U.brows * 128, &maps.b[U.lvar], &b_full[sb], kb * 128 + 64, U.brow);
        }
      }
    prod_b_done:
      if (*abort_flag) {
        volatile int zero = 0;
        WaitCtx dw{p.status, &zero, 1000000000ull};
        const uint32_t first = itb > static_cast<uint32_t>(BS) ? itb - BS : 0;
        for (uint32_t i = first; i < itb; ++i) mbar_wait(&b_full[i % BS], (i / BS) & 1, dw);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------ MMA issuer
    // the whole warp runs the loop; one elected lane issues.  With per-slice
    // promotion every slice has its own TMEM buffer and two issuing warps
    // take every other slice.
    {
      // Two issuers, taking alternate slices of the CTA's slice sequence
      // (global index ia, across units), so that issuer i consumes exactly
      // the slices that decode group i fills when the decode runs as two
      // groups; each of its ring waits then follows a fill of the same
      // producer that is known to be complete, and no parity wait can see
      // a phase one lap behind.  Promoted kinds: every slice has its own
      // buffer.  Whole-K kinds: each unit has a pair of accumulators, issuer
      // i summing its slices of the unit into buffer (2 * unit + i) % NB;
      // the epilogue adds the pair.  An issuer with no slice in a unit (a
      // one-slice unit whose slice is the other issuer's) hands over its
      // buffer unwritten, so every barrier phase stays in step.
      constexpr uint32_t NISS = 2;
      const uint32_t mine = (warp == 1) ? 0u : 1u;
      uint32_t ia = 0, ib = 0, au = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        const int brows = U.brows;
        const int nsl = U.kb1 - U.kb0;
        const uint32_t idesc =
            kind_f8mma(KIND) ? idesc_e4m3(128, U.n_inst)
                                : (kind_f16(KIND) ? idesc_f16(128, U.n_inst) : idesc_bf16(128, U.n_inst));
        uint32_t ubuf = 0;
        if (!PROMOTE) {
          const uint32_t tb = 2 * au + mine;
          ubuf = tb % NB;
          if (!mbar_wait_warp(&t_empty[ubuf], ((tb / NB) & 1) ^ 1, wc)) goto mma_done;
          if (nsl == 1 && ia % NISS != mine) {
            if (elect_one()) mma_commit(&t_full[ubuf]);
            __syncwarp();
          }
        }
        bool first = true;   // this issuer's first slice of the unit
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          const int l = kb - U.kb0;
          const bool take = ia % NISS == mine;
          if (!take) {
            ++ia;
            ++ib;
            if (PROMOTE) ++au;
            continue;
          }
          const uint32_t buf = PROMOTE ? au % NB : ubuf;
          if (PROMOTE)
            if (!mbar_wait_warp(&t_empty[buf], ((au / NB) & 1) ^ 1, wc)) goto mma_done;
          // FP8 x FP8 reads the A ring; the bf16 kinds read the decoded C ring
          constexpr int RA = kind_f8mma(KIND) ? AS : CS;
          const int sa = ia % RA;
          uint64_t* full = kind_f8mma(KIND) ? &a_full[sa] : &c_full[sa];
          if (!mbar_wait_warp(full, (ia / RA) & 1, wc)) goto mma_done;
          const int sb = ib % BS;
          // bf16 kinds: the token ring; F8Q: the quantized tokens of the stage
          if (KIND != KIND_F8F8)
            if (!mbar_wait_warp(&b_full[sb], (ib / BS) & 1, wc)) goto mma_done;
          tc_fence_after();
          const uint32_t d = tmem_base + buf * L::BSTRIDE;
          // accumulate except on the first K step of this issuer's first slice
          const bool fresh = PROMOTE || first;
          first = false;
          const bool leader = elect_one();
          if (leader) {
          if (kind_f8mma(KIND)) {
            const uint32_t a0 = smem_u32(sA + sa * L::A_BYTES);
            const uint32_t b0 = smem_u32(sB + sb * L::B_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t acc = (fresh && j == 0) ? 0u : 1u;
              mma_f8f6f4(d, sw128_desc(a0 + 32 * j), sw128_desc(b0 + 32 * j), idesc, acc);
            }
            mma_commit(&a_empty[sa]);
          } else {
            // A = the decoded slice in TMEM (row = lane, two bf16 per column:
            // K-step j of 16 reads columns 8j .. 8j+7), B = tokens in shared
            const uint32_t a0 = tmem_base + L::C_TCOL + sa * 64;
            const uint32_t b0 = smem_u32(sB + sb * L::B_BYTES);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t acc = (fresh && j == 0) ? 0u : 1u;
              const uint32_t bo = b0 + (j >> 2) * (brows * 128) + (j & 3) * 32;
              mma_f16_ts(d, a0 + 8 * j, sw128_desc(bo), idesc, acc);
            }
            mma_commit(&c_empty[sa]);
          }
          if (!kind_f8mma(KIND)) mma_commit(&b_empty[sb]);
          }
          ++ia;
          ++ib;
          if (PROMOTE) {
            if (leader) mma_commit(&t_full[buf]);
            ++au;
          } else if (l + static_cast<int>(NISS) >= nsl) {
            if (leader) mma_commit(&t_full[buf]);   // this issuer's last slice of the unit
          }
          __syncwarp();
        }
        if (!PROMOTE) ++au;
      }
    mma_done:
      if (*abort_flag) {
        // each issuer waits for its own MMAs before the TMEM is freed
        if (elect_one()) mma_commit(&drain[mine]);
        volatile int zero = 0;
        WaitCtx dw{p.status, &zero, 1000000000ull};
        mbar_wait(&drain[mine], 0, dw);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------ scale loader
    if (KIND == KIND_F8W && !PROMOTE) {
      // per-tensor weights: no slice scales
    } else if (kind_mx(KIND)) {
      // MXFP4: the decode threads load their own ue8m0 bytes
    } else if (epi_normal(EPI)) {
      // token-major: the epilogue threads read their own token scales; with
      // per-row weight scales ([1, 128] blocks) the weight rows are the
      // tile's columns, and this warp stages each slice's BT column scales
      // Ws(n, kb) in the shared ring, four slices ahead
      if (EPI == EPI_NORMAL_COLW) {
        constexpr int NW = BT / 32;
        uint32_t is = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
          const Unit U = get_unit<EPI, BT>(p, u);
          float rw[4][NW];
          auto fetch = [&](int kb, float* w) {
#pragma unroll
            for (int i = 0; i < NW; ++i) {
              const int n = U.n0 + lane + 32 * i;
              w[i] = n < p.N ? __ldg(p.w_scale + static_cast<int64_t>(n) * p.sw0 + kb * p.sw1) : 1.f;
            }
          };
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (U.kb0 + q < U.kb1) fetch(U.kb0 + q, rw[q]);
          for (int kb = U.kb0; kb < U.kb1; kb += 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (kb + q < U.kb1) {
                const int slot = is % SSL;
                if (!mbar_wait(&s_empty[slot], ((is / SSL) & 1) ^ 1, wc)) goto ncol_done;
#pragma unroll
                for (int i = 0; i < NW; ++i) sAsc[slot * BT + lane + 32 * i] = rw[q][i];
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_full[slot]);
                ++is;
                if (kb + q + 4 < U.kb1) fetch(kb + q + 4, rw[q]);
              }
            }
          }
        }
      ncol_done:;
      }
    } else if (PROMOTE) {
      // Four slices of look-ahead in registers hide the global-load latency.
      constexpr int NA = BT / 32;
      uint32_t is = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        float ra[4][NA], rw[4][4], ru[4];
        auto fetch = [&](int kb, float* a, float* w, float& uni) {
#pragma unroll
          for (int i = 0; i < NA; ++i) {
            const int j = lane + 32 * i;
            a[i] = (p.a_scale != nullptr && j < U.rows)
                       ? __ldg(p.a_scale + U.e * p.sa_e + static_cast<int64_t>(U.m0 + j) * p.sa0 +
                               kb * p.sa1)
                       : 1.f;
          }
          if (lane_ws) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = lane + 32 * i;
              const int row = lane_row_valid<EPI>(p, U, r) ? lane_row<EPI>(p, U, r) : 0;
              w[i] = __ldg(p.w_scale + U.e * p.sw_e + (row / p.block_n) * p.sw0 + kb * p.sw1);
            }
            uni = 1.f;
          } else {
            uni = (p.block_n == 0)
                      ? __ldg(p.w_scale + U.e * p.sw_e)
                      : __ldg(p.w_scale + U.e * p.sw_e + (U.n0 / p.block_n) * p.sw0 + kb * p.sw1);
          }
        };
        auto publish = [&](const float* a, const float* w, float uni) -> bool {
          const int slot = is % SSL;
          if (!mbar_wait(&s_empty[slot], ((is / SSL) & 1) ^ 1, wc)) return false;
#pragma unroll
          for (int i = 0; i < NA; ++i) sAsc[slot * BT + lane + 32 * i] = a[i] * uni;
          if (lane_ws) {
#pragma unroll
            for (int i = 0; i < 4; ++i) sWr[slot * 128 + lane + 32 * i] = w[i];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_full[slot]);
          ++is;
          return true;
        };
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (U.kb0 + q < U.kb1) fetch(U.kb0 + q, ra[q], rw[q], ru[q]);
        for (int kb = U.kb0; kb < U.kb1; kb += 4) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (kb + q < U.kb1) {
              if (!publish(ra[q], rw[q], ru[q])) goto scale_done;
              if (kb + q + 4 < U.kb1) fetch(kb + q + 4, ra[q], rw[q], ru[q]);
            }
          }
        }
      }
    }
  scale_done:;
  } else if (warp >= L::CONV_WARP0) {
    // ------------------------------------------- weight decode to bf16
    // Thread = weight row of the tile = TMEM lane; the two warps of a lane
    // quarter take the two 64-wide K halves of the slice.  Each thread reads
    // its row's bytes from the (swizzled) shared tile, decodes them and
    // stores 32 columns of bf16 pairs into the TMEM ring slot, which the
    // MMA then reads as its A operand.
    if constexpr (KIND == KIND_F8Q) {
      // --------------------------------------------- token quantization
      // Thread = (token row j = t / 4 of the tile, quarter q4 = t % 4 of the
      // slice's 128 K values).  Each 1 x 128 group is one K slice of a row:
      // amax over the group, s = max(amax, eps) / 448 and codes
      // e4m3(clamp(x / s, -448, 448)), both IEEE divisions, round to nearest
      // even, exactly as the per_token_group_quant_fp8 kernel; the codes go to
      // the slice's B stage in the 128-byte-swizzled layout the MMA reads,
      // s to the scale ring the epilogue reads.
      const int t = static_cast<int>(threadIdx.x) - L::CONV_WARP0 * 32;
      const int j = t >> 2, q4 = t & 3;
      uint32_t i = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++i) {
          const int st = static_cast<int>(i % AS), qs = static_cast<int>(i % 8);
          if (!mbar_wait(&a_full[st], (i / AS) & 1, wc)) goto quant_done;
          if (!mbar_wait(&qs_empty[qs], ((i / 8) & 1) ^ 1, wc)) goto quant_done;
          const bool valid = j < U.rows;
          float v[32];
          const uint8_t* xrow = sX + st * L::X_BYTES + (q4 >> 1) * (U.brows * 128) + j * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int chunk = 4 * (q4 & 1) + c;
            const uint4 w = *reinterpret_cast<const uint4*>(xrow + ((chunk ^ (j & 7)) << 4));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              v[8 * c + 2 * h] = __uint_as_float(wv[h] << 16);
              v[8 * c + 2 * h + 1] = __uint_as_float(wv[h] & 0xFFFF0000u);
            }
          }
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float a = fabsf(v[k]);
            amax = (a > amax) ? a : amax;
          }
#pragma unroll
          for (int off = 1; off <= 2; off <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, amax, off);
            amax = (o > amax) ? o : amax;
          }
          const float sc = __fdiv_rn((amax > p.q_eps) ? amax : p.q_eps, 448.f);
          uint32_t pk[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          if (valid) {   // rows past the tile's tokens stay zero
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float* vv = v + 4 * k;
              const uint16_t a = e4m3x2_rn(clamp448(__fdiv_rn(vv[0], sc)), clamp448(__fdiv_rn(vv[1], sc)));
              const uint16_t b = e4m3x2_rn(clamp448(__fdiv_rn(vv[2], sc)), clamp448(__fdiv_rn(vv[3], sc)));
              pk[k] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
            }
          }
          uint8_t* brow = sB + st * L::B_BYTES + j * 128;
          *reinterpret_cast<uint4*>(brow + (((2 * q4) ^ (j & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(brow + (((2 * q4 + 1) ^ (j & 7)) << 4)) =
              make_uint4(pk[4], pk[5], pk[6], pk[7]);
          if (q4 == 0) sQs[qs * BT + j] = valid ? sc : 1.f;
          // the codes are read by the tensor core (async proxy)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&q_full[st]);
            mbar_arrive(&qs_full[qs]);
          }
        }
      }
    quant_done:;
    } else if constexpr (KIND != KIND_F8F8) {
      const int cw = warp - L::CONV_WARP0;
      const uint32_t grp = static_cast<uint32_t>(cw >> 3);   // takes slices with ia % NDG == grp
      const int half = (cw >> 2) & 1;
      const int r = (warp & 3) * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                             L::C_TCOL + half * 32;
      uint32_t ia = 0, ic = 0;
      uint32_t sbase = 0;   // A stages of the CTA's earlier units
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit U = get_unit<EPI, BT>(p, u);
        const int nsl = U.kb1 - U.kb0;
        int emax = 0;   // MXH: the row's largest scale exponent (the f16 reference)
        // MXFP4: this thread's scale bytes, loaded by the thread itself two
        // of its slices ahead (sq0: the next slice it decodes, sq1: the one
        // after), so that no slice waits on a hand-off from another warp
        const uint8_t* srow = nullptr;
        uint32_t sq0 = 0, sq1 = 0;
        if (kind_mx(KIND)) {
          int64_t grow = (EPI == EPI_SILU) ? static_cast<int64_t>(r < 64 ? U.wrow0 + r : U.wrow1 + (r - 64))
                                           : static_cast<int64_t>(U.wrow0) + r;
          if (grow >= p.mx_rows_total) grow = p.mx_rows_total - 1;
          if (KIND == KIND_MXH) emax = __ldg(p.mx_emax + grow);
          srow = p.mx_scale + grow * p.mx_ld;
          // the unit's first slice of this group: kb0 + ((grp - ia) mod NDG)
          const int kf = U.kb0 + static_cast<int>((grp + L::NDG - ia % L::NDG) % L::NDG);
          sq0 = mx_scale2(p, srow, kf, U.kb1, half);
          sq1 = mx_scale2(p, srow, kf + L::NDG, U.kb1, half);
        }
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++ia, ++ic) {
          if (L::NDG > 1 && ia % L::NDG != grp) continue;
          // A stage of the slice (MXFP4: two slices of the unit per stage,
          // slice half h in bytes 64h .. 64h+63 of each 128-byte row)
          const int l = kb - U.kb0;
          const uint32_t sta = sbase + static_cast<uint32_t>(l / L::A_PER);
          const int h = l % L::A_PER;
          // the stage's only slice (odd unit length): its decode group
          // arrives for both halves
          const bool single = L::A_PER == 2 && l == nsl - 1 && (nsl & 1);
          const int sa = static_cast<int>(sta % AS), sc = ic % CS;
          if (!mbar_wait(&a_full[sa], (sta / AS) & 1, wc)) goto conv_done;
          if (!mbar_wait(&c_empty[sc], ((ic / CS) & 1) ^ 1, wc)) goto conv_done;
          tc_fence_after();
          const uint8_t* src = sA + sa * L::A_BYTES;
          uint32_t w[32];
          if (kind_f8w(KIND)) {
            // 64 fp8 of row r: 16-byte chunks 4*half .. 4*half+3 of the
            // 128-byte row, stored with the 128-byte swizzle
            uint4 raw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = 4 * half + i;
              raw[i] = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_empty[sa]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t in[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                if (kind_f16(KIND))
                  e4m3x4_to_f16x4(in[t], w[8 * i + 2 * t], w[8 * i + 2 * t + 1]);
                else
                  e4m3x4_to_bf16x4(in[t], w[8 * i + 2 * t], w[8 * i + 2 * t + 1]);
              }
            }
          } else {
            // 64 e2m1 of row r: 16-byte chunks 4h + 2*half, 4h + 2*half + 1
            // of the 128-byte row (128-byte swizzle); chunk 2*half + k of
            // the slice is the 32-group with ue8m0 scale byte 2*half + k
            const uint32_t e2 = sq0;   // bytes of groups 2*half, 2*half + 1
            sq0 = sq1;
            sq1 = mx_scale2(p, srow, kb + 2 * L::NDG, U.kb1, half);
            uint4 raw[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int c = 4 * h + 2 * half + k;
              raw[k] = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
            }
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&a_empty[sa]);
              if (single) mbar_arrive(&a_empty[sa]);
            }
            if (KIND == KIND_MXH) {
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int e = static_cast<int>((e2 >> (8 * k)) & 0xFFu);
                const uint32_t f2 = f16_pow2(e - emax) * 0x10001u;
                const uint32_t in[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) e2m1x8_to_f16x8(in[j], f2, &w[16 * k + 4 * j]);
              }
            } else
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t e = (e2 >> (8 * k)) & 0xFFu;
              // bf16 2^(e - 127 + 112) when representable; else two steps
              __nv_bfloat162 sc2;
              uint32_t two_step = 0;
              {
                const int ex = static_cast<int>(e) + 112;  // biased bf16 exponent of 2^(e-15)
                if (ex >= 1 && ex <= 254) {
                  const uint32_t bits = (static_cast<uint32_t>(ex) << 7) * 0x10001u;
                  sc2 = *reinterpret_cast<const __nv_bfloat162*>(&bits);
                } else {
                  two_step = 1;
                  const uint32_t bits = 0x77807780u;
                  sc2 = *reinterpret_cast<const __nv_bfloat162*>(&bits);
                }
              }
              const uint32_t in[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                e2m1x8_to_bf16x8(in[j], *reinterpret_cast<const uint32_t*>(&sc2), &w[16 * k + 4 * j]);
              if (two_step) {
                const float f = ldexpf(1.0f, static_cast<int>(e) - 127);
                const __nv_bfloat162 s2 = __floats2bfloat162_rn(f, f);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w[16 * k + j]);
                  v = __hmul2(v, s2);
                  w[16 * k + j] = *reinterpret_cast<uint32_t*>(&v);
                }
              }
            }
          }
          tmem_st32(t_row + sc * 64, w);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c_full[sc]);
        }
        sbase += static_cast<uint32_t>((nsl + L::A_PER - 1) / L::A_PER);
      }
    conv_done:;
    }
  } else if (warp >= 4 && epi_normal(EPI)) {
    // ------------------------------------- epilogue, tokens on TMEM lanes
    // Thread = token row m; its slice scale As(m, kb) * Ws(blk, kb) is one
    // scalar (a warpgroup's 64 columns lie in one 128-row weight block), so
    // promotion is one packed FMA per pair of accumulators.  The thread reads
    // its own scales, so no wait on another warp sits in the slice loop.
    const int g = (warp - 4) >> 2;
    const int et = (threadIdx.x - 128) & 127;
    const int col0 = g * COLS;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // [1, 128] weight blocks: a scale per column (weight row), staged per
    // slice by the scale warp; the lane's token scale multiplies it
    constexpr bool colw = EPI == EPI_NORMAL_COLW;
    uint32_t au = 0, is = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit U = get_unit<EPI, BT>(p, u);
      const bool mrow = et < U.rows;
      const int ncv = min(BT, p.N - U.n0);              // valid weight columns of the tile
      const int colv = max(0, min(COLS, ncv - col0));
      const int ngr = (colv + GRP - 1) / GRP;
      float acc[COLS];
#pragma unroll
      for (int j = 0; j < COLS; ++j) acc[j] = 0.f;
      // slice scales: this thread's token row As(m, kb) and its columns'
      // weight block Ws(blk, kb), read from global memory (L1) four slices
      // ahead; rows and blocks past the tile's valid ones read a valid entry
      const float* arow = p.a_scale + static_cast<int64_t>(U.m0 + min(et, U.rows - 1)) * p.sa0;
      const int wb = min((U.n0 + col0) / 128, (p.N - 1) / 128);
      const float* wrow = p.w_scale + (p.block_n != 128 ? 0 : static_cast<int64_t>(wb) * p.sw0);
      const int64_t wk = p.block_n != 128 ? 0 : p.sw1;
      // four slices' scales at a time, with one 16-byte load where the layout
      // allows it (a thread's As row and the block's Ws row contiguous and
      // aligned); the next four are loaded while these are used
      const bool va = p.sa1 == 1 && (p.sa0 & 3) == 0 && (U.kb0 & 3) == 0 &&
                      (reinterpret_cast<uintptr_t>(p.a_scale) & 15) == 0;
      const bool vw = !colw && wk == 1 && ((static_cast<int64_t>(wb) * p.sw0) & 3) == 0 &&
                      (U.kb0 & 3) == 0 && (reinterpret_cast<uintptr_t>(p.w_scale) & 15) == 0;
      auto scales4 = [&](int kb, float* a, float* w) {
        if (va && kb + 4 <= U.kb1) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(arow + kb));
          a[0] = t.x;
          a[1] = t.y;
          a[2] = t.z;
          a[3] = t.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) a[q] = __ldg(arow + min(kb + q, U.kb1 - 1) * p.sa1);
        }
        if (colw) {
#pragma unroll
          for (int q = 0; q < 4; ++q) w[q] = 1.f;
        } else if (vw && kb + 4 <= U.kb1) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(wrow + kb));
          w[0] = t.x;
          w[1] = t.y;
          w[2] = t.z;
          w[3] = t.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) w[q] = __ldg(wrow + min(kb + q, U.kb1 - 1) * wk);
        }
      };
      float ra[4], rw[4];
      scales4(U.kb0, ra, rw);
      for (int kb4 = U.kb0; kb4 < U.kb1; kb4 += 4) {
      float na[4] = {0.f, 0.f, 0.f, 0.f}, nw[4] = {0.f, 0.f, 0.f, 0.f};
      if (kb4 + 4 < U.kb1) scales4(kb4 + 4, na, nw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kb = kb4 + q;
        if (kb >= U.kb1) break;
        const float sc = ra[q] * rw[q];
        const uint32_t buf = au % NB;
        const int slot = is % SSL;
        if (colw && !mbar_wait(&s_full[slot], (is / SSL) & 1, wc)) goto epin_done;
        if (!mbar_wait(&t_full[buf], (au / NB) & 1, wc)) goto epin_done;
        tc_fence_after();
        const float2 s2 = make_float2(sc, sc);
        const float* wcol = sAsc + slot * BT + col0;
#pragma unroll
        for (int c = 0; c < COLS / GRP; ++c) {
          if (c < ngr) {
            float v[GRP];
            tmem_ld<GRP>(tmem_base + lane_addr + buf * L::BSTRIDE + col0 + c * GRP, v);
            if (c == COLS / GRP - 1 || c + 1 == ngr) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&t_empty[buf]);
            }
            if (colw) {
              // per column: As(m, kb) * Ws(n, kb), one packed multiply more
#pragma unroll
              for (int j = 0; j < GRP; j += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(wcol + c * GRP + j);
                const float2 lo = __fmul2_rn(make_float2(w4.x, w4.y), s2);
                const float2 hi = __fmul2_rn(make_float2(w4.z, w4.w), s2);
                float* a = acc + c * GRP + j;
                const float2 r0 = __ffma2_rn(make_float2(v[j], v[j + 1]), lo, make_float2(a[0], a[1]));
                const float2 r1 = __ffma2_rn(make_float2(v[j + 2], v[j + 3]), hi, make_float2(a[2], a[3]));
                a[0] = r0.x;
                a[1] = r0.y;
                a[2] = r1.x;
                a[3] = r1.y;
              }
            } else {
#pragma unroll
              for (int j = 0; j < GRP; j += 2) {
                const float2 r = __ffma2_rn(make_float2(v[j], v[j + 1]), s2,
                                            make_float2(acc[c * GRP + j], acc[c * GRP + j + 1]));
                acc[c * GRP + j] = r.x;
                acc[c * GRP + j + 1] = r.y;
              }
            }
          }
        }
        if (ngr == 0) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[buf]);
        }
        if (colw) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[slot]);
          ++is;
        }
        ++au;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ra[q] = na[q];
        rw[q] = nw[q];
      }
      }
      // ------------------------------------------------------- output
      if (mrow && colv > 0) {
        const int nbase = U.n0 + col0;
#pragma unroll
        for (int c8 = 0; c8 < COLS / 8; ++c8) {
          const int n = nbase + c8 * 8;
          if (c8 * 8 >= colv) break;
          float vv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) vv[i] = acc[c8 * 8 + i];
          const bool full8 = (n + 8 <= p.N);
          if (p.splits > 1) {
            float* dstp = p.partial + (static_cast<int64_t>(U.split) * p.M + U.m0 + et) * p.N + n;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (n + i < p.N) dstp[i] = vv[i];
            continue;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (n + i < p.N) vv[i] += load_bias(p, n + i);
          const int64_t o = static_cast<int64_t>(U.m0 + et) * p.ldo + n;
          if (p.out_dtype == DT_BF16) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
            if (p.vec_ok && full8) {
              uint4 pk;
              __nv_bfloat162 t0 = __floats2bfloat162_rn(vv[0], vv[1]);
              __nv_bfloat162 t1 = __floats2bfloat162_rn(vv[2], vv[3]);
              __nv_bfloat162 t2 = __floats2bfloat162_rn(vv[4], vv[5]);
              __nv_bfloat162 t3 = __floats2bfloat162_rn(vv[6], vv[7]);
              pk.x = *reinterpret_cast<uint32_t*>(&t0);
              pk.y = *reinterpret_cast<uint32_t*>(&t1);
              pk.z = *reinterpret_cast<uint32_t*>(&t2);
              pk.w = *reinterpret_cast<uint32_t*>(&t3);
              *reinterpret_cast<uint4*>(dst) = pk;
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (n + i < p.N) dst[i] = __float2bfloat16_rn(vv[i]);
            }
          } else {
            float* dst = reinterpret_cast<float*>(p.out) + o;
            if (p.vec_ok && full8) {
              reinterpret_cast<float4*>(dst)[0] = make_float4(vv[0], vv[1], vv[2], vv[3]);
              reinterpret_cast<float4*>(dst)[1] = make_float4(vv[4], vv[5], vv[6], vv[7]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (n + i < p.N) dst[i] = vv[i];
            }
          }
        }
      }
    }
  epin_done:;
  } else if (warp >= 4) {
    // --------------------------------------------------------- epilogue
    const int g = (warp - 4) >> 2;                    // epilogue warpgroup
    const int et = (threadIdx.x - 128) & 127;         // TMEM lane 0..127
    const int col0 = g * COLS;                        // first token column of this WG
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* stg = sOut + g * (STG * 128);
    uint32_t au = 0, is = 0, eph = 0;
    uint32_t esl = 0;   // the CTA's slice count before this unit (issuer of a one-slice unit)
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit U = get_unit<EPI, BT>(p, u);
      const int colv = max(0, min(COLS, U.rows - col0));   // valid columns of this WG
      const int ngr = (colv + GRP - 1) / GRP;              // column groups with valid tokens
      float acc[COLS];
      float fscale = 1.f;
      float rowf = 1.f;   // MXH: the weight row's 2^(emax - 127)
      uint32_t buf0 = 0, buf1 = 0;   // whole-K kinds: the unit's accumulator pair
      uint32_t rd0 = 0;              // the pair's first buffer to read
      bool two = false;
      if (PROMOTE) {
#pragma unroll
        for (int j = 0; j < COLS; ++j) acc[j] = 0.f;
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          const uint32_t buf = au % NB;
          const int slot = is % SSL;
          if (!mbar_wait(&s_full[slot], (is / SSL) & 1, wc)) goto epi_done;
          if (!mbar_wait(&t_full[buf], (au / NB) & 1, wc)) goto epi_done;
          // F8Q: the slice's token-group scales come from the quantizer warps
          const int qsl = static_cast<int>(is % 8);
          if (KIND == KIND_F8Q)
            if (!mbar_wait(&qs_full[qsl], (is / 8) & 1, wc)) goto epi_done;
          tc_fence_after();
          const float* sc = sAsc + slot * BT + col0;
          const float* qsc = sQs + qsl * BT + col0;
          const float wr = lane_ws ? sWr[slot * 128 + et] : 1.f;
#pragma unroll
          for (int c = 0; c < COLS / GRP; ++c) {
            if (c < ngr) {
              float v[GRP];
              tmem_ld<GRP>(tmem_base + lane_addr + buf * L::BSTRIDE + col0 + c * GRP, v);
              if (c == COLS / GRP - 1 || c + 1 == ngr) {
                // the last TMEM read of this slice is done: hand the buffer
                // back to the MMA before doing the arithmetic
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&t_empty[buf]);
              }
              if (lane_ws) {
                const float2 w2 = make_float2(wr, wr);
#pragma unroll
                for (int j = 0; j < GRP; j += 2) {
                  const float2 p2 = __fmul2_rn(make_float2(v[j], v[j + 1]), w2);
                  v[j] = p2.x;
                  v[j + 1] = p2.y;
                }
              }
              // packed fp32 FMA: two accumulator elements per instruction
#pragma unroll
              for (int j = 0; j < GRP; j += 4) {
                float4 s4 = *reinterpret_cast<const float4*>(sc + c * GRP + j);
                if (KIND == KIND_F8Q) {
                  const float4 q4v = *reinterpret_cast<const float4*>(qsc + c * GRP + j);
                  s4 = make_float4(s4.x * q4v.x, s4.y * q4v.y, s4.z * q4v.z, s4.w * q4v.w);
                }
                float* a = acc + c * GRP + j;
                const float2 lo = __ffma2_rn(make_float2(v[j], v[j + 1]), make_float2(s4.x, s4.y),
                                             make_float2(a[0], a[1]));
                const float2 hi = __ffma2_rn(make_float2(v[j + 2], v[j + 3]), make_float2(s4.z, s4.w),
                                             make_float2(a[2], a[3]));
                a[0] = lo.x;
                a[1] = lo.y;
                a[2] = hi.x;
                a[3] = hi.y;
              }
            }
          }
          if (ngr == 0) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&t_empty[buf]);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&s_empty[slot]);
            if (KIND == KIND_F8Q) mbar_arrive(&qs_empty[qsl]);
          }
          ++au;
          ++is;
        }
      } else {
        if (p.block_n == 0 && p.w_scale != nullptr) fscale = __ldg(p.w_scale + U.e * p.sw_e);
        if (KIND == KIND_MXH) {
          int64_t grow = (EPI == EPI_SILU) ? static_cast<int64_t>(et < 64 ? U.wrow0 + et : U.wrow1 + (et - 64))
                                           : static_cast<int64_t>(U.wrow0) + et;
          if (grow >= p.mx_rows_total) grow = p.mx_rows_total - 1;
          const uint32_t em = __ldg(p.mx_emax + grow);
          rowf = __uint_as_float(em != 0 ? em << 23 : 0x00400000u);   // 2^(em - 127)
        }
        // the unit's two accumulators (one per MMA issuer); the second is
        // unwritten when the unit has a single K slice
        const uint32_t tb0 = 2 * au, tb1 = 2 * au + 1;
        buf0 = tb0 % NB;
        buf1 = tb1 % NB;
        two = U.kb1 - U.kb0 >= 2;
        if (!mbar_wait(&t_full[buf0], (tb0 / NB) & 1, wc)) goto epi_done;
        if (!mbar_wait(&t_full[buf1], (tb1 / NB) & 1, wc)) goto epi_done;
        tc_fence_after();
        // a one-slice unit's slice went to issuer (esl % 2); its buffer is the
        // one to read (the other is unwritten)
        rd0 = (!two && (esl & 1u)) ? buf1 : buf0;
        // the accumulators are read one staging chunk at a time below, so
        // no register array holds the tile's columns
        ++au;
        esl += static_cast<uint32_t>(U.kb1 - U.kb0);
      }
      // ------------------------------------------------------- output
      {
        float bias_g = 0.f, bias_u = 0.f;
        if (EPI == EPI_SILU) {
          const int l = et & 63;
          if (U.n0 + l < p.n_half && p.bias != nullptr) {
            bias_g = load_bias(p, U.e * p.bias_e + U.n0 + l);
            bias_u = load_bias(p, U.e * p.bias_e + p.n_half + U.n0 + l);
          }
        }
        const int nl = (et & 31) * 4;          // DENSE / SCATTER: 4 weight rows per thread
        const int n = U.n0 + nl;
        float b4[4] = {0.f, 0.f, 0.f, 0.f};
        if (EPI != EPI_SILU && p.splits == 1) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (n + i < p.N) b4[i] = load_bias(p, U.e * p.bias_e + n + i);
        }
#pragma unroll
        for (int c = 0; c < COLS / STG; ++c) {
          if (c * STG < colv) {
            if constexpr (PROMOTE) {
#pragma unroll
              for (int j = 0; j < STG; ++j) stg[j * 128 + et] = acc[c * STG + j] * fscale;
            } else {
              float v0[STG];
              tmem_ld<STG>(tmem_base + lane_addr + rd0 * L::BSTRIDE + col0 + c * STG, v0);
              if (two) {
                float v1[STG];
                tmem_ld<STG>(tmem_base + lane_addr + buf1 * L::BSTRIDE + col0 + c * STG, v1);
#pragma unroll
                for (int j = 0; j < STG; ++j) v0[j] += v1[j];
              }
              if (KIND == KIND_MXH) {
                // row factor 2^(emax - 127), column factor = the token row's
                // inverse pre-scale
#pragma unroll
                for (int j = 0; j < STG; ++j) {
                  const int col = col0 + c * STG + j;
                  const float cs = col < U.rows ? __ldg(p.a_scale + U.m0 + col) : 0.f;
                  stg[j * 128 + et] = v0[j] * (rowf * cs);
                }
              } else {
#pragma unroll
                for (int j = 0; j < STG; ++j) stg[j * 128 + et] = v0[j] * fscale;
              }
            }
            if (!group_sync(&epi_bar[g], eph, wc)) goto epi_done;
            if (EPI == EPI_DENSE) {
              for (int jj = et >> 5; jj < STG; jj += 4) {
                const int col = col0 + c * STG + jj;
                if (col >= U.rows) break;
                const int m = U.m0 + col;
                const float4 v = *reinterpret_cast<const float4*>(&stg[jj * 128 + nl]);
                float vv[4] = {v.x, v.y, v.z, v.w};
                if (p.splits > 1) {
                  float* dstp = p.partial + (static_cast<int64_t>(U.split) * p.M + m) * p.N;
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    if (n + i < p.N) dstp[n + i] = vv[i];
                } else {
#pragma unroll
                  for (int i = 0; i < 4; ++i) vv[i] += b4[i];
                  const int64_t o = U.e * p.out_e + static_cast<int64_t>(m) * p.ldo + n;
                  if (p.out_dtype == DT_BF16) {
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
                    if (p.vec_ok && n + 3 < p.N) {
                      __nv_bfloat162 lo = __floats2bfloat162_rn(vv[0], vv[1]);
                      __nv_bfloat162 hi = __floats2bfloat162_rn(vv[2], vv[3]);
                      uint2 pk;
                      pk.x = *reinterpret_cast<uint32_t*>(&lo);
                      pk.y = *reinterpret_cast<uint32_t*>(&hi);
                      *reinterpret_cast<uint2*>(dst) = pk;
                    } else {
#pragma unroll
                      for (int i = 0; i < 4; ++i)
                        if (n + i < p.N) dst[i] = __float2bfloat16_rn(vv[i]);
                    }
                  } else {
                    float* dst = reinterpret_cast<float*>(p.out) + o;
                    if (p.vec_ok && n + 3 < p.N) {
                      *reinterpret_cast<float4*>(dst) = make_float4(vv[0], vv[1], vv[2], vv[3]);
                    } else {
#pragma unroll
                      for (int i = 0; i < 4; ++i)
                        if (n + i < p.N) dst[i] = vv[i];
                    }
                  }
                }
              }
            } else if (EPI == EPI_SILU) {
              const int l = et & 63;
              const bool ok = U.n0 + l < p.n_half;
              for (int jj = et >> 6; jj < STG; jj += 2) {
                const int col = col0 + c * STG + jj;
                if (col >= U.rows) break;
                if (ok) {
                  if (p.h_out != nullptr) {
                    const int64_t hs = __ldg(p.sorted_ids + static_cast<int64_t>(U.blk) * p.block_m + col);
                    float* hr = p.h_out + hs * (2 * static_cast<int64_t>(p.n_half));
                    hr[U.n0 + l] = stg[jj * 128 + l];
                    hr[p.n_half + U.n0 + l] = stg[jj * 128 + 64 + l];
                  }
                  float gt = stg[jj * 128 + l] + bias_g;
                  float up = stg[jj * 128 + 64 + l] + bias_u;
                  float a;
                  if (p.act == 0) {
                    a = gt / (1.0f + expf(-gt)) * up;
                  } else {
                    // clamped SwiGLU: gate <= limit, |up| <= limit,
                    // gate * sigmoid(alpha * gate) * (up + 1)
                    gt = fminf(gt, p.act_limit);
                    up = fminf(fmaxf(up, -p.act_limit), p.act_limit);
                    a = gt / (1.0f + expf(-p.act_alpha * gt)) * (up + 1.0f);
                  }
                  reinterpret_cast<__nv_bfloat16*>(p.out)[static_cast<int64_t>(U.m0 + col) * p.ldo +
                                                          U.n0 + l] = __float2bfloat16_rn(a);
                }
              }
            } else {  // EPI_SCATTER
              for (int jj = et >> 5; jj < STG; jj += 4) {
                const int col = col0 + c * STG + jj;
                if (col >= U.rows) break;
                const int slot =
                    __ldg(p.sorted_ids + static_cast<int64_t>(U.blk) * p.block_m + col);
                const float rw = __ldg(p.route_w + slot);
                const float4 v = *reinterpret_cast<const float4*>(&stg[jj * 128 + nl]);
                const float vv[4] = {v.x, v.y, v.z, v.w};
                float* dst = reinterpret_cast<float*>(p.out) + static_cast<int64_t>(slot) * p.ldo;
                const bool v4 = p.vec_ok && n + 3 < p.N;
                if (v4) {
                  *reinterpret_cast<float4*>(dst + n) =
                      make_float4((vv[0] + b4[0]) * rw, (vv[1] + b4[1]) * rw, (vv[2] + b4[2]) * rw,
                                  (vv[3] + b4[3]) * rw);
                } else {
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    if (n + i < p.N) dst[n + i] = (vv[i] + b4[i]) * rw;
                }
                if (p.combine_cnt != nullptr) {
                  // the last of the token's topk slots to reach this tile
                  // sums them (release: fence before the count; acquire: fence
                  // after seeing the others' counts)
                  const int t = slot / p.topk;
                  __syncwarp();
                  int last = 0;
                  if (lane == 0) {
                    __threadfence();
                    last = atomicAdd(p.combine_cnt + static_cast<int64_t>(t) * p.tiles_n + U.tn, 1) ==
                           p.topk - 1;
                    if (last) __threadfence();
                  }
                  last = __shfl_sync(0xffffffffu, last, 0);
                  if (last) {
                    float s4[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int k = 0; k < p.topk; ++k) {
                      const float* yr = reinterpret_cast<const float*>(p.out) +
                                        (static_cast<int64_t>(t) * p.topk + k) * p.ldo;
                      if (v4) {
                        const float4 y4 = __ldcg(reinterpret_cast<const float4*>(yr + n));
                        s4[0] += y4.x;
                        s4[1] += y4.y;
                        s4[2] += y4.z;
                        s4[3] += y4.w;
                      } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                          if (n + i < p.N) s4[i] += __ldcg(yr + n + i);
                      }
                    }
                    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.combine_out) +
                                       static_cast<int64_t>(t) * p.combine_ldo;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      if (n + i < p.N) o[n + i] = __float2bfloat16_rn(s4[i]);
                  }
                }
              }
            }
            if (!group_sync(&epi_bar[g], eph, wc)) goto epi_done;
          }
        }
        if constexpr (!PROMOTE) {
          // every chunk of the accumulator pair has been read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&t_empty[buf0]);
            mbar_arrive(&t_empty[buf1]);
          }
        }
      }
    }
  epi_done:;
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace mxq
