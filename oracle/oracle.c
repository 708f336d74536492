/*
 * oracle.c — plain, slow, obviously-correct CPU reference for the quantized
 * scaled-GEMM / fused-MoE hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: every format is decoded
 * here from its bit pattern, every accumulation runs in fp64, and the only
 * parallelism is an OpenMP loop over independent outputs (used for timing).
 *
 * Sources (page title, section):
 *   [vLLM-50949]  "[CPU] routed FP8/MXFP4 MoE: per-expert-block BRGEMM vs
 *                 TinyGEMM dispatch" — implementation breakdown and the
 *                 stage-1 tile loop excerpt of moe_fp8.cpp.
 *   [SGL-32618]   "[CPU] fp8_per_tensor_scaled_mm_cpu" — implementation
 *                 breakdown; test_fp8_per_tensor_gemm excerpt (reference =
 *                 dequantised fp32 matmul times the scale, plus bias).
 *   [SGL-35605]   "[XPU] block-FP8 linear via torch scaled_mm" — the
 *                 torch_w8a8_block_fp8_linear excerpt (block_size rules,
 *                 per_token_group_quant_fp8, BlockWise1x128 activations,
 *                 BlockWise128x128 / 1x128 weights) and the numerical test
 *                 (reference_block_fp8_matmul = dequantise, then matmul).
 *
 * Readings where the pages are silent:
 *   - group scale s = max(amax, eps) / 448 in fp32 with IEEE division, and
 *     q = e4m3_rne(clamp(x / s, -448, 448)) with IEEE fp32 division;
 *   - e4m3 encode = nearest finite code, ties to the even code, sign kept
 *     (so -0 and tiny negatives give 0x80);
 *   - block scales multiply the exact partial sum of each 128-wide K slice;
 *     a per-tensor scale with no activation scales multiplies the full sum;
 *   - results are rounded once to fp32, then to bf16 by round-to-nearest-even;
 *   - fused MoE: gate = first N rows of w1, act = bf16(silu(gate) * up),
 *     b1 before the activation, b2 before the routing weight, top-k sum in
 *     ascending k; MXFP4 low nibble = even K index, one ue8m0 per 32 K;
 *   - moe_align: stable (ascending slot) order inside each expert, experts
 *     ascending, blocks of block_m, padding value S, offsets = compact prefix
 *     sum of block sizes, expert_ids = -1 and offsets = S past the end.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoders */

/* float8_e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa; no infinities;
 * S.1111.111 is NaN.  Subnormals (E = 0) are m * 2^-9. */
double oracle_e4m3_decode(uint8_t b) {
  int s = (b >> 7) & 1;
  int E = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (E == 15 && m == 7) return NAN;
  if (E == 0)
    v = (double)m * ldexp(1.0, -9);
  else
    v = (1.0 + (double)m / 8.0) * ldexp(1.0, E - 7);
  return s ? -v : v;
}

/* FP4 e2m1 (OCP MX): 1 sign, 2 exponent (bias 1), 1 mantissa.
 * Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
double oracle_e2m1_decode(uint8_t nib) {
  int s = (nib >> 3) & 1;
  int E = (nib >> 1) & 3;
  int m = nib & 1;
  double v;
  if (E == 0)
    v = (double)m * 0.5;
  else
    v = (1.0 + (double)m / 2.0) * ldexp(1.0, E - 1);
  return s ? -v : v;
}

/* ue8m0 (OCP MX scale): 2^(e - 127); e = 255 is NaN. */
double oracle_ue8m0_decode(uint8_t e) {
  if (e == 255) return NAN;
  return ldexp(1.0, (int)e - 127);
}

/* bf16 is the top half of an IEEE binary32. */
double oracle_bf16_decode(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double f32_bits_value(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* fp32 -> bf16, round to nearest, ties to even, by comparing the two
 * candidates that bracket the value. */
uint16_t oracle_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t sign = u & 0x80000000u;
  uint32_t mag = u & 0x7FFFFFFFu;
  uint32_t lo = mag & 0xFFFF0000u;          /* toward zero */
  uint32_t hi = lo + 0x10000u;              /* next bf16 magnitude */
  if (lo == mag) return (uint16_t)((sign | lo) >> 16);
  double x = fabs((double)f);
  double vlo = f32_bits_value(lo);
  /* hi may be the infinity pattern: its "value" for rounding is 2^128 */
  double vhi = (hi >= 0x7F800000u) ? ldexp(1.0, 128) : f32_bits_value(hi);
  uint32_t pick;
  if (x - vlo < vhi - x)
    pick = lo;
  else if (x - vlo > vhi - x)
    pick = hi;
  else
    pick = ((lo >> 16) & 1u) ? hi : lo;     /* tie: even bf16 mantissa */
  if (pick >= 0x7F800000u) pick = 0x7F800000u;
  return (uint16_t)((sign | pick) >> 16);
}

/* The final rounding used for every bf16 output: fp64 -> fp32 (C cast,
 * round to nearest even) -> bf16 (round to nearest even). */
uint16_t oracle_bf16_round(double v) { return oracle_bf16_from_f32((float)v); }

/* ---------------------------------------------------------------- encoder */

/* Finite non-negative e4m3 codes 0x00..0x7E are strictly increasing in
 * value; 0x7F is NaN.  Encode = nearest code, ties to the even code. */
static double e4m3_pos_table[127];
static int e4m3_table_ready = 0;

static void e4m3_table_init(void) {
  if (e4m3_table_ready) return;
  for (int c = 0; c < 127; ++c) e4m3_pos_table[c] = oracle_e4m3_decode((uint8_t)c);
  e4m3_table_ready = 1;
}

/* Nearest finite e4m3 code to v (|v| <= 448 expected; larger magnitudes
 * saturate to 448).  Negative inputs (including -0) keep the sign bit. */
uint8_t oracle_e4m3_encode(float v) {
  e4m3_table_init();
  if (isnan(v)) return 0x7F;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs((double)v);
  int best;
  if (a >= e4m3_pos_table[126]) {
    best = 126;
  } else {
    /* largest code c with table[c] <= a (binary search) */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
      int mid = (lo + hi) / 2;
      if (e4m3_pos_table[mid] <= a) lo = mid; else hi = mid;
    }
    if (e4m3_pos_table[lo] == a) {
      best = lo;
    } else {
      double dlo = a - e4m3_pos_table[lo];
      double dhi = e4m3_pos_table[lo + 1] - a;
      if (dlo < dhi) best = lo;
      else if (dhi < dlo) best = lo + 1;
      else best = (lo % 2 == 0) ? lo : lo + 1;  /* tie: even mantissa LSB */
    }
  }
  return (uint8_t)(best | (neg ? 0x80 : 0));
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------- per-token group quant */

/* [SGL-35605] per_token_group_quant_fp8(input_2d, block_k): one fp32 scale
 * per row and per group of `group` consecutive K elements, scale shape
 * [M, ceil(K/group)] row-major; q has the shape of x, row stride K. */
void oracle_per_token_group_quant_fp8(const uint16_t* x, int64_t M, int64_t K,
                                      int64_t ldx, int32_t group, float eps,
                                      uint8_t* q, float* scales) {
  int64_t G = (K + group - 1) / group;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      int64_t k0 = g * group;
      int64_t k1 = k0 + group < K ? k0 + group : K;
      float amax = 0.0f;
      for (int64_t k = k0; k < k1; ++k) {
        float a = fabsf((float)oracle_bf16_decode(x[m * ldx + k]));
        if (a > amax) amax = a;
      }
      float s = (amax > eps ? amax : eps) / 448.0f;   /* IEEE fp32 division */
      scales[m * G + g] = s;
      for (int64_t k = k0; k < k1; ++k) {
        float xv = (float)oracle_bf16_decode(x[m * ldx + k]);
        float t = xv / s;                               /* IEEE fp32 division */
        if (t > 448.0f) t = 448.0f;
        if (t < -448.0f) t = -448.0f;
        q[m * K + k] = oracle_e4m3_encode(t);
      }
    }
  }
}

/* ------------------------------------------------------------ scaled mm */

enum { OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3 };

static double load_a(const void* A, int a_dtype, int64_t idx) {
  if (a_dtype == OR_E4M3) return oracle_e4m3_decode(((const uint8_t*)A)[idx]);
  return oracle_bf16_decode(((const uint16_t*)A)[idx]);
}

static double load_bias(const void* bias, int bias_dtype, int64_t n) {
  if (!bias) return 0.0;
  if (bias_dtype == OR_BF16) return oracle_bf16_decode(((const uint16_t*)bias)[n]);
  return (double)((const float*)bias)[n];
}

/* The exact scaled accumulator of one output element.
 *
 *   block mode (block_k = 128):
 *     acc = sum_kb  As[m,kb] * Ws[n / block_n, kb] * sum_{k in kb} a[m,k] w[n,k]
 *   per-tensor mode (block_n = block_k = 0, w_scale = one fp32):
 *     with activation group scales:  sum_kb As[m,kb] * s * partial_kb
 *     without (W8A16):               s * sum_k a[m,k] w[n,k]
 *   then + bias[n].
 * This is [SGL-35605] reference_block_fp8_matmul and [SGL-32618]'s
 * matmul(data.float(), weight.float().T) * scale + bias, in exact arithmetic
 * up to fp64 rounding. */
static double scaled_mm_one(const void* A, int a_dtype, int64_t K, int64_t lda,
                            const float* a_scale, int64_t sa0, int64_t sa1,
                            const uint8_t* W, int64_t ldw, const float* w_scale,
                            int32_t block_n, int32_t block_k, int64_t sw0,
                            int64_t sw1, const void* bias, int32_t bias_dtype,
                            int64_t m, int64_t n) {
  const int64_t slice = 128;
  double acc = 0.0;
  if (block_k == 0 && a_scale == NULL) {
    double sum = 0.0;
    for (int64_t k = 0; k < K; ++k)
      sum += load_a(A, a_dtype, m * lda + k) * oracle_e4m3_decode(W[n * ldw + k]);
    acc = (double)w_scale[0] * sum;
  } else {
    int64_t nkb = (K + slice - 1) / slice;
    for (int64_t kb = 0; kb < nkb; ++kb) {
      double part = 0.0;
      int64_t k1 = (kb + 1) * slice < K ? (kb + 1) * slice : K;
      for (int64_t k = kb * slice; k < k1; ++k)
        part += load_a(A, a_dtype, m * lda + k) * oracle_e4m3_decode(W[n * ldw + k]);
      double as = a_scale ? (double)a_scale[m * sa0 + kb * sa1] : 1.0;
      double ws;
      if (block_k == 0)
        ws = (double)w_scale[0];
      else
        ws = (double)w_scale[(n / block_n) * sw0 + kb * sw1];
      acc += as * ws * part;
    }
  }
  return acc + load_bias(bias, bias_dtype, n);
}

/* Full output.  out_f32 (nullable) = (float)acc, out_bf16 (nullable) =
 * bf16_rne((float)acc); both [M, N] with row stride ldo. */
void oracle_scaled_mm(const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
                      const float* a_scale, int64_t sa0, int64_t sa1,
                      const uint8_t* W, int64_t N, int64_t ldw,
                      const float* w_scale, int32_t block_n, int32_t block_k,
                      int64_t sw0, int64_t sw1, const void* bias, int32_t bias_dtype,
                      float* out_f32, uint16_t* out_bf16, int64_t ldo) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = scaled_mm_one(A, a_dtype, K, lda, a_scale, sa0, sa1, W, ldw, w_scale,
                                 block_n, block_k, sw0, sw1, bias, bias_dtype, m, n);
      if (out_f32) out_f32[m * ldo + n] = (float)acc;
      if (out_bf16) out_bf16[m * ldo + n] = oracle_bf16_round(acc);
    }
  }
}

/* The same accumulator at listed (m, n) pairs only (fp64, before rounding),
 * for sampled checks at sizes where the full output would take too long. */
void oracle_scaled_mm_at(const void* A, int32_t a_dtype, int64_t K, int64_t lda,
                         const float* a_scale, int64_t sa0, int64_t sa1,
                         const uint8_t* W, int64_t ldw, const float* w_scale,
                         int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
                         const void* bias, int32_t bias_dtype, const int64_t* ms,
                         const int64_t* ns, int64_t count, double* acc_out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    acc_out[i] = scaled_mm_one(A, a_dtype, K, lda, a_scale, sa0, sa1, W, ldw, w_scale,
                               block_n, block_k, sw0, sw1, bias, bias_dtype, ms[i], ns[i]);
}

/* ------------------------------------------------------------- moe_align */

/* [vLLM-50949] stage-1 excerpt consumes sorted_ids / expert_ids / offsets:
 * block mb holds expert expert_ids[mb], its rows are slots
 * sorted_ids[mb*block_m + m] for m < offsets[mb+1] - offsets[mb], and the
 * token of a slot is slot / topk.  Produced here by its plain definition.
 * Returns 0, or -1 if cap is too small, or -2 if an id is outside [0, E). */
int32_t oracle_moe_align(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                         int32_t block_m, int32_t* sorted_ids, int32_t* expert_ids,
                         int32_t* offsets, int32_t* num_blocks, int64_t cap) {
  int64_t S = T * (int64_t)topk;
  for (int64_t i = 0; i < S; ++i)
    if (topk_ids[i] < 0 || topk_ids[i] >= E) return -2;
  for (int64_t i = 0; i < cap * block_m; ++i) sorted_ids[i] = (int32_t)S;
  for (int64_t b = 0; b < cap; ++b) expert_ids[b] = -1;
  for (int64_t b = 0; b <= cap; ++b) offsets[b] = (int32_t)S;
  int64_t b = 0;       /* next block */
  int64_t pos = 0;     /* compact row of the next slot */
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    int64_t j = 0;     /* rank of the slot inside expert e */
    for (int64_t slot = 0; slot < S; ++slot) {
      if (topk_ids[slot] != e) continue;
      if (j % block_m == 0) {
        if (b >= cap) return -1;
        expert_ids[b] = e;
        offsets[b] = (int32_t)pos;
        ++b;
      }
      sorted_ids[(b - 1) * block_m + (j % block_m)] = (int32_t)slot;
      ++j;
      ++pos;
      offsets[b] = (int32_t)pos;
    }
  }
  *num_blocks = (int32_t)b;
  return 0;
}

/* ------------------------------------------------------------ fused MoE */

enum { OR_W_FP8_BLOCK128 = 1, OR_W_MXFP4 = 2 };

/* Weight element (row r, column k) of expert e of a [E, R, C] matrix in
 * either format, with its scale folded in only for MXFP4 (where the scale
 * belongs to each element); FP8-block scales multiply slice partials. */
static double w_elem(int32_t wtype, const void* w, int64_t e, int64_t R, int64_t C,
                     int64_t r, int64_t k, const void* ws) {
  if (wtype == OR_W_MXFP4) {
    const uint8_t* p = (const uint8_t*)w;
    uint8_t byte = p[(e * R + r) * (C / 2) + k / 2];
    uint8_t nib = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
    const uint8_t* s = (const uint8_t*)ws;
    return oracle_e2m1_decode(nib) * oracle_ue8m0_decode(s[(e * R + r) * (C / 32) + k / 32]);
  }
  return oracle_e4m3_decode(((const uint8_t*)w)[(e * R + r) * C + k]);
}

/* y[r] = sum_k a[k] * W[e][r][k] with the format's scales, in fp64.
 * FP8 block: scale Ws[e][r/128][kb] per 128x128 block, applied to each
 * 128-wide K slice partial. */
static double expert_row_dot(int32_t wtype, const void* w, const void* ws, int64_t e,
                             int64_t R, int64_t C, int64_t r, const double* a) {
  if (wtype == OR_W_MXFP4) {
    double sum = 0.0;
    for (int64_t k = 0; k < C; ++k) sum += a[k] * w_elem(wtype, w, e, R, C, r, k, ws);
    return sum;
  }
  int64_t nrb = (R + 127) / 128, nkb = (C + 127) / 128;
  const float* s = (const float*)ws;
  double acc = 0.0;
  for (int64_t kb = 0; kb < nkb; ++kb) {
    double part = 0.0;
    int64_t k1 = (kb + 1) * 128 < C ? (kb + 1) * 128 : C;
    for (int64_t k = kb * 128; k < k1; ++k) part += a[k] * w_elem(wtype, w, e, R, C, r, k, ws);
    acc += (double)s[(e * nrb + r / 128) * nkb + kb] * part;
  }
  return acc;
}

/* One expert GEMM of the fused MoE without its bias, the stage accumulators
 * of [vLLM-50949] (stage 1: hidden . W1[e]^T; stage 2: act . W2[e]^T):
 *   out[m, r] = sum_k x[m, k] * W[e][r][k]   (format scales as above, fp64)
 * x bf16 [M, C] row stride ldx; W [E, R, C] in either format; out fp64
 * [M, R].  Used to check a GPU stage accumulator on the GPU's own inputs. */
void oracle_expert_linear(const uint16_t* x, int64_t M, int64_t ldx, int32_t wtype,
                          const void* w, const void* ws, int64_t e, int64_t R, int64_t C,
                          double* out) {
  double* a = (double*)malloc(sizeof(double) * (M * C > 0 ? M * C : 1));
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < C; ++k) a[m * C + k] = oracle_bf16_decode(x[m * ldx + k]);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < M * R; ++i)
    out[i] = expert_row_dot(wtype, w, ws, e, R, C, i % R, a + (i / R) * C);
  free(a);
}

/* Routed fused MoE of [vLLM-50949] (stage 1 hidden @ w1, activation,
 * stage 2 @ w2) followed by the top-k weighted combine:
 *   for each slot (t, k), e = topk_ids[t,k]:
 *     h   = x[t] . W1[e]^T (+ b1[e])                       [2N]
 *     act = bf16( silu(h[:N]) * h[N:] )                      [N]
 *     z   = act . W2[e]^T (+ b2[e])                          [K]
 *   out[t] = bf16( sum_k topk_weights[t,k] * z_(t,k) )      ascending k
 * Shapes: hidden bf16 [T, K] row stride ldh; w1 [E, 2N, K] (e4m3, scales
 * fp32 [E, ceil(2N/128), ceil(K/128)]) or [E, 2N, K/2] packed e2m1 with
 * ue8m0 [E, 2N, K/32]; w2 [E, K, N] / [E, K, N/2] likewise; b1 [E, 2N],
 * b2 [E, K] fp32 or NULL; out bf16 [T, K] row stride ldo.  act_out (bf16
 * [T*topk, N]) and z_out (fp64 [T*topk, K]) are optional checkpoints in
 * slot order.  Returns -2 if an id is out of range. */
/* The stage-1 activation of the fused MoE on one pair (gate g, up u):
 *   kind 0, SiLU-and-mul ([vLLM-50949] "activation" between the stages):
 *       silu(g) * u with silu(v) = v / (1 + e^-v)
 *   kind 1, GPT-OSS-style clamped SwiGLU (GPT-OSS is among the MXFP4 models
 *       [vLLM-50949] serves): g' = min(g, limit), u' = clamp(u, -limit, limit),
 *       g' / (1 + e^(-alpha g')) * (u' + 1)
 * evaluated in fp64. */
static double moe_activation(int32_t kind, double alpha, double limit, double g, double u) {
  if (kind == 1) {
    if (g > limit) g = limit;
    if (u > limit) u = limit;
    if (u < -limit) u = -limit;
    return g / (1.0 + exp(-alpha * g)) * (u + 1.0);
  }
  return g / (1.0 + exp(-g)) * u;
}

int32_t oracle_fused_experts_act(const uint16_t* hidden, int64_t T, int64_t K, int64_t ldh,
                                 int32_t wtype, int32_t E, int64_t N,
                                 const void* w1, const void* w1_scale, const float* b1,
                                 const void* w2, const void* w2_scale, const float* b2,
                                 const float* topk_weights, const int32_t* topk_ids,
                                 int32_t topk, int32_t act_kind, double alpha, double limit,
                                 uint16_t* out, int64_t ldo, uint16_t* act_out, double* z_out) {
  for (int64_t i = 0; i < T * topk; ++i)
    if (topk_ids[i] < 0 || topk_ids[i] >= E) return -2;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* x = (double*)malloc(sizeof(double) * K);
    double* h = (double*)malloc(sizeof(double) * 2 * N);
    double* act = (double*)malloc(sizeof(double) * N);
    double* z = (double*)malloc(sizeof(double) * K);
    double* o = (double*)calloc(K, sizeof(double));
    for (int64_t k = 0; k < K; ++k) x[k] = oracle_bf16_decode(hidden[t * ldh + k]);
    for (int32_t j = 0; j < topk; ++j) {
      int64_t slot = t * topk + j;
      int64_t e = topk_ids[slot];
      for (int64_t r = 0; r < 2 * N; ++r) {
        h[r] = expert_row_dot(wtype, w1, w1_scale, e, 2 * N, K, r, x);
        if (b1) h[r] += (double)b1[e * 2 * N + r];
      }
      for (int64_t i = 0; i < N; ++i) {
        uint16_t a16 = oracle_bf16_round(moe_activation(act_kind, alpha, limit, h[i], h[N + i]));
        act[i] = oracle_bf16_decode(a16);
        if (act_out) act_out[slot * N + i] = a16;
      }
      for (int64_t r = 0; r < K; ++r) {
        z[r] = expert_row_dot(wtype, w2, w2_scale, e, K, N, r, act);
        if (b2) z[r] += (double)b2[e * K + r];
        if (z_out) z_out[slot * K + r] = z[r];
        o[r] += (double)topk_weights[slot] * z[r];
      }
    }
    for (int64_t r = 0; r < K; ++r) out[t * ldo + r] = oracle_bf16_round(o[r]);
    free(x); free(h); free(act); free(z); free(o);
  }
  return 0;
}

/* The fused MoE with the SiLU-and-mul activation. */
int32_t oracle_fused_experts(const uint16_t* hidden, int64_t T, int64_t K, int64_t ldh,
                             int32_t wtype, int32_t E, int64_t N,
                             const void* w1, const void* w1_scale, const float* b1,
                             const void* w2, const void* w2_scale, const float* b2,
                             const float* topk_weights, const int32_t* topk_ids,
                             int32_t topk, uint16_t* out, int64_t ldo,
                             uint16_t* act_out, double* z_out) {
  return oracle_fused_experts_act(hidden, T, K, ldh, wtype, E, N, w1, w1_scale, b1, w2, w2_scale,
                                  b2, topk_weights, topk_ids, topk, 0, 0.0, 0.0, out, ldo,
                                  act_out, z_out);
}

/* ------------------------------------------------------ MXFP4 quantizer */

/* Conversion of fp32 values to MXFP4 by the OCP Microscaling (MX) v1.0 rule,
 * the format of the MXFP4 expert weights of [vLLM-50949] (its related PR
 * 49347 quantizes weights to MXFP4 online).  Per block of 32 consecutive
 * values of a row:
 *   E = floor(log2(max |v|)) - 2  (2 = largest exponent of E2M1), clamped to
 *       [-127, 127]; an all-zero block takes E = -127;
 *   scale byte = E + 127 (ue8m0, value 2^E);
 *   each element = the E2M1 value nearest to v / 2^E (searched over the 8
 *       magnitudes), ties to the code with an even last bit, magnitudes above
 *       6 saturated to 6; the sign bit copies the sign of v, so negative
 *       values that round to zero give -0 (code 8).
 * x fp32 [R, C] row stride ldx, C a multiple of 32; packed [R, C/2] (low
 * nibble = even column); scales [R, C/32]. */
void oracle_mxfp4_quantize(const float* x, int64_t R, int64_t C, int64_t ldx, uint8_t* packed,
                           uint8_t* scales) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t g = 0; g < C / 32; ++g) {
      const float* v = x + r * ldx + g * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i)
        if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
      int E = -127;
      if (amax > 0.0) {
        int e2;
        (void)frexp(amax, &e2);  /* amax = f * 2^e2 with f in [0.5, 1) */
        E = (e2 - 1) - 2;
        if (E < -127) E = -127;
        if (E > 127) E = 127;
      }
      scales[r * (C / 32) + g] = (uint8_t)(E + 127);
      for (int i = 0; i < 32; ++i) {
        double t = ldexp((double)v[i], -E);
        double a = fabs(t);
        int best = 7;
        if (a < 6.0) {
          best = 0;
          for (int c = 1; c < 8; ++c) {
            double dc = fabs(a - mag[c]), db = fabs(a - mag[best]);
            if (dc < db || (dc == db && (c & 1) == 0)) best = c;
          }
        }
        uint8_t nib = (uint8_t)best;
        if (signbit(t)) nib |= 8;
        int64_t col = g * 32 + i;
        uint8_t* dst = packed + r * (C / 2) + col / 2;
        if (col % 2 == 0)
          *dst = (uint8_t)((*dst & 0xF0) | nib);
        else
          *dst = (uint8_t)((*dst & 0x0F) | (nib << 4));
      }
    }
  }
}

/* ------------------------------------------------------------- threading */

int32_t oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int32_t n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
