/*
 * mxq.h — C ABI of libmxq: weight-quantized scaled GEMM and routed fused MoE
 * on one NVIDIA GB300 (sm_103a).
 *
 * Conventions (all entry points):
 *   - The caller owns all memory.  Tensor arguments are DEVICE pointers on the
 *     current CUDA device unless stated otherwise.  Scratch comes from a
 *     caller-provided device workspace sized by the matching *_workspace_size
 *     query; the library never calls cudaMalloc/cudaFree.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns an mxq_status.
 *   - Arguments are validated on the host before anything is launched; on an
 *     error nothing is launched, outputs are untouched, and
 *     mxq_last_error() (thread-local) describes the problem.
 *   - Problems detected on the device (an expert id outside [0, E), a bounded
 *     wait that expired) set a device status word that mxq_sync_status reads.
 *   - The device must be compute capability 10.3 (GB300, sm_103a); any other
 *     device gives MXQ_ERR_UNSUPPORTED.
 *   - Row strides (ld*) are in elements.  Operands read by the tensor-memory
 *     accelerator (A, W, hidden, expert weights) need a 16-byte aligned base
 *     and a row stride that is a multiple of 16 bytes, else
 *     MXQ_ERR_UNSUPPORTED.
 *
 * Page references are "title, section" of the pages this library follows:
 *   [CPU-MoE]  vLLM PR 50949 "[CPU] routed FP8/MXFP4 MoE: per-expert-block
 *              BRGEMM vs TinyGEMM dispatch"
 *   [CPU-GEMM] SGLang PR 32618 "[CPU] fp8_per_tensor_scaled_mm_cpu"
 *   [XPU-FP8]  SGLang PR 35605 "[XPU] block-FP8 linear via torch scaled_mm"
 */
#ifndef MXQ_H_
#define MXQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mxq_status;
typedef void* mxq_stream_t; /* a cudaStream_t */

enum {
  MXQ_OK = 0,
  MXQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride, ... */
  MXQ_ERR_UNSUPPORTED = 2, /* wrong device, block size, dtype combination, alignment */
  MXQ_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
  MXQ_ERR_TIMEOUT = 4,     /* a bounded device wait expired (mxq_sync_status) */
  MXQ_ERR_DEVICE = 5       /* device-detected bad input, e.g. expert id out of range */
};

/* dtype tags */
enum {
  MXQ_BF16 = 1,
  MXQ_F32 = 2,
  MXQ_E4M3 = 3,   /* float8_e4m3fn, one byte */
  MXQ_E2M1X2 = 4, /* two FP4 e2m1 codes per byte, low nibble = even index */
  MXQ_UE8M0 = 5   /* one byte, value 2^(e-127) */
};

/* expert weight formats of mxq_fused_experts */
enum {
  MXQ_W_FP8_BLOCK128 = 1, /* e4m3 weights, fp32 scale per [128, 128] block */
  MXQ_W_MXFP4 = 2         /* e2m1x2 weights, ue8m0 scale per 32 K elements */
};

/* stage-1 activations of the fused MoE (gate = rows [0, N) of w1[e], up =
 * rows [N, 2N)) */
enum {
  MXQ_ACT_SILU = 0,         /* act = silu(gate) * up, silu(v) = v / (1 + e^-v) */
  MXQ_ACT_SWIGLU_CLAMP = 1  /* GPT-OSS-style clamped SwiGLU:
                               g = min(gate, limit), u = clamp(up, -limit, limit),
                               act = g / (1 + e^(-alpha g)) * (u + 1) */
};

/* options (process-wide; mxq_set_option / mxq_get_option) */
enum {
  MXQ_OPT_SMALL_M_MAX = 1,  /* expert blocks with m_size <= this use the narrowest MMA
                               instruction covering them; larger blocks use the full
                               block_m width.  Default 4, the [CPU-MoE] page's small-block
                               threshold (its tests put 4 on the small path, 5 and 33 on
                               the large one). */
  MXQ_OPT_FORCE_PATH = 2,   /* 0 per expert block (auto), 1 always narrow (fit), 2 always
                               full width, 3 one path for the whole layer: narrow when
                               max(1, S / E) <= SMALL_M_MAX (the global crossover) */
  MXQ_OPT_WAIT_BUDGET_NS = 3, /* limit of every device-side wait, default 2e9 ns */
  MXQ_OPT_SPLIT_K = 4,      /* fp8_scaled_mm split-K: 0 auto, else the factor */
  MXQ_OPT_INJECT_STALL = 5, /* TEST ONLY: GEMM producers issue no copy, so every
                               consumer wait runs out (exercises MXQ_ERR_TIMEOUT) */
  MXQ_OPT_NUM_SMS = 6,      /* persistent grid size cap; 0 = all SMs */
  MXQ_OPT_TILE_N = 7,       /* fp8_scaled_mm token-tile width: 0 auto, or 32, 64, 128,
                               256 (256 for FP8 activations only) */
  MXQ_OPT_NORMAL_TILE = 8,  /* fp8_scaled_mm weight-tile width when the tokens sit on
                               the MMA M side (large-M W8A8): 0 auto, 128, 192 or 256 */
  MXQ_OPT_PDL = 9,          /* 1 (default): kernels are launched with programmatic stream
                               serialization, so a kernel's launch and prologue overlap the
                               end of the previous kernel on the stream (each waits for it
                               before touching global memory); 0: plain stream order */
  MXQ_OPT_FUSE_COMBINE = 10, /* fused MoE: 1 the top-k combine runs inside the stage-2
                               GEMM (the last of a token's slots to finish a weight tile sums
                               its rows, ascending k); 0 (default, measured faster on GB300):
                               a separate combine kernel.  Bit-identical results either way. */
  MXQ_OPT_MOE_F16 = 11,     /* fused MoE operand type: 3 (default) f16 for FP8-block
                               experts, and for MXFP4 when T * topk > 16 (below, the f16
                               path's extra launches cost more than its decode saves);
                               2 f16 for both formats; 1 f16 for FP8-block experts, bf16
                               for MXFP4; 0 bf16 for both.  With f16 the
                               expert GEMMs multiply f16 operands:
                               weights decode to f16 in one conversion per pair (MXFP4
                               groups scaled by 2^(e - emax of their weight row), the row's
                               2^(emax-127) applied in fp32 by the epilogue), and token
                               rows are converted to f16 after a power-of-two row scaling
                               that the epilogue undoes; 0: bf16 operands (weights decoded
                               to bf16, tokens as given).  The f16 operands are exact
                               except for elements more than ~2^31 below their token row's
                               maximum and MXFP4 groups more than 2^23 below the largest
                               group scale of their row. */
  MXQ_OPT_FUSE_QUANT = 12   /* mxq_w8a8_block_fp8_linear: 1 up to 32 token rows the activation
                               quantization runs inside the GEMM; 0 (default, measured faster
                               on GB300: the in-kernel IEEE divisions of four quantizer warps
                               are latency-bound) a separate quantization kernel first.
                               Bit-identical results. */
};

const char* mxq_last_error(void);
const char* mxq_version(void);
mxq_status mxq_set_option(int32_t option, int64_t value);
mxq_status mxq_get_option(int32_t option, int64_t* value);

/* Synchronizes `stream`, then reads and clears the device status word of the
 * current device: MXQ_OK, MXQ_ERR_TIMEOUT or MXQ_ERR_DEVICE. */
mxq_status mxq_sync_status(mxq_stream_t stream);

/*
 * Per-token-group FP8 quantization of activations ([XPU-FP8], key code
 * excerpts: per_token_group_quant_fp8(input_2d, block_k) producing the
 * BlockWise1x128 activation operand and its [M, K/128] scale).
 * For every row m and group g of `group` consecutive K elements:
 *     s[m, g] = max(amax_g, eps) / 448          (fp32, IEEE division)
 *     q[m, k] = e4m3_rne(clamp(x[m, k] / s, -448, 448))  (IEEE division)
 *   x       bf16 [M, K], row stride ldx (>= K), inner stride 1
 *   q       e4m3 [M, K], row stride K (written)
 *   scales  fp32 [M, ceil(K/group)] row-major (written); a ragged last group
 *           uses its own amax
 *   group   multiple of 8, 8..1024 (the pages use 128); eps > 0
 * M == 0 is a no-op.
 */
mxq_status mxq_per_token_group_quant_fp8(const void* x, int64_t M, int64_t K, int64_t ldx,
                                         int32_t group, float eps, void* q, float* scales,
                                         mxq_stream_t stream);

/*
 * Weight quantization to MXFP4 (the expert-weight format of [CPU-MoE]; its
 * related-PR list names online MXFP4 quantization of the weights), by the OCP
 * Microscaling (MX) v1.0 rule.  For every block of 32 consecutive values of a
 * row:
 *   E = floor(log2(max |v|)) - 2, clamped to [-127, 127]; -127 when all zero
 *   scales[r, g] = E + 127                      (ue8m0, value 2^E)
 *   code = E2M1 nearest to v / 2^E, ties to the even code, |.| > 6 -> 6;
 *          the sign bit is the sign of v (negatives rounding to 0 give -0)
 *   x       [R, C] MXQ_BF16 or MXQ_F32, row stride ldx; C a multiple of 32
 *   packed  e2m1x2 [R, C/2] (low nibble = even column), 16-byte aligned
 *   scales  ue8m0 [R, C/32]
 * R == 0 is a no-op.
 */
mxq_status mxq_quantize_mxfp4(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                              void* packed, void* scales, mxq_stream_t stream);

/*
 * Scaled FP8 GEMM  out[m, n] = sum_k A[m, k] * W[n, k] * scales (+ bias[n]).
 * W8A8 block mode ([XPU-FP8], torch_w8a8_block_fp8_linear excerpt):
 *   a_dtype = MXQ_E4M3, a_scale fp32 [M, ceil(K/128)] (strides sa0, sa1),
 *   w_scale fp32 [ceil(N/block_n), ceil(K/128)] (strides sw0, sw1, any
 *   layout, e.g. the transposed-contiguous storage of the load-time relayout),
 *   block_n in {1, 128}, block_k = 128:
 *     out = sum_kb As[m,kb] * Ws[n/block_n, kb] * sum_{k in kb} qA[m,k] W[n,k]
 * W8A16 per-tensor mode ([CPU-GEMM], implementation breakdown: the per-tensor
 *   scale is the block-scale case with every block equal):
 *   a_dtype = MXQ_BF16, a_scale = NULL, w_scale = one fp32 (0-d or [1]),
 *   block_n = block_k = 0:   out = (A . W^T) * s
 * W8A16 with block weights (a_dtype = MXQ_BF16, a_scale = NULL, block scales)
 * and W8A8 with a per-tensor weight scale are also accepted.
 *   A      [M, K] e4m3 or bf16, row stride lda
 *   W      e4m3 [N, K], row stride ldw
 *   bias   NULL, or [N] of bias_dtype MXQ_F32 / MXQ_BF16
 *   out    [M, N] row stride ldo; out_dtype MXQ_BF16 (rounded to nearest even
 *          from the fp32 accumulator) or MXQ_F32 (the accumulator itself)
 *   workspace / ws_bytes: device scratch for split-K, 16-byte aligned, of
 *          at least mxq_fp8_scaled_mm_workspace_size bytes for the same
 *          arguments (a smaller non-NULL workspace is MXQ_ERR_INVALID_ARG);
 *          NULL runs the same GEMM without split-K.
 * Block sizes other than [128,128], [1,128] and per-tensor (e.g. MXFP8
 * [1, 32]) give MXQ_ERR_UNSUPPORTED, as the page's block_size check does.
 * M == 0 or N == 0 is a no-op; K must be positive.
 */
mxq_status mxq_fp8_scaled_mm(const void* A, int32_t a_dtype, int64_t M, int64_t K, int64_t lda,
                             const float* a_scale, int64_t sa0, int64_t sa1, const void* W,
                             int64_t N, int64_t ldw, const float* w_scale, int32_t block_n,
                             int32_t block_k, int64_t sw0, int64_t sw1, const void* bias,
                             int32_t bias_dtype, void* out, int32_t out_dtype, int64_t ldo,
                             void* workspace, size_t ws_bytes, mxq_stream_t stream);

/*
 * mxq_fp8_scaled_mm for callers that cannot allocate device memory (no
 * counterpart on the pages; it exists for this library's users).  Some callers
 * cannot call cudaMalloc or hand over a workspace: plugins that receive only
 * their input and output buffers, code inside a framework whose memory pool
 * forbids raw allocations, or serving loops that must not allocate after
 * start-up.  This entry point takes exactly the arguments of mxq_fp8_scaled_mm
 * minus the workspace and computes the same result; the split-K partial sums
 * it needs live in one fixed array inside the library,
 * MXQ_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, held from library load until the
 * process exits.  It allocates nothing.
 *   - A shape whose split-K plan needs more scratch than that is rejected with
 *     MXQ_ERR_UNSUPPORTED (mxq_last_error says how much it needs); shapes that
 *     need no split (large M) need no scratch and are always accepted.
 *   - Every call looks up the array's device address on the current device
 *     (a host-side query, no allocation); the set-up is therefore the same
 *     on every call, and a first call before any stream capture is advised
 *     only because the library loads its kernels then.
 *   - Every call on a device shares the one array and its contents are left
 *     from the previous call (the partials are fully rewritten, so nothing
 *     needs to start at zero).  Calls whose executions overlap on the GPU,
 *     e.g. on two streams at once, race on the array: serialize them.
 */
#define MXQ_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
mxq_status mxq_fp8_scaled_mm_noalloc(const void* A, int32_t a_dtype, int64_t M, int64_t K,
                                     int64_t lda, const float* a_scale, int64_t sa0, int64_t sa1,
                                     const void* W, int64_t N, int64_t ldw, const float* w_scale,
                                     int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
                                     const void* bias, int32_t bias_dtype, void* out,
                                     int32_t out_dtype, int64_t ldo, mxq_stream_t stream);

/*
 * Load-time weight prepack for mxq_fp8_scaled_mm ([CPU-GEMM], implementation
 * breakdown: the FP8 weight is transposed and packed once after loading into
 * the layout the kernel reads; [XPU-FP8], process_weights_after_loading_block_quant:
 * the block scales are stored transposed-contiguous).  Here:
 *   Wp    ceil(N/128) * ceil(K/128) tiles of 16384 bytes; tile (tn, kb) at
 *         byte offset (tn * ceil(K/128) + kb) * 16384 holds rows
 *         tn*128 .. tn*128+127 and K bytes kb*128 .. kb*128+127 of W as the
 *         tensor core's 128-byte-swizzled operand image: byte b of 16-byte
 *         chunk c of tile row r at r*128 + ((c ^ (r % 8)) * 16) + b.  Rows
 *         past N and columns past K are zero.  256-byte aligned.
 *   ws_p  block scales K-block-major: Ws[nb, kb] at ws_p[kb * ceil(N/bn) + nb]
 *         ([ceil(K/128), ceil(N/bn)] contiguous); per-tensor: the one scale.
 *   W, w_scale, block_n, block_k, sw0, sw1 as in mxq_fp8_scaled_mm (W row
 *   stride ldw, a multiple of 16).  Sizes of Wp and ws_p come from
 *   mxq_prepacked_weight_size.  Asynchronous on `stream`.
 */
mxq_status mxq_prepacked_weight_size(int64_t N, int64_t K, int32_t block_n, int32_t block_k,
                                     size_t* w_bytes, size_t* s_bytes);
mxq_status mxq_prepack_weight(const void* W, int64_t N, int64_t K, int64_t ldw,
                              const float* w_scale, int32_t block_n, int32_t block_k, int64_t sw0,
                              int64_t sw1, void* Wp, float* ws_p, mxq_stream_t stream);

/*
 * mxq_fp8_scaled_mm with weights prepacked by mxq_prepack_weight (Wp, ws_p
 * for the same N, K, block_n, block_k).  Every other argument, the split-K
 * plan and its workspace (mxq_fp8_scaled_mm_workspace_size) are those of
 * mxq_fp8_scaled_mm, and the result is bit-identical to it: only the way
 * the weight tiles reach shared memory differs (one contiguous bulk copy per
 * tile instead of a tensor-map copy of 128 strided rows).
 */
mxq_status mxq_fp8_scaled_mm_prepacked(const void* A, int32_t a_dtype, int64_t M, int64_t K,
                                       int64_t lda, const float* a_scale, int64_t sa0, int64_t sa1,
                                       const void* Wp, int64_t N, const float* ws_p,
                                       int32_t block_n, int32_t block_k, const void* bias,
                                       int32_t bias_dtype, void* out, int32_t out_dtype,
                                       int64_t ldo, void* workspace, size_t ws_bytes,
                                       mxq_stream_t stream);

/*
 * Block-FP8 linear on bf16 activations ([XPU-FP8], torch_w8a8_block_fp8_linear
 * excerpt: with no input scale the input is quantized per 1 x block_k group by
 * per_token_group_quant_fp8 before scaled_mm):
 *   out = fp8_scaled_mm(per_token_group_quant_fp8(x, 128, 1e-10), W, w_scale)
 * x bf16 [M, K] (row stride ldx, 16-byte rows); W, w_scale, block_n in {1, 128},
 * block_k = 128, bias, out as in mxq_fp8_scaled_mm.  With MXQ_OPT_FUSE_QUANT = 1,
 * up to 32 rows the quantization runs inside the GEMM: each K slice of
 * a token row is one 1 x 128 group, turned into e4m3 codes and a scale by the
 * same IEEE arithmetic as mxq_per_token_group_quant_fp8, so codes, scales and
 * output are bit-identical to the two-step path; otherwise the two steps run.
 * workspace: mxq_w8a8_block_fp8_linear_workspace_size bytes (256-byte
 * aligned; may be 0: then NULL), holding the quantized activations when not
 * fused and the split-K partials.
 */
mxq_status mxq_w8a8_block_fp8_linear(const void* x, int64_t M, int64_t K, int64_t ldx,
                                     const void* W, int64_t N, int64_t ldw, const float* w_scale,
                                     int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
                                     const void* bias, int32_t bias_dtype, void* out,
                                     int32_t out_dtype, int64_t ldo, void* workspace,
                                     size_t ws_bytes, mxq_stream_t stream);
mxq_status mxq_w8a8_block_fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K,
                                                    int32_t block_n, size_t* bytes);

/*
 * Batched scaled FP8 GEMM: `batch` independent mxq_fp8_scaled_mm problems of
 * one shape in one launch ([CPU-GEMM], motivation: the existing FP8 scaled
 * GEMM of bmm_cpu serves batched GEMMs such as the DeepSeek MLA projections).
 * For every b < batch:
 *   out[b] = scaled_mm(A[b], a_scale[b], W[b], w_scale[b]) (+ bias[b])
 * with every per-problem argument as in mxq_fp8_scaled_mm, and batch strides
 * (in elements) between consecutive problems:
 *   a_bstride   must equal M * lda  (A problems stacked row-contiguously)
 *   w_bstride   must equal N * ldw  (W problems stacked row-contiguously)
 *   sa_bstride, sw_bstride, bias_bstride (0 = one bias for all), out_bstride:
 *               any value >= 0
 * Other strides give MXQ_ERR_UNSUPPORTED.  No split-K (no workspace).
 * batch == 0, M == 0 or N == 0 is a no-op.
 */
mxq_status mxq_fp8_scaled_bmm(int64_t batch, const void* A, int32_t a_dtype, int64_t M, int64_t K,
                              int64_t lda, int64_t a_bstride, const float* a_scale, int64_t sa0,
                              int64_t sa1, int64_t sa_bstride, const void* W, int64_t N,
                              int64_t ldw, int64_t w_bstride, const float* w_scale,
                              int32_t block_n, int32_t block_k, int64_t sw0, int64_t sw1,
                              int64_t sw_bstride, const void* bias, int32_t bias_dtype,
                              int64_t bias_bstride, void* out, int32_t out_dtype, int64_t ldo,
                              int64_t out_bstride, mxq_stream_t stream);

/* Workspace bytes of the split-K plan mxq_fp8_scaled_mm runs for this shape
 * on the current device (0 when it does not split).  The plan depends on the
 * activation type and the weight block size (a_dtype, block_n, block_k take
 * the values the call will get), so the size describes exactly that call.
 * Unsupported block sizes give MXQ_ERR_UNSUPPORTED as in the call. */
mxq_status mxq_fp8_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t a_dtype,
                                            int32_t block_n, int32_t block_k, size_t* bytes);

/*
 * Expert-block alignment ([CPU-MoE], the stage-1 tile loop consumes
 * sorted_ids / expert_ids / offsets: block mb holds expert expert_ids[mb];
 * its token slots are sorted_ids[mb*block_m + m] for
 * m < offsets[mb+1] - offsets[mb]; the token of a slot is slot / topk).
 *   topk_ids   int32 [T, topk], values in [0, E)
 *   sorted_ids int32 [cap * block_m]: slots sorted by expert (ascending),
 *              stable (ascending slot) within an expert, each expert's slots
 *              split into blocks of block_m; padding = S = T*topk
 *   expert_ids int32 [cap]: expert of each block, -1 past num_blocks
 *   offsets    int32 [cap + 1]: compact prefix sum of block sizes,
 *              offsets[0] = 0, = S past num_blocks
 *   num_blocks int32 [1]
 *   cap        >= ceil(S/block_m) + min(E, S) (the bound on the block count)
 * Limits: 1 <= E <= 1024, block_m in {16, 32, 64, 128}.  Ids outside [0, E)
 * are skipped and flagged (MXQ_ERR_DEVICE from mxq_sync_status).
 * workspace: none needed (pass NULL, 0).
 */
mxq_status mxq_moe_align_block(const int32_t* topk_ids, int64_t T, int32_t topk, int32_t E,
                               int32_t block_m, int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* offsets, int32_t* num_blocks, int64_t cap,
                               void* workspace, size_t ws_bytes, mxq_stream_t stream);

/*
 * Routed fused MoE ([CPU-MoE], implementation breakdown: stage 1
 * hidden @ w1 per expert block, the activation, stage 2 @ w2; followed by the
 * top-k weighted combine).  For every slot (t, k), e = topk_ids[t, k]:
 *     h   = hidden[t] . W1[e]^T (+ b1[e])            [2N], fp32
 *     act = bf16( silu(h[:N]) * h[N:] )                [N]
 *     z   = act . W2[e]^T (+ b2[e])                    [K], fp32
 *   out[t] = bf16( sum_k topk_weights[t, k] * z_(t,k) ), ascending k.
 * Activations stay bf16 (W8A16): weights are decoded exactly to bf16.
 *   hidden   bf16 [T, K], row stride ldh
 *   wtype MXQ_W_FP8_BLOCK128:
 *     w1 e4m3 [E, 2N, K], w1_scale fp32 [E, ceil(2N/128), ceil(K/128)]
 *     w2 e4m3 [E, K, N],  w2_scale fp32 [E, ceil(K/128), ceil(N/128)]
 *   wtype MXQ_W_MXFP4 (K, N multiples of 32):
 *     w1 e2m1x2 [E, 2N, K/2], w1_scale ue8m0 [E, 2N, K/32]
 *     w2 e2m1x2 [E, K, N/2],  w2_scale ue8m0 [E, K, N/32]
 *   w1_bias fp32 [E, 2N] or NULL; w2_bias fp32 [E, K] or NULL
 *   topk_weights fp32 [T, topk]; topk_ids int32 [T, topk]
 *   block_m  in {16, 32, 64, 128}: tokens per expert block; 0 = the
 *            library's choice (32 when S = T*topk <= 16*E, else 64), the
 *            same value for mxq_fused_experts_workspace_size
 *   out      bf16 [T, K], row stride ldo
 *   workspace: mxq_fused_experts_workspace_size bytes, 256-byte aligned
 */
mxq_status mxq_fused_experts(const void* hidden, int64_t T, int64_t K, int64_t ldh, int32_t wtype,
                             int32_t E, int64_t N, const void* w1, const void* w1_scale,
                             const float* w1_bias, const void* w2, const void* w2_scale,
                             const float* w2_bias, const float* topk_weights,
                             const int32_t* topk_ids, int32_t topk, int32_t block_m, void* out,
                             int64_t ldo, void* workspace, size_t ws_bytes, mxq_stream_t stream);

/* Same as mxq_fused_experts, and additionally writes the checkpoints in slot
 * order (slot = t*topk + k): act_out bf16 [T*topk, N], y_out fp32
 * [T*topk, K] = topk_weight * z, and h_out fp32 [T*topk, 2N] = the stage-1
 * accumulator hidden . W1[e]^T before the bias (gate rows first).  Any of
 * them may be NULL. */
mxq_status mxq_fused_experts_debug(const void* hidden, int64_t T, int64_t K, int64_t ldh,
                                   int32_t wtype, int32_t E, int64_t N, const void* w1,
                                   const void* w1_scale, const float* w1_bias, const void* w2,
                                   const void* w2_scale, const float* w2_bias,
                                   const float* topk_weights, const int32_t* topk_ids,
                                   int32_t topk, int32_t block_m, void* out, int64_t ldo,
                                   void* workspace, size_t ws_bytes, void* act_out,
                                   float* y_out, float* h_out, mxq_stream_t stream);

/* mxq_fused_experts / _debug with a choice of stage-1 activation
 * (MXQ_ACT_SILU, or MXQ_ACT_SWIGLU_CLAMP with its alpha > 0 and limit > 0;
 * [CPU-MoE] names GPT-OSS among the MXFP4 MoE models its path serves).  The
 * checkpoint pointers may be NULL; the workspace is that of
 * mxq_fused_experts_workspace_size. */
mxq_status mxq_fused_experts_ex(const void* hidden, int64_t T, int64_t K, int64_t ldh,
                                int32_t wtype, int32_t E, int64_t N, const void* w1,
                                const void* w1_scale, const float* w1_bias, const void* w2,
                                const void* w2_scale, const float* w2_bias,
                                const float* topk_weights, const int32_t* topk_ids, int32_t topk,
                                int32_t block_m, int32_t activation, float alpha, float limit,
                                void* out, int64_t ldo, void* workspace, size_t ws_bytes,
                                void* act_out, float* y_out, float* h_out, mxq_stream_t stream);

mxq_status mxq_fused_experts_workspace_size(int64_t T, int64_t K, int32_t E, int64_t N,
                                            int32_t topk, int32_t block_m, int32_t wtype,
                                            size_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H_ */
