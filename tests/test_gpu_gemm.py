"""fp8_scaled_mm on the GPU vs the oracle.

W8A8 block (both weight block shapes) and W8A16 per-tensor at sizes that span
several tiles and ragged tails, the per-tensor == constant-block identity,
the scale-layout bit-identity, split-K, and the full-size block workloads
(sampled full rows)."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, assert_probe_close, bits16, u8

pytestmark = pytest.mark.gpu
E4M3, BF16 = 3, 1


def block_case(oracle, M, N, K, block_n, seed, bias=None, x=None):
    if x is None:
        x = synth.activations(M, K, seed=seed)
    wq, ws = synth.block_fp8_weight(N, K, block_n, seed=seed + 1)
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x), 128)
    b_np = None if bias is None else (bits16(bias) if bias.dtype == torch.bfloat16 else bias.numpy())
    rf, rb = oracle.scaled_mm(rq, E4M3, rs, u8(wq), ws.numpy(), block_n, 128, b_np)
    xc = x.cuda()
    q, s = mxq.per_token_group_quant_fp8(xc)
    bc = None if bias is None else bias.cuda()
    o32 = mxq.fp8_scaled_mm(q, wq.cuda(), ws.cuda(), [block_n, 128], a_scale=s, bias=bc,
                            out_dtype=torch.float32)
    o16 = mxq.fp8_scaled_mm(q, wq.cuda(), ws.cuda(), [block_n, 128], a_scale=s, bias=bc)
    mxq.sync_status()
    assert_probe_close(o32, rf)
    assert_bf16_close(o16, rb)
    return o32, o16


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (17, 384, 896), (97, 200, 640),
                                   (130, 256, 384), (64, 128, 128), (33, 640, 1024),
                                   (300, 384, 256)])
def test_w8a8_block128(oracle, M, N, K):
    bias = torch.randn(N, generator=torch.Generator().manual_seed(M))
    block_case(oracle, M, N, K, 128, seed=M + N, bias=bias)


@pytest.mark.parametrize("M,N,K", [(16, 256, 256), (65, 300, 512), (2, 4096, 1024)])
def test_w8a8_block1x128(oracle, M, N, K):
    block_case(oracle, M, N, K, 1, seed=M * 3 + 1)


def test_w8a8_page_numerical_case_bf16_bias(oracle):
    """The XPU page's numerical test shape: M, K, N = 16, 256, 256, block
    [128, 128], weight_scale = rand + 0.1, bf16 bias."""
    g = torch.Generator().manual_seed(0)
    x = torch.randn(16, 256, generator=g).to(torch.bfloat16)
    w = torch.randn(256, 256, generator=g).to(torch.float8_e4m3fn)
    ws = torch.rand(2, 2, generator=g) + 0.1
    bias = torch.randn(256, generator=g).to(torch.bfloat16)
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x), 128)
    rf, rb = oracle.scaled_mm(rq, E4M3, rs, u8(w), ws.numpy(), 128, 128, bits16(bias))
    out = mxq.w8a8_block_fp8_linear(x.cuda(), w.cuda(), [128, 128], ws.cuda(), bias=bias.cuda())
    assert out.dtype == torch.bfloat16
    assert_bf16_close(out, rb)
    # post-load transposed-contiguous scale storage: bit-identical output
    ws_t = torch.empty_strided(ws.shape, (1, ws.shape[0]), device="cuda")
    ws_t.copy_(ws.cuda())
    out_t = mxq.w8a8_block_fp8_linear(x.cuda(), w.cuda(), [128, 128], ws_t, bias=bias.cuda())
    assert torch.equal(out, out_t)
    # pre-quantized input path returns bf16 as well
    q, s = mxq.per_token_group_quant_fp8(x.cuda())
    out_q = mxq.w8a8_block_fp8_linear(q, w.cuda(), [128, 128], ws.cuda(), input_scale=s,
                                      bias=bias.cuda())
    assert out_q.dtype == torch.bfloat16 and torch.equal(out_q, out)


def test_linear_rejects_mxfp8_block():
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, 256, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(ValueError):
        mxq.w8a8_block_fp8_linear(x, w, [1, 32], torch.ones(128, 8, device="cuda"))
    with pytest.raises(mxq.MxqError) as ei:
        q, s = mxq.per_token_group_quant_fp8(x)
        mxq.fp8_scaled_mm(q, w, torch.ones(128, 8, device="cuda"), [1, 32], a_scale=s)
    assert ei.value.status == _lib.ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [1, 11, 97])
@pytest.mark.parametrize("N", [128, 224])
@pytest.mark.parametrize("K", [512, 576])
@pytest.mark.parametrize("has_bias", [False, True])
def test_w8a16_per_tensor_page_grid(oracle, M, N, K, has_bias):
    a, w, scale, bias = synth.per_tensor_fp8_problem(M=M, N=N, K=K, seed=M + N + K, bias=has_bias)
    rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(w), scale.numpy(), 0, 0,
                              None if bias is None else bias.numpy())
    bc = None if bias is None else bias.cuda()
    for sc in (scale.cuda(), scale.reshape(1).cuda()):        # 0-d and [1] scales
        o16 = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), sc, None, bias=bc)
        o32 = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), sc, None, bias=bc, out_dtype=torch.float32)
        assert_bf16_close(o16, rb)
        assert_probe_close(o32, rf)


def test_w8a16_per_tensor_config(oracle):
    """The per-tensor W8A16 workload: A [97, 576], B [224, 576], scale 0.01, bias."""
    a, w, scale, bias = synth.per_tensor_fp8_problem(seed=0)
    rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(w), scale.numpy(), 0, 0, bias.numpy())
    o16 = mxq.fp8_per_tensor_linear(a.cuda(), w.cuda(), scale.cuda(), bias.cuda())
    assert_bf16_close(o16, rb)


@pytest.mark.parametrize("K,split", [(64, 0), (128, 0), (192, 0), (256, 0), (384, 3), (640, 2)])
def test_w8a16_per_tensor_short_k_and_split(oracle, K, split):
    """Whole-K accumulation over one or two 128-wide slices (the two MMA
    issuers then hold one slice each, or one holds none), and split-K units of
    a single slice."""
    a, w, scale, bias = synth.per_tensor_fp8_problem(M=33, N=256, K=K, seed=K)
    rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(w), scale.numpy(), 0, 0, bias.numpy())
    try:
        mxq.set_option(_lib.OPT_SPLIT_K, split)
        o32 = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), scale.cuda(), None, bias=bias.cuda(),
                                out_dtype=torch.float32)
        o16 = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), scale.cuda(), None, bias=bias.cuda())
        mxq.sync_status()
    finally:
        mxq.set_option(_lib.OPT_SPLIT_K, 0)
    assert_probe_close(o32, rf)
    assert_bf16_close(o16, rb)


def test_per_tensor_equals_constant_blocks_on_gpu():
    a, w, scale, bias = synth.per_tensor_fp8_problem(M=40, N=256, K=512, seed=3)
    ac, wc = a.cuda(), w.cuda()
    pt = mxq.fp8_scaled_mm(ac, wc, scale.cuda(), None, out_dtype=torch.float32)
    blk = mxq.fp8_scaled_mm(ac, wc, torch.full((2, 4), 0.01, device="cuda"), [128, 128],
                            out_dtype=torch.float32)
    assert_probe_close(blk, pt.double().cpu().numpy())


def test_w8a16_with_block_weights(oracle):
    M, N, K = 20, 256, 384
    a = synth.activations(M, K, seed=4)
    wq, ws = synth.block_fp8_weight(N, K, 128, seed=5)
    rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(wq), ws.numpy(), 128, 128)
    o = mxq.fp8_scaled_mm(a.cuda(), wq.cuda(), ws.cuda(), [128, 128], out_dtype=torch.float32)
    assert_probe_close(o, rf)


def test_split_k_matches(oracle):
    M, N, K = 8, 256, 2048
    x = synth.activations(M, K, seed=21)
    wq, ws = synth.block_fp8_weight(N, K, 128, seed=22)
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x), 128)
    rf, _ = oracle.scaled_mm(rq, E4M3, rs, u8(wq), ws.numpy(), 128, 128)
    q, s = mxq.per_token_group_quant_fp8(x.cuda())
    try:
        for sp in (2, 3, 16):
            mxq.set_option(_lib.OPT_SPLIT_K, sp)
            o = mxq.fp8_scaled_mm(q, wq.cuda(), ws.cuda(), [128, 128], a_scale=s,
                                  out_dtype=torch.float32)
            assert_probe_close(o, rf, what="split %d" % sp)
    finally:
        mxq.set_option(_lib.OPT_SPLIT_K, 0)


def test_persistent_loop_several_units_per_cta(oracle):
    """Cap the grid at 3 CTAs so each CTA runs many tiles back to back."""
    try:
        mxq.set_option(_lib.OPT_NUM_SMS, 3)
        block_case(oracle, 150, 520, 512, 128, seed=31)
        a, w, scale, bias = synth.per_tensor_fp8_problem(M=97, N=600, K=576, seed=32)
        rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(w), scale.numpy(), 0, 0, bias.numpy())
        o = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), scale.cuda(), None, bias=bias.cuda())
        assert_bf16_close(o, rb)
    finally:
        mxq.set_option(_lib.OPT_NUM_SMS, 0)


def test_empty_problems_are_noops():
    w = torch.zeros(128, 256, dtype=torch.float8_e4m3fn, device="cuda")
    a = torch.zeros(0, 256, dtype=torch.bfloat16, device="cuda")
    out = mxq.fp8_scaled_mm(a, w, torch.tensor(1.0, device="cuda"), None)
    assert out.shape == (0, 128)


# ------------------------------------------------------------ full size

@pytest.fixture(scope="module")
def big_w128():
    wq, ws = synth.block_fp8_weight(18432, 7168, 128, seed=0, device="cuda")
    return wq, ws, u8(wq), ws.cpu().numpy()


def sample_rows(M):
    """Row 0, the last row, and one row of every 128-token tile (at a
    varying offset inside the tile), so every token tile of the launch is
    checked."""
    rows = {0, M - 1, M // 2, (M * 7) // 11}
    for t in range((M + 127) // 128):
        rows.add(min(M - 1, t * 128 + (t * 37 + 5) % 128))
    return sorted(rows)


@pytest.mark.parametrize("M", [1, 8, 17, 128, 1024, 4096])
def test_full_size_block128_sampled_rows(oracle, big_w128, M):
    wq, ws, w_np, ws_np = big_w128
    x = synth.activations(M, 7168, seed=100 + M, device="cuda")
    q, s = mxq.per_token_group_quant_fp8(x)
    o32 = mxq.fp8_scaled_mm(q, wq, ws, [128, 128], a_scale=s, out_dtype=torch.float32)
    o16 = mxq.fp8_scaled_mm(q, wq, ws, [128, 128], a_scale=s)
    rows = sample_rows(M)
    ridx = torch.tensor(rows, device="cuda")
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x[ridx]), 128)
    rf, rb = oracle.scaled_mm(rq, E4M3, rs, w_np, ws_np, 128, 128)
    assert_probe_close(o32[ridx], rf)
    assert_bf16_close(o16[ridx], rb)


@pytest.mark.parametrize("M", [1, 64, 2048])
def test_full_size_block1x128_sampled_rows(oracle, M):
    wq, ws = synth.block_fp8_weight(4096, 7168, 1, seed=1, device="cuda")
    if M >= 64:
        base = synth.activations(M, 7168 + 128, seed=200 + M, device="cuda").view(2, M // 2, 7296)
        x = base[:, :, :7168]                       # non-contiguous 3-D input
    else:
        x = synth.activations(M, 7168, seed=200 + M, device="cuda")
    out = mxq.w8a8_block_fp8_linear(x, wq, [1, 128], ws)
    assert out.shape == (*x.shape[:-1], 4096)
    flat = out.reshape(-1, 4096)
    xf = x.reshape(-1, 7168)
    # the fp32 accumulator of the same call (quantized input, same plan)
    q, s = mxq.per_token_group_quant_fp8(xf)
    o32 = mxq.fp8_scaled_mm(q, wq, ws, [1, 128], a_scale=s, out_dtype=torch.float32)
    rows = sample_rows(M)
    ridx = torch.tensor(rows, device="cuda")
    rq, rs = oracle.per_token_group_quant_fp8(bits16(xf[ridx]), 128)
    rf, rb = oracle.scaled_mm(rq, E4M3, rs, u8(wq), ws.cpu().numpy(), 1, 128)
    assert_bf16_close(flat[ridx], rb)
    assert_probe_close(o32[ridx], rf)
    if M > 128:
        # token-major tiles, scales stored [kb][n]: the same bits
        t32 = mxq.fp8_scaled_mm(q, wq, transposed(ws), [1, 128], a_scale=s, out_dtype=torch.float32)
        assert torch.equal(t32, o32)


@pytest.mark.parametrize("tile", [128, 192, 256])
def test_token_major_tile_widths(oracle, tile):
    """Every weight-tile width of the token-major path (tokens on the MMA M
    side) on ragged shapes: partial last token and weight tiles, 192-wide
    tiles that start inside a 128-row weight block, bias, bf16 and f32 out."""
    try:
        mxq.set_option(_lib.OPT_NORMAL_TILE, tile)
        block_case(oracle, 300, 384, 640, 128, seed=61 + tile)
        block_case(oracle, 260, 704, 512, 128, seed=62 + tile,
                   bias=torch.randn(704, generator=torch.Generator().manual_seed(tile)))
        block_case(oracle, 129, 640, 384, 128, seed=63 + tile)
    finally:
        mxq.set_option(_lib.OPT_NORMAL_TILE, 0)


@pytest.mark.parametrize("seed", [71, 72])
def test_per_row_weight_scales_large_m(oracle, seed):
    """[1,128] weight scales at M > 512 with ragged token and weight tails and
    a bias (weight-major tiles, per-row scale per TMEM lane)."""
    block_case(oracle, 530, 448, 640, 1, seed=seed)
    block_case(oracle, 600, 200, 384, 1, seed=seed + 10,
               bias=torch.randn(200, generator=torch.Generator().manual_seed(seed)))


def transposed(t):
    """The same values stored column-major ([kb][n] in memory)."""
    out = torch.empty_strided(t.shape, (1, t.shape[0]), dtype=t.dtype, device=t.device)
    out.copy_(t)
    return out


@pytest.mark.parametrize("M,N,K", [(260, 392, 2400), (140, 136, 4224)])
def test_per_row_weight_scales_long_k_both_layouts(oracle, M, N, K):
    """[1,128] weight scales on the token-major tiles with K slice counts of
    19 (a ragged K tail) and 33, more than the scale ring's eight slots; scales
    stored [n][kb] and [kb][n] give the same bits."""
    bias = torch.randn(N, generator=torch.Generator().manual_seed(K))
    o32, o16 = block_case(oracle, M, N, K, 1, seed=M + K, bias=bias)
    x = synth.activations(M, K, seed=M + K).cuda()
    wq, ws = synth.block_fp8_weight(N, K, 1, seed=M + K + 1)
    q, s = mxq.per_token_group_quant_fp8(x)
    wst = transposed(ws.cuda())
    t32 = mxq.fp8_scaled_mm(q, wq.cuda(), wst, [1, 128], a_scale=s, bias=bias.cuda(),
                            out_dtype=torch.float32)
    t16 = mxq.fp8_scaled_mm(q, wq.cuda(), wst, [1, 128], a_scale=s, bias=bias.cuda())
    mxq.sync_status()
    assert torch.equal(t32, o32) and torch.equal(t16, o16)


@pytest.mark.parametrize("tile", [32, 64, 128, 256])
def test_forced_token_tile_widths(oracle, tile):
    """Every token-tile width (MMA N and epilogue split) on a ragged shape."""
    try:
        mxq.set_option(_lib.OPT_TILE_N, tile)
        block_case(oracle, 300, 384, 640, 128, seed=41 + tile)
        block_case(oracle, 70, 256, 384, 1, seed=43 + tile)
        a, w, scale, bias = synth.per_tensor_fp8_problem(M=97, N=224, K=576, seed=44)
        rf, rb = oracle.scaled_mm(bits16(a), BF16, None, u8(w), scale.numpy(), 0, 0, bias.numpy())
        o = mxq.fp8_scaled_mm(a.cuda(), w.cuda(), scale.cuda(), None, bias=bias.cuda())
        assert_bf16_close(o, rb)
    finally:
        mxq.set_option(_lib.OPT_TILE_N, 0)


@pytest.mark.parametrize("case", ["block128_decode", "block1x128_large_m", "block1x128_decode",
                                  "per_tensor_bf16"])
def test_workspace_query_describes_the_call(case):
    """The split-K workspace query takes the call's activation type and block
    size, so it sizes the plan the call runs: with exactly that many bytes the
    call succeeds, with 16 fewer (when the plan splits) it is refused, and the
    result equals the no-split run within the accumulator tolerance."""
    import ctypes
    lib = _lib.load()
    M, N, K, bn, a_dt = {"block128_decode": (8, 4096, 7168, 128, E4M3),
                         "block1x128_large_m": (512, 4608, 7168, 1, E4M3),
                         "block1x128_decode": (4, 4096, 7168, 1, E4M3),
                         "per_tensor_bf16": (8, 4096, 7168, 0, BF16)}[case]
    bk = 0 if bn == 0 else 128
    x = synth.activations(M, K, seed=90, device="cuda")
    if bn == 0:
        _, w, _, _ = synth.per_tensor_fp8_problem(M=M, N=N, K=K, seed=91)
        w, ws = w.cuda(), torch.full((1,), 0.01, device="cuda")
        a, s = x, None
    else:
        w, ws = synth.block_fp8_weight(N, K, bn, seed=91, device="cuda")
        a, s = mxq.per_token_group_quant_fp8(x)
    sz = ctypes.c_size_t(0)
    assert lib.mxq_fp8_scaled_mm_workspace_size(M, N, K, a_dt, bn, bk, ctypes.byref(sz)) == 0
    need = sz.value
    ref = mxq.fp8_scaled_mm(a, w, ws, None if bn == 0 else [bn, bk], a_scale=s,
                            out_dtype=torch.float32, workspace=torch.empty(0, dtype=torch.uint8,
                                                                           device="cuda"))
    nosplit = torch.empty_like(ref)

    def call(out, work, nbytes):
        return lib.mxq_fp8_scaled_mm(
            ctypes.c_void_p(a.data_ptr()), a_dt, M, K, K,
            None if s is None else ctypes.c_void_p(s.data_ptr()), 0 if s is None else s.stride(0),
            0 if s is None else s.stride(1), ctypes.c_void_p(w.data_ptr()), N, K,
            ctypes.c_void_p(ws.data_ptr()), bn, bk, ws.stride(0) if ws.dim() == 2 else 0,
            ws.stride(1) if ws.dim() == 2 else 0, None, 0, ctypes.c_void_p(out.data_ptr()),
            _lib.F32, N, None if work is None else ctypes.c_void_p(work.data_ptr()), nbytes,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    assert call(nosplit, None, 0) == 0
    if need > 0:
        work = torch.empty(need, dtype=torch.uint8, device="cuda")
        assert call(ref, work, need - 16) == _lib.ERR_INVALID_ARG
        assert b"workspace" in lib.mxq_last_error()
        assert call(ref, work, need) == 0
    else:
        assert call(ref, None, 0) == 0
    torch.cuda.synchronize()
    assert_probe_close(ref, nosplit.double().cpu().numpy())
    # the expected plans: decode-size shapes split, the [1, 128] large-M one does not
    assert (need > 0) == (M <= 8)
