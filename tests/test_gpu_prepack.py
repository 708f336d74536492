"""Load-time weight prepack (mxq_prepack_weight) and the GEMM on prepacked
weights (mxq_fp8_scaled_mm_prepacked).

The packed bytes are checked against the layout's definition (a numpy
restatement: tile (tn, kb) at (tn * ceil(K/128) + kb) * 16384, byte b of
16-byte chunk c of tile row r at r*128 + ((c ^ (r % 8)) * 16) + b, zeros
outside W), the scales against their K-block-major relayout, and the GEMM on
prepacked weights must be bit-identical to the GEMM on the original weights
(fp32 and bf16 outputs) in every orientation and block mode."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, bits16, u8

pytestmark = pytest.mark.gpu


def packed_reference(w_u8, N, K):
    nkb, ntn = -(-K // 128), -(-N // 128)
    full = np.zeros((ntn * 128, nkb * 128), np.uint8)
    full[:N, :K] = w_u8[:N, :K]
    out = np.zeros((ntn, nkb, 128, 8, 16), np.uint8)
    t = full.reshape(ntn, 128, nkb, 8, 16).transpose(0, 2, 1, 3, 4)   # [tn, kb, r, c, b]
    r = np.arange(128).reshape(-1, 1)
    c = np.arange(8).reshape(1, -1)
    out[:, :, r, c ^ (r % 8), :] = t[:, :, r, c, :]
    return out.reshape(-1)


@pytest.mark.parametrize("N,K,bn", [(256, 512, 128), (300, 200, 128), (130, 640, 1), (64, 96, 0)])
def test_prepack_layout_matches_its_definition(N, K, bn):
    ldw = -(-K // 16) * 16
    g = torch.Generator().manual_seed(N + K)
    wfull = torch.randint(0, 256, (N, ldw), generator=g, dtype=torch.uint8)
    w = wfull.cuda().view(torch.float8_e4m3fn)[:, :K]
    if bn == 0:
        ws = torch.full((1,), 0.5, device="cuda")
    else:
        ws = (torch.rand(-(-N // bn), -(-K // 128), generator=g) + 0.1).cuda()
    pw = mxq.prepack_weight(w, ws, None if bn == 0 else [bn, 128])
    torch.cuda.synchronize()
    ref = packed_reference(u8(wfull)[:, :K], N, K)
    assert np.array_equal(u8(pw.tiles)[:ref.size], ref)
    if bn:
        assert torch.equal(pw.scales.cpu()[:ws.numel()], ws.cpu().T.contiguous().reshape(-1))


def _both(q, w, ws, pw, block, a_scale, bias=None):
    outs = []
    for dt in (torch.float32, torch.bfloat16):
        o1 = mxq.fp8_scaled_mm(q, w, ws, block, a_scale=a_scale, bias=bias, out_dtype=dt)
        o2 = mxq.fp8_scaled_mm(q, pw, None, block, a_scale=a_scale, bias=bias, out_dtype=dt)
        mxq.sync_status()
        assert torch.equal(o1, o2), dt
        outs.append(o1)
    return outs


@pytest.mark.parametrize("M,N,K,bn,tile", [
    (1, 18432, 7168, 128, 0), (8, 4096, 7168, 128, 0), (17, 1000, 896, 128, 0),
    (128, 384, 640, 128, 0), (300, 704, 512, 128, 128), (300, 704, 512, 128, 192),
    (260, 384, 640, 128, 256), (1024, 2048, 1024, 128, 0), (64, 4096, 7168, 1, 0),
    (530, 448, 640, 1, 0)])
def test_prepacked_gemm_is_bit_identical(oracle, M, N, K, bn, tile):
    x = synth.activations(M, K, seed=M + N, device="cuda")
    w, ws = synth.block_fp8_weight(N, K, bn, seed=K, device="cuda")
    q, s = mxq.per_token_group_quant_fp8(x)
    pw = mxq.prepack_weight(w, ws, [bn, 128])
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3)).cuda()
    try:
        mxq.set_option(_lib.OPT_NORMAL_TILE, tile)
        o32, o16 = _both(q, w, ws, pw, [bn, 128], s, bias)
    finally:
        mxq.set_option(_lib.OPT_NORMAL_TILE, 0)
    # and the oracle on a few rows
    rows = sorted({0, M - 1, M // 2})
    ridx = torch.tensor(rows, device="cuda")
    rf, rb = oracle.scaled_mm(u8(q[ridx]), 3, s[ridx].cpu().numpy(), u8(w), ws.cpu().numpy(), bn,
                              128, bias.cpu().numpy())
    assert_bf16_close(o16[ridx], rb)


def test_prepacked_per_tensor_w8a16(oracle):
    a, w, scale, bias = synth.per_tensor_fp8_problem(seed=0)
    a, w, scale, bias = a.cuda(), w.cuda(), scale.cuda(), bias.cuda()
    pw = mxq.prepack_weight(w, scale, None)
    for dt in (torch.float32, torch.bfloat16):
        o1 = mxq.fp8_scaled_mm(a, w, scale, None, bias=bias, out_dtype=dt)
        o2 = mxq.fp8_scaled_mm(a, pw, None, None, bias=bias, out_dtype=dt)
        assert torch.equal(o1, o2)


def test_prepacked_linear_wrapper_and_3d_input():
    wq, ws = synth.block_fp8_weight(4096, 7168, 1, seed=1, device="cuda")
    pw = mxq.prepack_weight(wq, ws, [1, 128])
    base = synth.activations(64, 7296, seed=9, device="cuda").view(2, 32, 7296)
    x = base[:, :, :7168]
    assert torch.equal(mxq.w8a8_block_fp8_linear(x, wq, [1, 128], ws),
                       mxq.w8a8_block_fp8_linear(x, pw, [1, 128], None))
    with pytest.raises(ValueError):
        mxq.w8a8_block_fp8_linear(x, pw, [128, 128], None)    # packed for [1, 128]
