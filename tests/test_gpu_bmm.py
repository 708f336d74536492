"""Batched scaled FP8 GEMM (mxq_fp8_scaled_bmm) against the oracle applied to
each problem of the batch: W8A16 and W8A8, [128,128], [1,128] and per-tensor
weight scales, ragged M / N / K tails, shared and per-batch bias, and an
MLA-like shape (many small per-head problems)."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import synth
from gpu_util import assert_bf16_close, assert_probe_close, bits16, u8

pytestmark = pytest.mark.gpu
E4M3, BF16 = 3, 1


def make(B, M, N, K, bn, w8a8, seed, bias):
    xs = [synth.activations(M, K, seed=seed + b, scale_div=4) for b in range(B)]
    ws, ss = [], []
    for b in range(B):
        if bn == 0:
            _, w, sc, _ = synth.per_tensor_fp8_problem(M=M, N=N, K=K, seed=seed + 50 + b)
            sc = sc.reshape(1) * (1 + 0.25 * b)
        else:
            w, sc = synth.block_fp8_weight(N, K, bn, seed=seed + 50 + b)
        ws.append(w)
        ss.append(sc)
    g = torch.Generator().manual_seed(seed)
    bias_t = None
    if bias == "shared":
        bias_t = torch.randn(N, generator=g)
    elif bias == "batch":
        bias_t = torch.randn(B, N, generator=g)
    return xs, ws, ss, bias_t


@pytest.mark.parametrize("B,M,N,K,bn,w8a8,bias", [
    (4, 17, 192, 512, 128, False, "shared"), (3, 33, 256, 640, 128, True, None),
    (2, 5, 130, 384, 1, True, "batch"), (5, 9, 128, 576, 0, False, "batch"),
    (16, 64, 512, 128, 128, False, None), (3, 150, 256, 256, 128, True, "shared")])
def test_bmm_matches_oracle_per_problem(oracle, B, M, N, K, bn, w8a8, bias):
    xs, ws, ss, bias_t = make(B, M, N, K, bn, w8a8, seed=B * 10 + M, bias=bias)
    x = torch.stack(xs).cuda()
    w = torch.stack(ws).cuda()
    wsc = torch.stack(ss).cuda()
    a_scale = None
    if w8a8:
        q, a_scale = mxq.per_token_group_quant_fp8(x)
        a = q
    else:
        a = x
    bc = None if bias_t is None else bias_t.cuda()
    block = None if bn == 0 else [bn, 128]
    o32 = mxq.fp8_scaled_bmm(a, w, wsc, block, a_scale=a_scale, bias=bc, out_dtype=torch.float32)
    o16 = mxq.fp8_scaled_bmm(a, w, wsc, block, a_scale=a_scale, bias=bc)
    mxq.sync_status()
    assert o16.shape == (B, M, N)
    for b in range(B):
        bb = None if bias_t is None else (bias_t if bias_t.dim() == 1 else bias_t[b]).numpy()
        if w8a8:
            rq, rs = oracle.per_token_group_quant_fp8(bits16(xs[b]), 128)
            rf, rb = oracle.scaled_mm(rq, E4M3, rs, u8(ws[b]), ss[b].numpy(), bn, 0 if bn == 0 else 128, bb)
        else:
            rf, rb = oracle.scaled_mm(bits16(xs[b]), BF16, None, u8(ws[b]), ss[b].numpy(), bn,
                                      0 if bn == 0 else 128, bb)
        assert_probe_close(o32[b], rf, what="batch %d accumulator" % b)
        assert_bf16_close(o16[b], rb, what="batch %d output" % b)


def test_bmm_empty_and_stride_rules():
    a = torch.zeros(0, 4, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(0, 128, 256, dtype=torch.float8_e4m3fn, device="cuda")
    out = mxq.fp8_scaled_bmm(a, w, torch.ones(0, device="cuda"), None)
    assert out.shape == (0, 4, 128)
    import ctypes
    from mxfp4_quantized_gemm_token_gb300 import _lib
    lib = _lib.load()
    x = torch.zeros(2, 4, 256, dtype=torch.bfloat16, device="cuda")
    wt = torch.zeros(2, 128, 256, dtype=torch.float8_e4m3fn, device="cuda")
    sc = torch.ones(2, device="cuda")
    o = torch.empty(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.mxq_fp8_scaled_bmm(2, P(x), BF16, 4, 256, 256, 4 * 256 + 8, None, 0, 0, 0, P(wt), 128,
                                256, 128 * 256, P(sc), 0, 0, 0, 0, 1, None, 0, 0, P(o), BF16, 128,
                                4 * 128, None)
    assert rc == _lib.ERR_UNSUPPORTED                      # A batches not stacked contiguously
