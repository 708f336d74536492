"""Block-FP8 linear on bf16 input (mxq_w8a8_block_fp8_linear): up to 32 token
rows the per-token-group quantization runs inside the GEMM.  The result must
be bit-identical to the two-step path (mxq_per_token_group_quant_fp8, then
mxq_fp8_scaled_mm) and to the unfused linear (MXQ_OPT_FUSE_QUANT = 0), and
match the oracle; ragged K and N, split-K plans, both weight block shapes,
bf16 and fp32 bias, a strided 3-D input and the full-size decode shapes."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, bits16, u8

pytestmark = pytest.mark.gpu
E4M3 = 3


class fuse_quant:
    """MXQ_OPT_FUSE_QUANT on inside the block (off is the default)."""

    def __enter__(self):
        mxq.set_option(_lib.OPT_FUSE_QUANT, 1)

    def __exit__(self, *exc):
        mxq.set_option(_lib.OPT_FUSE_QUANT, 0)


def two_step(x, w, ws, bn, bias):
    q, s = mxq.per_token_group_quant_fp8(x)
    return mxq.fp8_scaled_mm(q, w, ws, [bn, 128], a_scale=s, bias=bias)


@pytest.mark.parametrize("M,N,K,bn", [(1, 256, 512, 128), (8, 384, 896, 128), (17, 200, 640, 1),
                                      (32, 640, 1024, 128), (5, 130, 200, 1), (31, 4096, 7168, 1),
                                      (3, 512, 4096, 128)])
def test_fused_linear_bit_identical(oracle, M, N, K, bn):
    ld = -(-K // 16) * 16                       # 16-byte rows (bf16 and fp8)
    base = synth.activations(M, ld, seed=M + K, device="cuda")
    x = base[:, :K]
    wc, ws = synth.block_fp8_weight(N, K, bn, seed=N, device="cuda")
    w = torch.zeros(N, ld * 2, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)[:, :K]
    w.copy_(wc)                                 # 16-byte weight rows for a ragged K
    bias = torch.randn(N, generator=torch.Generator().manual_seed(M)).cuda()
    with fuse_quant():
        fused = mxq.w8a8_block_fp8_linear(x, w, [bn, 128], ws, bias=bias)
        mxq.sync_status()
    if K % 16 == 0:
        assert torch.equal(fused, two_step(x.contiguous(), w, ws, bn, bias))
        assert torch.equal(fused, mxq.w8a8_block_fp8_linear(x, w, [bn, 128], ws, bias=bias))
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x), 128)
    _, rb = oracle.scaled_mm(rq, E4M3, rs, u8(w), ws.cpu().numpy(), bn, 128, bias.cpu().numpy())
    assert_bf16_close(fused, rb)


def test_fused_linear_split_k_and_3d_input(oracle):
    """Few weight tiles and long K: the plan splits K, and every split
    quantizes the groups of its own K range."""
    M, N, K = 6, 256, 7168
    big = synth.activations(M, K + 64, seed=2, device="cuda").view(2, 3, K + 64)
    x = big[:, :, :K]                             # strided 3-D input
    w, ws = synth.block_fp8_weight(N, K, 128, seed=3, device="cuda")
    with fuse_quant():
        out = mxq.w8a8_block_fp8_linear(x, w, [128, 128], ws)
    assert out.shape == (2, 3, N)
    ref = two_step(x.reshape(M, K).contiguous(), w, ws, 128, None)
    assert torch.equal(out.reshape(M, N), ref)


@pytest.mark.parametrize("M", [1, 8, 17])
def test_fused_linear_full_size(oracle, M):
    w, ws = synth.block_fp8_weight(18432, 7168, 128, seed=0, device="cuda")
    x = synth.activations(M, 7168, seed=100 + M, device="cuda")
    with fuse_quant():
        out = mxq.w8a8_block_fp8_linear(x, w, [128, 128], ws)
    assert torch.equal(out, two_step(x, w, ws, 128, None))
