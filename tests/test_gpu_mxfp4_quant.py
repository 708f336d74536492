"""GPU MXFP4 weight quantizer (mxq_quantize_mxfp4) against the oracle's OCP MX
restatement: codes and scales bit-exact, for bf16 and fp32 inputs, strided
rows, rows spanning many binades, the hand-derived tie / saturation block,
all-zero and subnormal blocks; and weights it produced run through the fused
MoE against the oracle."""
import os

import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import synth
from gpu_util import assert_bf16_close, bits16, u8

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden_block():
    vals = []
    with open(os.path.join(GOLDEN, "mxfp4_ocp_rounding_block.txt")) as f:
        for line in f:
            if not line.startswith("#") and line.strip():
                vals.append(float(line.split()[0]))
    return vals


def check(oracle, x):
    pg, sg = mxq.quantize_mxfp4(x)
    torch.cuda.synchronize()
    pr, sr = oracle.mxfp4_quantize(x.float().cpu().numpy())
    assert np.array_equal(u8(sg), sr), "scales differ"
    assert np.array_equal(u8(pg), pr), "codes differ"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_random_rows_many_binades(oracle, dtype):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(96, 2880, generator=g) * torch.exp(torch.randn(96, 1, generator=g) * 4)
    check(oracle, x.to(dtype).cuda())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_edge_blocks(oracle, dtype):
    x = torch.zeros(4, 128)
    x[0, :32] = torch.tensor(golden_block())
    x[1, 32:64] = 0.0                                   # all-zero block
    x[1, 64:96] = torch.linspace(-1e-38, 1e-38, 32)     # tiny (subnormal range) values
    x[2, :32] = torch.tensor([3.0e38, -1.0e38] * 16)    # top of the exponent range
    x[3, :] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5] * 16) * 2.0 ** -20
    check(oracle, x.to(dtype).cuda())


def test_strided_rows(oracle):
    base = synth.activations(40, 2880 + 64, seed=3, device="cuda")
    check(oracle, base[:, :2880])


def test_quantized_weights_run_through_the_moe(oracle):
    E, N, K, T, topk = 4, 128, 256, 7, 2
    g = torch.Generator().manual_seed(9)
    w1f = (torch.randn(E, 2 * N, K, generator=g) * 0.05).cuda()
    w2f = (torch.randn(E, K, N, generator=g) * 0.05).cuda()
    w1, s1 = mxq.quantize_mxfp4(w1f)
    w2, s2 = mxq.quantize_mxfp4(w2f)
    x = synth.activations(T, K, seed=10, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=11)
    out = mxq.fused_experts(x.cuda(), w1, s1, w2, s2, tw.cuda(), ids.cuda(), wtype=mxq.W_MXFP4,
                            block_m=16)
    ref = oracle.fused_experts(bits16(x), oracle.W_MXFP4, u8(w1), u8(s1), None, u8(w2), u8(s2),
                               None, tw.numpy(), ids.numpy(), N)
    assert_bf16_close(out, ref)
