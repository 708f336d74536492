"""Fused MoE at the full workload sizes, checked on sampled tokens.

FP8-block W8A16: E = 256, topk = 8, K = 7168, N = 2048; MXFP4 with bias:
E = 128, topk = 4, K = N = 2880.  The GPU runs the whole batch; the oracle
recomputes a deterministic sample of tokens (a token's output depends only on
its own routes), using only the experts those tokens touch (expert ids are
renumbered, which leaves the result unchanged)."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import synth
from gpu_util import assert_bf16_close, bits16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8_weights():
    return synth.moe_fp8_weights(256, 2048, 7168, seed=0, device="cuda")


@pytest.fixture(scope="module")
def mx_weights():
    w = synth.moe_mxfp4_weights(128, 2880, 2880, seed=0, device="cuda")
    b = synth.moe_biases(128, 2880, 2880, seed=1, device="cuda")
    return w + b


def check_sampled(oracle, out, x, tw, ids, sample, w1, s1, w2, s2, b1, b2, wtype, N):
    sample = np.asarray(sample)
    sids = ids[sample].cpu()
    used = torch.unique(sids)
    remap = {int(e): i for i, e in enumerate(used)}
    new_ids = torch.tensor([[remap[int(e)] for e in row] for row in sids], dtype=torch.int32)
    idx = used.long().cuda()
    sc = u8 if wtype == mxq.W_MXFP4 else (lambda t: t.cpu().numpy())
    ref = oracle.fused_experts(
        bits16(x[sample]), wtype, u8(w1[idx]), sc(s1[idx]),
        None if b1 is None else b1[idx].cpu().numpy(), u8(w2[idx]), sc(s2[idx]),
        None if b2 is None else b2[idx].cpu().numpy(), tw[sample].cpu().numpy(),
        new_ids.numpy(), N)
    assert_bf16_close(out[torch.from_numpy(sample).cuda()], ref, what="sampled MoE tokens")


@pytest.mark.parametrize("T,routing", [(4, "uniform"), (32, "zipf"), (256, "uniform"),
                                       (1024, "zipf")])
def test_moe_fp8_full_size(oracle, fp8_weights, T, routing):
    w1, s1, w2, s2 = fp8_weights
    fn = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
    tw, ids = fn(T, 256, 8, seed=T)
    x = synth.activations(T, 7168, seed=T, scale_div=10, device="cuda")
    out = mxq.fused_experts(x, w1, s1, w2, s2, tw.cuda(), ids.cuda(), block_m=64)
    mxq.sync_status()
    sample = sorted(set([0, T - 1, T // 2]))
    check_sampled(oracle, out, x, tw, ids, sample, w1, s1, w2, s2, None, None,
                  mxq.W_FP8_BLOCK128, 2048)


def test_moe_fp8_full_size_small_expert_blocks(oracle, fp8_weights):
    """Blocks of 0, 4, 5 and 33 tokens at the full expert dimensions."""
    w1, s1, w2, s2 = fp8_weights
    tw, ids = synth.routing_blocks((0, 4, 5, 33), topk=8, E=256)
    T = ids.shape[0]
    x = synth.activations(T, 7168, seed=5, scale_div=10, device="cuda")
    out = mxq.fused_experts(x, w1, s1, w2, s2, tw.cuda(), ids.cuda(), block_m=16)
    mxq.sync_status()
    check_sampled(oracle, out, x, tw, ids, [0, 4, 9, 41], w1, s1, w2, s2, None, None,
                  mxq.W_FP8_BLOCK128, 2048)


@pytest.mark.parametrize("T,routing", [(1, "uniform"), (32, "zipf"), (64, "uniform"),
                                       (512, "zipf")])
def test_moe_mxfp4_full_size(oracle, mx_weights, T, routing):
    w1, s1, w2, s2, b1, b2 = mx_weights
    fn = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
    tw, ids = fn(T, 128, 4, seed=T)
    x = synth.activations(T, 2880, seed=T, scale_div=10, device="cuda")
    out = mxq.fused_experts(x, w1, s1, w2, s2, tw.cuda(), ids.cuda(), wtype=mxq.W_MXFP4,
                            w1_bias=b1, w2_bias=b2, block_m=64)
    mxq.sync_status()
    sample = sorted(set([0, T - 1, T // 3]))
    check_sampled(oracle, out, x, tw, ids, sample, w1, s1, w2, s2, b1, b2, mxq.W_MXFP4, 2880)
