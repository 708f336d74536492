"""Fused MoE at the full workload sizes, checked on sampled tokens.

FP8-block W8A16: E = 256, topk = 8, K = 7168, N = 2048; MXFP4 with bias:
E = 128, topk = 4, K = N = 2880.  Each case runs at block_m 0 (the library's
choice, the shipped default: 32-slot blocks with two weight-decode groups
except FP8 at T = 1024) and at 64.  The GPU runs the whole batch; the oracle
recomputes a deterministic sample of tokens (a token's output depends only on
its own routes), using only the experts those tokens touch (expert ids are
renumbered, which leaves the result unchanged).  The two fp32 stage
accumulators (h before the bias, y = w * z) of every slot of the sampled
tokens are checked at the accumulator tolerance against the oracle's
per-expert GEMM on the GPU's own stage inputs."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import synth
from gpu_util import assert_bf16_close, bits16, moe_stage_probes, u8

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


def run_full(oracle, wts, wtype, N, K, T, tw, ids, x, block_m, sample):
    w1, s1, w2, s2, b1, b2 = wts
    out = mxq.fused_experts(x, w1, s1, w2, s2, tw.cuda(), ids.cuda(), wtype=wtype, w1_bias=b1,
                            w2_bias=b2, block_m=block_m)
    mxq.sync_status()
    check_sampled(oracle, out, x, tw, ids, sample, w1, s1, w2, s2, b1, b2, wtype, N)
    out2, act, y, h = mxq.fused_experts(x, w1, s1, w2, s2, tw.cuda(), ids.cuda(), wtype=wtype,
                                        w1_bias=b1, w2_bias=b2, block_m=block_m,
                                        checkpoints=True)
    mxq.sync_status()
    assert torch.equal(out, out2)
    sc = u8 if wtype == mxq.W_MXFP4 else (lambda t: t.cpu().numpy())

    def expert(e):
        return (u8(w1[e:e + 1]), sc(s1[e:e + 1]), u8(w2[e:e + 1]), sc(s2[e:e + 1]),
                None if b2 is None else b2[e].cpu().numpy())
    topk = ids.shape[1]
    slots = [t * topk + k for t in sample for k in range(topk)]
    moe_stage_probes(oracle, wtype, bits16(x), ids.numpy(), tw.numpy(), expert, act, y, h, slots)


@pytest.mark.parametrize("block_m", [0, 64])
@pytest.mark.parametrize("T,routing", [(4, "uniform"), (32, "zipf"), (256, "uniform"),
                                       (1024, "zipf")])
def test_moe_fp8_full_size(oracle, fp8_weights, T, routing, block_m):
    fn = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
    tw, ids = fn(T, 256, 8, seed=T)
    x = synth.activations(T, 7168, seed=T, scale_div=10, device="cuda")
    run_full(oracle, fp8_weights + (None, None), mxq.W_FP8_BLOCK128, 2048, 7168, T, tw, ids, x,
             block_m, sorted(set([0, T - 1, T // 2])))


def test_moe_fp8_full_size_small_expert_blocks(oracle, fp8_weights):
    """Blocks of 0, 4, 5 and 33 tokens at the full expert dimensions."""
    tw, ids = synth.routing_blocks((0, 4, 5, 33), topk=8, E=256)
    T = ids.shape[0]
    x = synth.activations(T, 7168, seed=5, scale_div=10, device="cuda")
    run_full(oracle, fp8_weights + (None, None), mxq.W_FP8_BLOCK128, 2048, 7168, T, tw, ids, x,
             16, [0, 4, 9, 41])


@pytest.mark.parametrize("block_m", [0, 64])
@pytest.mark.parametrize("T,routing", [(1, "uniform"), (32, "zipf"), (64, "uniform"),
                                       (512, "zipf")])
def test_moe_mxfp4_full_size(oracle, mx_weights, T, routing, block_m):
    fn = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
    tw, ids = fn(T, 128, 4, seed=T)
    x = synth.activations(T, 2880, seed=T, scale_div=10, device="cuda")
    run_full(oracle, mx_weights, mxq.W_MXFP4, 2880, 2880, T, tw, ids, x, block_m,
             sorted(set([0, T - 1, T // 3])))
