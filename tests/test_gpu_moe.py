"""moe_align_block and fused_experts on the GPU vs the oracle.

Alignment is bit-exact; the fused MoE output is compared after bf16 rounding
(rtol = atol = 1e-2), with its checkpoints (act, y) as well.  Covers both
weight formats, biases, ragged K / N tails, empty experts and the expert block
sizes 4 / 5 / 33, topk > 1, every block_m, and both instruction-width paths."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, bits16, moe_stage_probes, u8

pytestmark = pytest.mark.gpu
W_FP8, W_MX = 1, 2


# ------------------------------------------------------------- align

@pytest.mark.parametrize("T,topk,E,BM,kind", [
    (1, 4, 128, 16, "uniform"), (37, 8, 256, 64, "uniform"), (64, 4, 128, 32, "zipf"),
    (300, 8, 256, 128, "zipf"), (5, 2, 3, 16, "uniform"), (1024, 8, 256, 64, "uniform"),
    (4096, 8, 256, 128, "zipf")])
def test_align_bit_exact(oracle, T, topk, E, BM, kind):
    fn = synth.routing_uniform if kind == "uniform" else synth.routing_zipf
    _, ids = fn(T, E, topk, seed=T + E)
    ref = oracle.moe_align(ids.numpy(), E, BM)
    got = mxq.moe_align_block(ids.cuda(), E, BM)
    for r, g in zip(ref[:3], got[:3]):
        assert np.array_equal(r, g.cpu().numpy())
    assert int(got[3].item()) == ref[3]


def test_align_small_blocks_and_empty_experts(oracle):
    _, ids = synth.routing_blocks((0, 4, 5, 33), topk=8, E=256)
    for BM in (16, 32, 64, 128):
        ref = oracle.moe_align(ids.numpy(), 256, BM)
        got = mxq.moe_align_block(ids.cuda(), 256, BM)
        for r, g in zip(ref[:3], got[:3]):
            assert np.array_equal(r, g.cpu().numpy())


def test_align_flags_out_of_range_ids():
    ids = torch.tensor([[0, 1], [7, 2]], dtype=torch.int32, device="cuda")
    mxq.moe_align_block(ids, 4, 16)
    with pytest.raises(mxq.MxqError) as ei:
        mxq.sync_status()
    assert ei.value.status == _lib.ERR_DEVICE
    mxq.sync_status()          # the word was cleared


# ------------------------------------------------------------ fused MoE

def weights(wtype, E, N, K, seed, bias):
    if wtype == W_FP8:
        w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=seed)
    else:
        w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=seed)
    b1 = b2 = None
    if bias:
        b1, b2 = synth.moe_biases(E, N, K, seed=seed + 1)
    return w1, s1, w2, s2, b1, b2


def run_moe(oracle, wtype, E, N, K, x, tw, ids, block_m, seed=1, bias=False, check_ckpt=True,
            wts=None, activation="silu", alpha=1.702, limit=7.0):
    w1, s1, w2, s2, b1, b2 = weights(wtype, E, N, K, seed, bias) if wts is None else wts
    sc = (lambda s: u8(s)) if wtype == W_MX else (lambda s: s.numpy())
    ref, ract, rz = oracle.fused_experts(
        bits16(x), wtype, u8(w1), sc(s1), None if b1 is None else b1.numpy(), u8(w2), sc(s2),
        None if b2 is None else b2.numpy(), tw.numpy(), ids.numpy(), N, checkpoints=True,
        activation=0 if activation == "silu" else 1, alpha=alpha, limit=limit)
    cu = lambda t: None if t is None else t.cuda()
    kw = dict(wtype=wtype, w1_bias=cu(b1), w2_bias=cu(b2), block_m=block_m,
              activation=activation, alpha=alpha, limit=limit)
    out, act, y, h = mxq.fused_experts(cu(x), cu(w1), cu(s1), cu(w2), cu(s2), cu(tw), cu(ids),
                                       checkpoints=True, **kw)
    plain = mxq.fused_experts(cu(x), cu(w1), cu(s1), cu(w2), cu(s2), cu(tw), cu(ids), **kw)
    mxq.sync_status()
    assert torch.equal(plain, out)          # the checkpoints do not change the result
    assert_bf16_close(out, ref, what="moe output")
    if check_ckpt:
        assert_bf16_close(act, ract, what="act checkpoint")

        def expert(e):
            return (u8(w1[e:e + 1]), sc(s1[e:e + 1]), u8(w2[e:e + 1]), sc(s2[e:e + 1]),
                    None if b2 is None else b2[e].numpy())
        moe_stage_probes(oracle, wtype, bits16(x), ids.numpy(), tw.numpy(), expert, act, y, h,
                         range(ids.numel()))
    return out


@pytest.mark.parametrize("block_m", [0, 16, 32, 64, 128])
def test_fused_fp8_small(oracle, block_m):
    E, N, K, T, topk = 8, 128, 256, 13, 2
    x = synth.activations(T, K, seed=3, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=4)
    run_moe(oracle, W_FP8, E, N, K, x, tw, ids, block_m)


def test_fused_fp8_ragged_dims_and_many_tokens(oracle):
    E, N, K, T, topk = 6, 192, 400, 70, 3       # K, N not multiples of 128
    x = synth.activations(T, K, seed=5, scale_div=10)
    tw, ids = synth.routing_zipf(T, E, topk, seed=6)
    run_moe(oracle, W_FP8, E, N, K, x, tw, ids, 32)


@pytest.mark.parametrize("block_m", [0, 16, 64])
def test_fused_mxfp4_bias(oracle, block_m):
    E, N, K, T, topk = 4, 160, 288, 9, 4
    x = synth.activations(T, K, seed=7, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=8)
    run_moe(oracle, W_MX, E, N, K, x, tw, ids, block_m, bias=True)


@pytest.mark.parametrize("wtype,block_m", [(W_MX, 32), (W_MX, 64), (W_FP8, 32)])
def test_fused_odd_slice_units_two_decode_groups(oracle, wtype, block_m):
    """K = N = 384: both stages reduce over three 128-wide slices, so the CTA's
    slice sequence changes parity at every unit boundary, with several units
    per CTA (64 experts x 6 or 3 tiles) and the weight decode split into two
    groups taking alternate slices (the layouts where the MMA issuers and
    the decode groups must agree on the alternation)."""
    E, N, K, T, topk = 64, 384, 384, 96, 4
    x = synth.activations(T, K, seed=21, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=22)
    run_moe(oracle, wtype, E, N, K, x, tw, ids, block_m, bias=(wtype == W_MX))


@pytest.mark.parametrize("wtype", [W_FP8, W_MX])
def test_fused_single_slice_stages(oracle, wtype):
    """K = 128 and N = 64: both GEMM stages reduce over one 128-wide slice,
    so one of the two MMA issuers has no slice in any unit."""
    E, N, K, T, topk = 4, 64, 128, 11, 2
    x = synth.activations(T, K, seed=13, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=14)
    run_moe(oracle, wtype, E, N, K, x, tw, ids, 16, bias=(wtype == W_MX))


@pytest.mark.parametrize("topk", [1, 8])
def test_fused_small_expert_blocks_4_5_33(oracle, topk):
    """Expert blocks of exactly 0, 4, 5 and 33 tokens (the vLLM CPU page's
    small-block test, plus topk > 1 and N != K which it left out)."""
    E = 256 if topk == 8 else 8
    tw, ids = synth.routing_blocks((0, 4, 5, 33), topk=topk, E=E)
    T = ids.shape[0]
    N, K = 128, 256
    x = synth.activations(T, K, seed=9, scale_div=10)
    run_moe(oracle, W_FP8, E, N, K, x, tw, ids, 16)


@pytest.mark.parametrize("N,K", [(128, 256), (160, 224)])
def test_fused_narrow_and_wide_paths_agree(oracle, N, K):
    """Per-block choice (threshold 4), always narrow, always full width and one
    path for the whole layer all give the oracle's result, also when the
    last weight tile of each stage is a ragged tail (N = 160: the SiLU
    stage's last 64-row tile holds 32 rows; K = 224: stage 2's last 128-row
    tile holds 96)."""
    E, T, topk = 8, 21, 2
    x = synth.activations(T, K, seed=11, scale_div=10)
    tw, ids = synth.routing_zipf(T, E, topk, seed=12)
    old = mxq.get_option(_lib.OPT_SMALL_M_MAX)
    try:
        mxq.set_option(_lib.OPT_SMALL_M_MAX, 4)
        for force in (0, 1, 2, 3):
            mxq.set_option(_lib.OPT_FORCE_PATH, force)
            run_moe(oracle, W_FP8, E, N, K, x, tw, ids, 64)
            run_moe(oracle, W_MX, E, N, K, x, tw, ids, 64)
    finally:
        mxq.set_option(_lib.OPT_FORCE_PATH, 0)
        mxq.set_option(_lib.OPT_SMALL_M_MAX, old)


@pytest.mark.parametrize("mode", [1, 2])
def test_fused_mxfp4_scales_beyond_bf16_single_step(oracle, mode):
    """ue8m0 exponents of 143 and above (scales of 2^16 and more, which the
    bf16 decode, mode 1, folds into the weights in two multiplications and
    the f16 decode, mode 2, applies as the row's fp32 factor) in stage 1,
    and small ones in stage 2, against the oracle, with the stage
    accumulators checked too."""
    E, N, K, T, topk = 4, 128, 256, 9, 2
    w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=51)
    s1 = (s1.to(torch.int32) + 21).clamp(max=254).to(torch.uint8)   # 141 .. 143
    s2 = (s2.to(torch.int32) - 21).clamp(min=1).to(torch.uint8)
    assert bool((s1 >= 143).any()) and bool((s1 < 143).any())
    b1, b2 = synth.moe_biases(E, N, K, seed=52)
    x = synth.activations(T, K, seed=53, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=54)
    try:
        mxq.set_option(_lib.OPT_MOE_F16, mode)
        run_moe(oracle, W_MX, E, N, K, x, tw, ids, 16, wts=(w1, s1, w2, s2, b1, b2))
    finally:
        mxq.set_option(_lib.OPT_MOE_F16, 3)


def test_fused_mxfp4_f16_decode_wide_exponent_spread(oracle):
    """The f16 decode scales each 32-group by 2^(e - emax of its weight row):
    every row's first group gets an exponent 20 above the rest but zero
    codes, so the whole result comes from groups 2^20 below the row's
    reference, which must stay exact (within 2^23 of it)."""
    E, N, K, T, topk = 4, 128, 256, 9, 2
    w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=61)
    w1, s1, w2, s2 = w1.clone(), s1.clone(), w2.clone(), s2.clone()
    for w, sc in ((w1, s1), (w2, s2)):
        w[..., :16] = 0                                     # group 0: all codes zero
        sc[..., 0] = (sc[..., 1:].to(torch.int32).amax(dim=-1) + 20).clamp(max=254).to(torch.uint8)
    b1, b2 = synth.moe_biases(E, N, K, seed=62)
    x = synth.activations(T, K, seed=63, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=64)
    try:
        mxq.set_option(_lib.OPT_MOE_F16, 2)
        run_moe(oracle, W_MX, E, N, K, x, tw, ids, 16, wts=(w1, s1, w2, s2, b1, b2))
    finally:
        mxq.set_option(_lib.OPT_MOE_F16, 3)


@pytest.mark.parametrize("wtype", [W_FP8, W_MX])
@pytest.mark.parametrize("limit", [7.0, 0.05])
def test_fused_clamped_swiglu(oracle, wtype, limit):
    """GPT-OSS-style clamped SwiGLU between the stages, with a limit the
    stage-1 values stay under (7) and one that clamps most of them (0.05),
    both weight formats, biases, topk 4."""
    E, N, K, T, topk = 6, 160, 288, 11, 4
    x = synth.activations(T, K, seed=81, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=82)
    run_moe(oracle, wtype, E, N, K, x, tw, ids, 16, bias=True, activation="swiglu_clamp",
            alpha=1.702, limit=limit)


@pytest.mark.parametrize("wtype,T,topk,E", [(W_FP8, 37, 8, 32), (W_MX, 50, 4, 16),
                                            (W_FP8, 5, 2, 3)])
def test_fused_combine_is_bit_identical_to_the_combine_kernel(oracle, wtype, T, topk, E):
    """The top-k combine inside the stage-2 GEMM (default) and the separate
    combine kernel give the same bits (same fp32 adds, ascending k), and
    agree with the oracle."""
    N, K = 128, 384
    x = synth.activations(T, K, seed=T, scale_div=10)
    tw, ids = synth.routing_zipf(T, E, topk, seed=T + 1)
    outs = []
    try:
        for fuse in (1, 0):
            mxq.set_option(_lib.OPT_FUSE_COMBINE, fuse)
            outs.append(run_moe(oracle, wtype, E, N, K, x, tw, ids, 16, bias=(wtype == W_MX),
                                check_ckpt=False))
    finally:
        mxq.set_option(_lib.OPT_FUSE_COMBINE, 0)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("wtype,block_m", [(W_FP8, 32), (W_MX, 32), (W_FP8, 64), (W_MX, 64)])
def test_fused_operand_modes(oracle, mode, wtype, block_m):
    """The expert GEMMs with bf16 operands (mode 0), f16 operands for FP8
    experts only (mode 1) and f16 for both formats (mode 2), against the
    oracle with the checkpoints and the stage-accumulator probes (the
    default mode 3 runs everywhere else)."""
    E, N, K, T, topk = 12, 256, 384, 40, 4
    x = synth.activations(T, K, seed=91, scale_div=10)
    tw, ids = synth.routing_zipf(T, E, topk, seed=92)
    try:
        mxq.set_option(_lib.OPT_MOE_F16, mode)
        run_moe(oracle, wtype, E, N, K, x, tw, ids, block_m, bias=(wtype == W_MX))
    finally:
        mxq.set_option(_lib.OPT_MOE_F16, 3)
