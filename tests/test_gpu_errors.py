"""Device-side failure detection without a GPU fault.

With the test-only stall switch set, the GEMM producers issue no copy, so
every consumer wait in the kernel runs out after the (shortened) wait budget;
the kernel must then stop, report MXQ_ERR_TIMEOUT through mxq_sync_status and
leave the context usable: the next normal call must be correct."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, bits16, u8

pytestmark = pytest.mark.gpu


def _gemm_case(oracle, M=20, N=256, K=512):
    x = synth.activations(M, K, seed=77)
    w, ws = synth.block_fp8_weight(N, K, 128, seed=78)
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x), 128)
    _, rb = oracle.scaled_mm(rq, 3, rs, u8(w), ws.numpy(), 128, 128)
    q, s = mxq.per_token_group_quant_fp8(x.cuda())
    return q, s, w.cuda(), ws.cuda(), rb


@pytest.mark.parametrize("kind", ["w8a8", "w8a16", "moe"])
def test_stalled_pipeline_times_out_and_recovers(oracle, kind):
    q, s, w, ws, rb = _gemm_case(oracle)
    mxq.sync_status()                                     # start clean
    old_budget = mxq.get_option(_lib.OPT_WAIT_BUDGET_NS)
    try:
        mxq.set_option(_lib.OPT_WAIT_BUDGET_NS, 20_000_000)   # 20 ms
        mxq.set_option(_lib.OPT_INJECT_STALL, 1)
        if kind == "w8a8":
            mxq.fp8_scaled_mm(q, w, ws, [128, 128], a_scale=s)
        elif kind == "w8a16":
            a, wt, scale, bias = synth.per_tensor_fp8_problem(seed=5)
            mxq.fp8_scaled_mm(a.cuda(), wt.cuda(), scale.cuda(), None, bias=bias.cuda())
        else:
            E, Nm, Km, T = 4, 128, 256, 5
            w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, Nm, Km, seed=3)
            tw, ids = synth.routing_uniform(T, E, 2, seed=4)
            x = synth.activations(T, Km, seed=5, scale_div=10)
            mxq.fused_experts(x.cuda(), w1.cuda(), s1.cuda(), w2.cuda(), s2.cuda(), tw.cuda(),
                              ids.cuda(), wtype=mxq.W_MXFP4, block_m=16)
        with pytest.raises(mxq.MxqError) as ei:
            mxq.sync_status()
        assert ei.value.status == _lib.ERR_TIMEOUT
    finally:
        mxq.set_option(_lib.OPT_INJECT_STALL, 0)
        mxq.set_option(_lib.OPT_WAIT_BUDGET_NS, old_budget)
    # the context is intact: a normal call runs and is correct
    out = mxq.fp8_scaled_mm(q, w, ws, [128, 128], a_scale=s)
    mxq.sync_status()
    assert_bf16_close(out, rb)
