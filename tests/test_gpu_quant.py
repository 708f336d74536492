"""per_token_group_quant_fp8 on the GPU vs the oracle: codes and scales must
be bit-exact."""
import numpy as np
import pytest
import torch

import mxfp4_quantized_gemm_token_gb300 as mxq
from mxfp4_quantized_gemm_token_gb300 import synth
from gpu_util import bits16, u8

pytestmark = pytest.mark.gpu


def check(oracle, x, group=128):
    q, s = mxq.per_token_group_quant_fp8(x.cuda(), group)
    torch.cuda.synchronize()
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x.reshape(-1, x.shape[-1])), group)
    gq = u8(q.reshape(-1, x.shape[-1]))
    gs = s.reshape(-1, s.shape[-1]).cpu().numpy()
    assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32)), "scales differ"
    bad = np.argwhere(gq != rq)
    assert bad.size == 0, "codes differ at %s: got %s ref %s" % (
        bad[:5].tolist(), gq[tuple(bad[:5].T)], rq[tuple(bad[:5].T)])


@pytest.mark.parametrize("M,K", [(1, 7168), (8, 7168), (17, 7168), (128, 1024), (97, 576),
                                 (5, 200), (300, 384), (33, 128)])
def test_quant_bit_exact(oracle, M, K):
    check(oracle, synth.activations(M, K, seed=M * 7 + K))


@pytest.mark.parametrize("scale", [1e-6, 1e-2, 3e2, 1e4])
def test_quant_bit_exact_magnitudes(oracle, scale):
    x = (synth.activations(16, 1024, seed=5).float() * scale).to(torch.bfloat16)
    check(oracle, x)


def test_quant_special_groups(oracle):
    x = synth.activations(6, 512, seed=9)
    x[0] = 0                       # all-zero row: scale eps/448, codes 0
    x[1, :128] = -0.0              # signed zeros -> 0x80
    x[2, 5] = 1e30                 # one huge value dominates its group
    x[3, 130:140] = 2.0 ** -130    # bf16 subnormals
    x[4, 256:384] = 7.0            # constant group -> all 448
    check(oracle, x)


def test_quant_strided_and_3d(oracle):
    base = synth.activations(2 * 9, 7168 + 128, seed=11).view(2, 9, 7168 + 128)
    x = base[:, :, :7168]          # non-contiguous rows, 3-D
    q, s = mxq.per_token_group_quant_fp8(x.cuda())
    assert q.shape == (2, 9, 7168) and s.shape == (2, 9, 56)
    check(oracle, x)


def test_quant_generic_group_sizes(oracle):
    x = synth.activations(7, 1000, seed=12)
    for g in (32, 64, 256):
        check(oracle, x, group=g)


def test_quant_full_size_block_workload_sampled_rows(oracle):
    """M = 4096, K = 7168 on the GPU; a deterministic sample of rows checked
    bit for bit (rows are independent)."""
    x = synth.activations(4096, 7168, seed=0, device="cuda")
    q, s = mxq.per_token_group_quant_fp8(x)
    rows = np.unique(np.concatenate([[0, 1, 4095], np.random.default_rng(0).integers(0, 4096, 61)]))
    ridx = torch.from_numpy(rows).cuda()
    rq, rs = oracle.per_token_group_quant_fp8(bits16(x[ridx]), 128)
    assert np.array_equal(u8(q[ridx]), rq)
    assert np.array_equal(s[ridx].cpu().numpy().view(np.uint32), rs.view(np.uint32))


def every_bf16_below(amax, binades=14):
    """All bf16 magnitudes from amax * 2^-binades up to amax, with both signs."""
    top = int(torch.tensor([amax], dtype=torch.bfloat16).view(torch.int16).item())
    lo = top - binades * 128
    mags = torch.arange(max(lo, 1), top + 1, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return torch.cat([mags, -mags])


@pytest.mark.parametrize("amax", [1.0, 3.0, 5.0, 7.0, 0.3, 123.0, 1e-3, 2.5e4, 448.0, 1e-20])
def test_quant_every_bf16_input_per_scale(oracle, amax):
    """Every bf16 value within 2^14 of the group's largest, for scales s =
    amax / 448 that are and are not powers of two: the quotients x / s fall
    on, near and between all e4m3 rounding midpoints (and in the e4m3
    subnormal range), so any code reached by a route other than the IEEE
    division that disagrees with it shows up here."""
    vals = every_bf16_below(amax)
    a = torch.tensor([amax], dtype=torch.bfloat16)
    n = (vals.numel() + 126) // 127
    pad = torch.zeros(n * 127 - vals.numel(), dtype=torch.bfloat16)
    body = torch.cat([vals, pad]).view(n, 127)
    groups = torch.cat([a.expand(n, 1), body], dim=1)          # each group's largest is amax
    rows = (n + 7) // 8
    x = torch.cat([groups, torch.zeros(rows * 8 - n, 128, dtype=torch.bfloat16)]).view(rows, 8 * 128)
    check(oracle, x)
