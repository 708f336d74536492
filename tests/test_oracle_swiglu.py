"""Pins of the oracle's clamped-SwiGLU activation (GPT-OSS style,
g' = min(g, limit), u' = clamp(u, -limit, limit), act = g' sigmoid(alpha g')
(u' + 1)) through relations to the SiLU-and-mul path, which is itself pinned
against library dense-MLP matmuls:
- limit far above every value and alpha = 1: act = silu(g) * (u + 1), i.e.
  the SiLU path with the up bias raised by one;
- alpha = 2: g sigmoid(2 g) = silu(2 g) / 2, i.e. half the SiLU path with the
  gate rows doubled (alpha sits inside the sigmoid, on the gate);
- identity weights feeding chosen values: gates above the limit saturate to
  limit * sigmoid(alpha * limit) * (u' + 1), ups are clamped on both sides."""
import math

import numpy as np
import torch

from mxfp4_quantized_gemm_token_gb300 import synth

W_FP8 = 1


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.contiguous().view(torch.uint8).numpy()


def bf(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def run(oracle, x, w1, s1, b1, w2, s2, N, act, alpha=1.702, limit=7.0):
    T = x.shape[0]
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)
    _, a, _ = oracle.fused_experts(bits(x), W_FP8, u8(w1), s1.numpy(), b1, u8(w2), s2.numpy(),
                                   None, tw, ids, N, checkpoints=True, activation=act,
                                   alpha=alpha, limit=limit)
    return bf(a)


def test_no_clamp_alpha_one_is_silu_with_shifted_up_bias(oracle):
    E, N, K, T = 1, 128, 256, 4
    w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=61)
    b1 = (torch.randn(E, 2 * N, generator=torch.Generator().manual_seed(62)) * 0.01).numpy()
    x = synth.activations(T, K, seed=63, scale_div=10)
    sw = run(oracle, x, w1, s1, b1, w2, s2, N, 1, alpha=1.0, limit=1e30)
    b1p = b1.copy()
    b1p[:, N:] += 1.0
    si = run(oracle, x, w1, s1, b1p, w2, s2, N, 0)
    assert np.allclose(sw, si, rtol=2 ** -7, atol=0)


def test_alpha_two_is_half_silu_of_doubled_gate(oracle):
    E, N, K, T = 1, 128, 256, 4
    w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=71)
    x = synth.activations(T, K, seed=72, scale_div=10)
    b1 = np.zeros((E, 2 * N), np.float32)
    sw = run(oracle, x, w1, s1, b1, w2, s2, N, 1, alpha=2.0, limit=1e30)
    s1d = s1.clone()
    s1d[:, : N // 128] *= 2.0                            # gate rows doubled (exact)
    b1p = b1.copy()
    b1p[:, N:] = 1.0                                     # (u + 1)
    si = run(oracle, x, w1, s1d, b1p, w2, s2, N, 0)
    assert np.allclose(sw, si / 2.0, rtol=2 ** -7, atol=0)


def test_clamps_with_identity_weights(oracle):
    N, K = 128, 256
    eye1 = torch.zeros(1, 2 * N, K)
    eye1[0, torch.arange(2 * N), torch.arange(2 * N)] = 1.0
    eye2 = torch.zeros(1, K, N)
    eye2[0, torch.arange(N), torch.arange(N)] = 1.0
    w1 = eye1.to(torch.float8_e4m3fn)
    w2 = eye2.to(torch.float8_e4m3fn)
    s1 = torch.ones(1, 2 * N // 128, K // 128)
    s2 = torch.ones(1, K // 128, N // 128)
    g = torch.tensor([100.0, 8.0, 7.0, -3.0] * 32)
    u = torch.tensor([50.0, -50.0, 2.0, -7.5] * 32)
    x = torch.zeros(1, K)
    x[0, :N], x[0, N:2 * N] = g, u
    x = x.to(torch.bfloat16)
    a = run(oracle, x, w1, s1, None, w2, s2, N, 1, alpha=1.702, limit=7.0)[0]
    sat = 7.0 / (1.0 + math.exp(-1.702 * 7.0))
    expect = [sat * 8.0, sat * -6.0, sat * 3.0, -3.0 / (1.0 + math.exp(1.702 * 3.0)) * -6.0]
    for i in range(4):
        assert a[i] == float(torch.tensor(expect[i]).to(torch.bfloat16))
