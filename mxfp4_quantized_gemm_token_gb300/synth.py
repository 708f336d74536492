"""Seeded synthetic inputs for the quantized scaled-GEMM / fused-MoE path.

This module only *draws* inputs: random activations, pre-quantized weights
(as a checkpoint would hold them) and routing decisions.  It implements none
of the hot-path steps (activation group quantization, the scaled GEMMs,
expert alignment, the MoE stages, the combine); the CUDA library and the CPU
oracle both consume exactly the bytes produced here.

Recipes (workload shapes from the pages' tests and the stated configs):
  * per-tensor W8A16: A = randn/10 bf16, B = randn cast to e4m3, scale 0.01,
    fp32 bias randn  ("[CPU] fp8_per_tensor_scaled_mm_cpu", test section);
  * block FP8 weights: randn * 0.05, one fp32 scale amax/448 per
    [block_n, 128] block, elements cast to e4m3 (round to nearest even);
  * MXFP4 weights: randn * 0.05; per 32 consecutive K elements a shared
    power of two 2^(floor(log2 amax) - 2), elements rounded to the nearest
    e2m1 value (ties to the even code) with saturation at +-6, two codes per
    byte with the even K index in the low nibble, the exponent stored as
    ue8m0 (e + 127);
  * routing: uniform (softmax of randn logits, top-k), Zipf(s) concentrated
    (log-popularity -s*log(rank) over a random rank permutation plus Gumbel
    noise, softmax top-k), or deterministic expert blocks of given sizes
    ("[CPU] routed FP8/MXFP4 MoE" test helper that builds exact block sizes
    from consecutive tokens).  Top-k weights are the softmax values, not
    renormalised.
All CPU draws use ``torch.Generator`` seeded explicitly, so the data is
identical on any machine; large weights may be drawn on a CUDA device with a
seeded CUDA generator.
"""
from __future__ import annotations

import math

import torch

FP8 = torch.float8_e4m3fn


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    return torch.randn(*shape, generator=_gen(seed, device), device=device,
                       dtype=torch.float32).to(dtype)


def activations(M: int, K: int, seed: int, scale_div: float = 1.0, device="cpu",
                row_pad: int = 0) -> torch.Tensor:
    """bf16 randn[M, K] / scale_div.  row_pad > 0 returns a strided view of a
    [M, K + row_pad] buffer (non-contiguous rows)."""
    x = randn((M, K + row_pad), seed, device=device) / scale_div
    x = x.to(torch.bfloat16)
    return x[:, :K] if row_pad else x


# --------------------------------------------------------------- weights

def per_tensor_fp8_problem(M=97, N=224, K=576, seed=0, bias=True):
    """The per-tensor W8A16 GEMM workload: A bf16 randn/10 [M,K], B = randn[N,K]
    cast to e4m3, scale 0.01 (0-d fp32), fp32 bias randn[N]."""
    g = _gen(seed)
    a = (torch.randn(M, K, generator=g) / 10).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(FP8)
    scale = torch.tensor(0.01, dtype=torch.float32)
    b = torch.randn(N, generator=g, dtype=torch.float32) if bias else None
    return a, w, scale, b


def block_fp8_weight(N: int, K: int, block_n: int, seed: int, std: float = 0.05,
                     device="cpu", block_k: int = 128):
    """W e4m3 [N, K] and fp32 scales [ceil(N/block_n), ceil(K/block_k)] from
    randn * std, one scale amax/448 per [block_n, block_k] block."""
    w = randn((N, K), seed, device=device) * std
    return _quantize_blocks(w, block_n, block_k)


def _quantize_blocks(w: torch.Tensor, block_n: int, block_k: int):
    N, K = w.shape
    nb, kb = -(-N // block_n), -(-K // block_k)
    pad = torch.zeros(nb * block_n, kb * block_k, dtype=torch.float32, device=w.device)
    pad[:N, :K] = w
    blocks = pad.view(nb, block_n, kb, block_k)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.clamp(amax, min=1e-10) / 448.0
    q = (blocks / scale[:, None, :, None]).clamp(-448.0, 448.0).to(FP8)
    q = q.view(nb * block_n, kb * block_k)[:N, :K].contiguous()
    return q, scale.contiguous()


def moe_fp8_weights(E: int, N: int, K: int, seed: int, std: float = 0.05, device="cpu"):
    """w1 e4m3 [E, 2N, K] + fp32 [E, ceil(2N/128), ceil(K/128)];
    w2 e4m3 [E, K, N] + fp32 [E, ceil(K/128), ceil(N/128)]."""
    w1 = torch.empty(E, 2 * N, K, dtype=FP8, device=device)
    w2 = torch.empty(E, K, N, dtype=FP8, device=device)
    s1 = torch.empty(E, -(-2 * N // 128), -(-K // 128), dtype=torch.float32, device=device)
    s2 = torch.empty(E, -(-K // 128), -(-N // 128), dtype=torch.float32, device=device)
    g = _gen(seed, device)
    for e in range(E):
        a = torch.randn(2 * N, K, generator=g, device=device) * std
        w1[e], s1[e] = _quantize_blocks(a, 128, 128)
        b = torch.randn(K, N, generator=g, device=device) * std
        w2[e], s2[e] = _quantize_blocks(b, 128, 128)
    return w1, s1, w2, s2


# e2m1 magnitudes by code 0..7 (OCP Microscaling Formats v1.0, FP4 E2M1)
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _mx_quantize(x: torch.Tensor):
    """[R, C] fp32 -> packed e2m1 [R, C/2] uint8 and ue8m0 [R, C/32] uint8."""
    R, C = x.shape
    assert C % 32 == 0
    blocks = x.view(R, C // 32, 32)
    amax = blocks.abs().amax(dim=2)
    _, ex = torch.frexp(amax)                    # amax = f * 2^ex, f in [0.5, 1)
    shared = torch.where(amax > 0, ex - 1 - 2, torch.full_like(ex, -127))
    shared = shared.clamp(-127, 127)
    scale = torch.pow(2.0, shared.to(torch.float32))
    v = blocks / scale[:, :, None]
    mag = v.abs().clamp(max=6.0)
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], device=x.device)
    code = torch.bucketize(mag, mids, right=True)
    # exact midpoints go to the even code: 0.25->0, 1.25->2, 2.5->4, 5->6
    for i in (0, 2, 4, 6):
        code = torch.where(mag == mids[i], torch.full_like(code, i), code)
    sign = (v < 0) & (code > 0)
    nib = (code | (sign.to(code.dtype) << 3)).to(torch.uint8).view(R, C)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).contiguous()
    ue8m0 = (shared + 127).to(torch.uint8).contiguous()
    return packed, ue8m0


def moe_mxfp4_weights(E: int, N: int, K: int, seed: int, std: float = 0.05,
                      device="cpu"):
    """w1 e2m1x2 [E, 2N, K/2] + ue8m0 [E, 2N, K/32]; w2 [E, K, N/2] + [E, K, N/32]."""
    w1 = torch.empty(E, 2 * N, K // 2, dtype=torch.uint8, device=device)
    s1 = torch.empty(E, 2 * N, K // 32, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, K, N // 2, dtype=torch.uint8, device=device)
    s2 = torch.empty(E, K, N // 32, dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    for e in range(E):
        a = torch.randn(2 * N, K, generator=g, device=device) * std
        w1[e], s1[e] = _mx_quantize(a)
        b = torch.randn(K, N, generator=g, device=device) * std
        w2[e], s2[e] = _mx_quantize(b)
    return w1, s1, w2, s2


def moe_biases(E: int, N: int, K: int, seed: int, std: float = 0.01, device="cpu"):
    g = _gen(seed, device)
    b1 = torch.randn(E, 2 * N, generator=g, device=device) * std
    b2 = torch.randn(E, K, generator=g, device=device) * std
    return b1, b2


# --------------------------------------------------------------- routing

def routing_uniform(T: int, E: int, topk: int, seed: int):
    """softmax(randn[T, E]) top-k -> (weights fp32 [T,k], ids int32 [T,k])."""
    logits = torch.randn(T, E, generator=_gen(seed))
    p = torch.softmax(logits, dim=-1)
    w, ids = torch.topk(p, topk, dim=-1)
    return w.contiguous(), ids.to(torch.int32).contiguous()


def routing_zipf(T: int, E: int, topk: int, seed: int, s: float = 1.2):
    """Concentrated routing: expert popularity ~ rank^-s (random rank order),
    sampled without replacement through Gumbel noise; softmax top-k weights."""
    g = _gen(seed)
    ranks = torch.randperm(E, generator=g).to(torch.float32) + 1.0
    base = -s * torch.log(ranks)
    u = torch.rand(T, E, generator=g).clamp(1e-12, 1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    p = torch.softmax(base[None, :] + gumbel, dim=-1)
    w, ids = torch.topk(p, topk, dim=-1)
    return w.contiguous(), ids.to(torch.int32).contiguous()


def routing_blocks(block_sizes=(0, 4, 5, 33), topk: int = 8, E: int = 256):
    """Deterministic routes giving exact expert block sizes.

    Consecutive tokens are assigned to a "base" index b (b-th entry of
    block_sizes, repeated that many times); token t then uses experts
    (E // topk) * k + b for k = 0..topk-1, so expert (E//topk)*k + b receives
    exactly block_sizes[b] tokens and all other experts receive none.
    Weights are 1/topk.
    """
    stride = E // topk
    assert len(block_sizes) <= stride
    bases = []
    for b, n in enumerate(block_sizes):
        bases += [b] * n
    T = len(bases)
    ids = torch.tensor([[stride * k + b for k in range(topk)] for b in bases],
                       dtype=torch.int32).reshape(T, topk)
    w = torch.full((T, topk), 1.0 / topk, dtype=torch.float32)
    return w, ids


def distinct_experts(ids: torch.Tensor) -> int:
    return int(torch.unique(ids).numel())


def zipf_hint(E: int, s: float) -> float:
    """Share of the most popular expert under rank^-s popularity (for docs)."""
    h = sum(1.0 / math.pow(r, s) for r in range(1, E + 1))
    return 1.0 / h
