"""Pins of the oracle's expert alignment and fused MoE.

moe_align: a hand-derived golden case (the small-block routes of the vLLM
CPU MoE page), an independent brute force (sort of (expert, slot) pairs) and
structural invariants.  fused MoE: reduction to a dense MLP computed with a
library fp64 matmul of dequantised weights (topk = 1 and E = 1), an
independent numpy decode of MXFP4 (nibble order and scale indexing), expert
permutation invariance and linearity in the routing weights.
"""
import os

import numpy as np
import pytest
import torch

from mxfp4_quantized_gemm_token_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
W_FP8, W_MX = 1, 2


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.contiguous().view(torch.uint8).numpy()


def bf16_of(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def read_golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            d[k] = [int(x) for x in v]
    return d


# ------------------------------------------------------------- align

def test_align_golden_blocks_4_5_33(oracle):
    g = read_golden("moe_align_blocks_4_5_33.txt")
    ids = np.array(g["topk_ids"], np.int32).reshape(-1, g["topk"][0])
    sid, eid, off, nb = oracle.moe_align(ids, g["E"][0], g["block_m"][0], g["cap"][0])
    BM = g["block_m"][0]
    assert nb == g["num_blocks"][0]
    assert eid.tolist() == g["expert_ids"]
    assert off.tolist() == g["offsets"]
    for b in range(nb):
        rows = g["block%d" % b]
        assert sid[b * BM: b * BM + len(rows)].tolist() == rows
        assert np.all(sid[b * BM + len(rows): (b + 1) * BM] == g["pad"][0])
    assert np.all(sid[nb * BM:] == g["pad"][0])


def brute_align(ids, E, BM, cap):
    S = ids.size
    flat = ids.ravel()
    pairs = sorted((int(flat[s]), s) for s in range(S))
    sid = np.full(cap * BM, S, np.int32)
    eid = np.full(cap, -1, np.int32)
    off = np.full(cap + 1, S, np.int32)
    b, i = 0, 0
    off[0] = 0
    while i < S:
        e = pairs[i][0]
        j = i
        while j < S and pairs[j][0] == e:
            j += 1
        for c0 in range(i, j, BM):
            c1 = min(c0 + BM, j)
            eid[b] = e
            off[b] = c0
            sid[b * BM: b * BM + (c1 - c0)] = [p[1] for p in pairs[c0:c1]]
            off[b + 1] = c1
            b += 1
        i = j
    return sid, eid, off, b


@pytest.mark.parametrize("T,topk,E,BM,kind", [
    (1, 4, 128, 16, "uniform"), (37, 8, 256, 64, "uniform"), (64, 4, 128, 32, "zipf"),
    (300, 8, 256, 128, "zipf"), (5, 2, 3, 16, "uniform")])
def test_align_matches_brute_force_and_invariants(oracle, T, topk, E, BM, kind):
    if kind == "uniform":
        _, ids = synth.routing_uniform(T, E, topk, seed=T)
    else:
        _, ids = synth.routing_zipf(T, E, topk, seed=T)
    ids = ids.numpy()
    S = T * topk
    cap = oracle.align_capacity(S, E, BM)
    got = oracle.moe_align(ids, E, BM, cap)
    ref = brute_align(ids, E, BM, cap)
    for a, b in zip(got[:3], ref[:3]):
        assert np.array_equal(a, b)
    assert got[3] == ref[3]
    sid, eid, off, nb = got
    valid = np.concatenate([sid[b * BM: b * BM + off[b + 1] - off[b]] for b in range(nb)])
    assert np.array_equal(np.sort(valid), np.arange(S))          # a permutation
    for b in range(nb):
        rows = sid[b * BM: b * BM + off[b + 1] - off[b]]
        assert np.all(ids.ravel()[rows] == eid[b])
        assert 0 < off[b + 1] - off[b] <= BM
    assert off[nb] == S and nb <= cap


# ------------------------------------------------------------- fused MoE

def deq_fp8(w, s):
    """[E, R, C] e4m3 with [E, ceil(R/128), ceil(C/128)] scales -> fp64."""
    wd = torch.from_numpy(u8(w)).view(torch.float8_e4m3fn).double()
    E, R, C = wd.shape
    sc = s.double().repeat_interleave(128, 1).repeat_interleave(128, 2)[:, :R, :C]
    return wd * sc


def deq_mx(w, s):
    """Independent numpy MXFP4 decode: OCP table lookup, low nibble first."""
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            table[int(c)] = float(v)
    lut = np.array([table[c] for c in range(16)])
    p = u8(w)
    lo, hi = p & 15, p >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(p.shape[0], p.shape[1], p.shape[2] * 2)
    vals = lut[nib]
    sc = np.ldexp(1.0, u8(s).astype(np.int64) - 127)
    return torch.from_numpy(vals * np.repeat(sc, 32, axis=2))


def dense_mlp(x, W1, b1, W2, b2, N):
    """Library fp64 matmuls of dequantised weights: bf16(silu(g)*u) between."""
    h = x.double() @ W1.T
    if b1 is not None:
        h = h + b1.double()
    g, u = h[:, :N], h[:, N:]
    act = (g / (1 + torch.exp(-g)) * u).float().to(torch.bfloat16)
    z = act.double() @ W2.T
    if b2 is not None:
        z = z + b2.double()
    return act, z


@pytest.mark.parametrize("wtype", [W_FP8, W_MX])
def test_topk1_reduces_to_dense_mlp(oracle, wtype):
    E, N, K, T = 3, 128, 256, 6
    if wtype == W_FP8:
        w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=1)
        W1, W2 = deq_fp8(w1, s1), deq_fp8(w2, s2)
        b1 = b2 = None
    else:
        w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=1)
        W1, W2 = deq_mx(w1, s1), deq_mx(w2, s2)
        b1, b2 = synth.moe_biases(E, N, K, seed=2)
    x = synth.activations(T, K, seed=3, scale_div=10)
    ids = torch.tensor([[0], [2], [1], [2], [0], [0]], dtype=torch.int32)
    tw = torch.ones(T, 1)
    out, act, z = oracle.fused_experts(
        bits(x), wtype, u8(w1), u8(s1) if wtype == W_MX else s1.numpy(),
        None if b1 is None else b1.numpy(), u8(w2), u8(s2) if wtype == W_MX else s2.numpy(),
        None if b2 is None else b2.numpy(), tw.numpy(), ids.numpy(), N, checkpoints=True)
    for t in range(T):
        e = int(ids[t, 0])
        ra, rz = dense_mlp(x[t:t + 1], W1[e], None if b1 is None else b1[e], W2[e],
                           None if b2 is None else b2[e], N)
        ga = bf16_of(act[t]).float()
        # act may differ by one bf16 step where fp64 summation order puts a
        # value on the other side of a rounding boundary
        assert torch.allclose(ga, ra.float()[0], rtol=2 ** -7, atol=1e-6)
        assert np.allclose(z[t], rz.numpy()[0], rtol=2e-2, atol=1e-4)
        ref = rz.float().to(torch.bfloat16).float()[0]
        assert torch.allclose(bf16_of(out[t]).float(), ref, rtol=1e-2, atol=1e-2)


def test_mxfp4_nibble_order_and_scale_indexing(oracle):
    """E = 1, topk = 1: out must equal the dense MLP built from the numpy
    decode; flipping the nibble order in the weights must change it."""
    E, N, K, T = 1, 128, 128, 3
    w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=7)
    x = synth.activations(T, K, seed=8, scale_div=10)
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)
    out, act, z = oracle.fused_experts(bits(x), W_MX, u8(w1), u8(s1), None, u8(w2), u8(s2),
                                       None, tw, ids, N, checkpoints=True)
    _, rz = dense_mlp(x, deq_mx(w1, s1)[0], None, deq_mx(w2, s2)[0], None, N)
    assert np.allclose(z, rz.numpy(), rtol=2e-2, atol=1e-4)
    swapped = ((u8(w1) & 15) << 4) | (u8(w1) >> 4)
    out2 = oracle.fused_experts(bits(x), W_MX, swapped.astype(np.uint8), u8(s1), None, u8(w2),
                                u8(s2), None, tw, ids, N)
    assert not np.array_equal(out, out2)


def test_expert_permutation_invariance_and_weight_linearity(oracle):
    E, N, K, T, topk = 4, 128, 128, 5, 2
    w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=21)
    x = synth.activations(T, K, seed=22, scale_div=10)
    tw, ids = synth.routing_uniform(T, E, topk, seed=23)
    base = oracle.fused_experts(bits(x), W_FP8, u8(w1), s1.numpy(), None, u8(w2), s2.numpy(),
                                None, tw.numpy(), ids.numpy(), N)
    perm = torch.tensor([2, 0, 3, 1])                 # new index of old expert e
    inv = torch.argsort(perm)
    pw1, ps1, pw2, ps2 = w1[inv], s1[inv], w2[inv], s2[inv]
    pids = perm[ids.long()].to(torch.int32)
    got = oracle.fused_experts(bits(x), W_FP8, u8(pw1), ps1.numpy(), None, u8(pw2),
                               ps2.numpy(), None, tw.numpy(), pids.numpy(), N)
    assert np.array_equal(base, got)
    twice = oracle.fused_experts(bits(x), W_FP8, u8(w1), s1.numpy(), None, u8(w2), s2.numpy(),
                                 None, (2 * tw).numpy(), ids.numpy(), N)
    assert torch.equal(bf16_of(twice).float(), 2 * bf16_of(base).float())


@pytest.mark.parametrize("wtype,topk,E", [(W_FP8, 2, 3), (W_MX, 2, 4), (W_FP8, 8, 10),
                                          (W_MX, 8, 9)])
def test_topk_combine_matches_weighted_dense_mlps(oracle, wtype, topk, E):
    """topk > 1 with deliberately unequal routing weights: every checkpoint row
    at slot t*topk + k must be the dense MLP of token t through expert
    ids[t, k], and the output must be sum_k w[t, k] * z_(t,k) in ascending k.
    The reference is built from library fp64 matmuls of independently
    dequantised weights, so a transposed weight index (w[k*T + t]) or a
    token-major / expert-major slot mix-up in act or z fails it."""
    N, K, T = 128, 256, 5
    if wtype == W_FP8:
        w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=31)
        W1, W2 = deq_fp8(w1, s1), deq_fp8(w2, s2)
        b1 = b2 = None
        sc = lambda s: s.numpy()
    else:
        w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=31)
        W1, W2 = deq_mx(w1, s1), deq_mx(w2, s2)
        b1, b2 = synth.moe_biases(E, N, K, seed=32)
        sc = u8
    x = synth.activations(T, K, seed=33, scale_div=10)
    g = torch.Generator().manual_seed(34)
    ids = torch.stack([torch.randperm(E, generator=g)[:topk] for _ in range(T)]).to(torch.int32)
    base = (torch.tensor([0.7, 0.2, 0.1]) if topk == 2 else
            torch.tensor([0.31, 0.22, 0.15, 0.11, 0.09, 0.07, 0.04, 0.01]))
    tw = torch.stack([base[torch.randperm(base.numel(), generator=g)][:topk] * (1 + 0.5 * t)
                      for t in range(T)]).float()
    out, act, z = oracle.fused_experts(
        bits(x), wtype, u8(w1), sc(s1), None if b1 is None else b1.numpy(), u8(w2), sc(s2),
        None if b2 is None else b2.numpy(), tw.numpy(), ids.numpy(), N, checkpoints=True)
    for t in range(T):
        o = torch.zeros(K, dtype=torch.float64)
        for k in range(topk):
            e, slot = int(ids[t, k]), t * topk + k
            ra, _ = dense_mlp(x[t:t + 1], W1[e], None if b1 is None else b1[e], W2[e],
                              None if b2 is None else b2[e], N)
            ga = bf16_of(act[slot]).double()
            # act: one bf16 step of freedom where the fp64 summation order
            # lands on the other side of a rounding boundary
            assert torch.allclose(ga, ra.double()[0], rtol=2 ** -7, atol=1e-6), (t, k)
            # z from the oracle's own act row: only summation order differs
            rz = ga @ W2[e].T + (0 if b2 is None else b2[e].double())
            assert np.allclose(z[slot], rz.numpy(), rtol=1e-9, atol=1e-12), (t, k)
            o += float(tw[t, k]) * rz
        ref = o.float().to(torch.bfloat16).float()
        assert torch.equal(bf16_of(out[t]).float(), ref), t


@pytest.mark.parametrize("wtype", [W_FP8, W_MX])
def test_expert_linear_matches_dequantised_matmul(oracle, wtype):
    """The per-expert GEMM (the stage accumulators h and z without bias)
    against a library fp64 matmul of independently dequantised weights, for
    every expert, with ragged 128-blocks in both dimensions (FP8)."""
    E, R, C, M = 3, 320 if wtype == W_FP8 else 192, 384 if wtype == W_FP8 else 288, 4
    if wtype == W_FP8:
        w1, s1, _, _ = synth.moe_fp8_weights(E, R // 2, C, seed=41)
        W = deq_fp8(w1, s1)
        sc = s1.numpy()
    else:
        w1, s1, _, _ = synth.moe_mxfp4_weights(E, R // 2, C, seed=41)
        W = deq_mx(w1, s1)
        sc = u8(s1)
    x = synth.activations(M, C, seed=42, scale_div=10)
    for e in range(E):
        got = oracle.expert_linear(bits(x), wtype, u8(w1), sc, e)
        ref = (x.double() @ W[e].T).numpy()
        assert got.shape == (M, R)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-15), e
