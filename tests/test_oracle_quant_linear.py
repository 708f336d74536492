"""Pins of the oracle's activation quantization and scaled GEMM.

Quantization: invariants fixed by the definition (group max maps to 448,
half-ulp error bound, zero group, signed zero).  GEMM: exact integer
arithmetic, the per-tensor == constant-block-scale identity, special cases
that reduce to a copy or a column selection, agreement with a library fp64
matmul of the dequantised operands (the pages' own reference formula), and
bit-identical results under a scale-storage layout change.
"""
import numpy as np
import pytest
import torch

from mxfp4_quantized_gemm_token_gb300 import synth

BF16, E4M3 = 1, 3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def e4m3_lib(codes: np.ndarray) -> np.ndarray:
    """Library decode (torch CPU cast), independent of the oracle's decoder."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


# ------------------------------------------------------------ quantization

@pytest.mark.parametrize("scale", [1.0, 1e-3, 37.0])
def test_group_quant_invariants(oracle, scale):
    x = (torch.randn(7, 640, generator=torch.Generator().manual_seed(3)) * scale).to(torch.bfloat16)
    q, s = oracle.per_token_group_quant_fp8(bits(x), 128)
    assert s.shape == (7, 5)
    xf = x.float().numpy().astype(np.float64)
    qd = e4m3_lib(q)
    for m in range(7):
        for g in range(5):
            sl = slice(g * 128, (g + 1) * 128)
            amax = np.abs(xf[m, sl]).max()
            # the scale is the fp32 quotient amax / 448
            assert s[m, g] == np.float32(np.float32(amax) / np.float32(448.0))
            # the group maximum lands exactly on the largest finite code
            assert np.abs(qd[m, sl]).max() == 448.0
            # each code is the nearest e4m3 value to x/s: error <= half the
            # spacing of e4m3 at that magnitude (1/16 relative, 2^-10 absolute
            # in the subnormal range), with a little room for the fp32 quotient
            t = xf[m, sl] / np.float64(s[m, g])
            ulp = np.where(np.abs(t) >= 2.0 ** -6,
                           2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 1e-30))) - 3),
                           2.0 ** -9)
            assert np.all(np.abs(qd[m, sl] - t) <= ulp / 2 * (1 + 1e-6) + 1e-7 * np.abs(t))


def test_group_quant_zero_group_and_signed_zero(oracle):
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    x[1, 128:] = torch.randn(128).to(torch.bfloat16)
    x[1, 130] = -0.0
    q, s = oracle.per_token_group_quant_fp8(bits(x), 128)
    assert s[0, 0] == np.float32(np.float32(1e-10) / np.float32(448.0))
    assert np.all(q[0] == 0)
    assert q[1, 130] == 0x80
    # a ragged last group (K not a multiple of 128)
    y = torch.randn(3, 200, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    q, s = oracle.per_token_group_quant_fp8(bits(y), 128)
    assert s.shape == (3, 2)
    assert np.abs(e4m3_lib(q[:, 128:])).max(axis=1).tolist() == [448.0] * 3


# ------------------------------------------------------------ scaled GEMM

def test_block_partials_exact_against_integer_arithmetic(oracle):
    """e4m3 x e4m3 products are integers times 2^-18: with unit scales the
    fp64 accumulator must equal an int64 computation exactly."""
    g = torch.Generator().manual_seed(5)
    M, N, K = 5, 9, 384
    qa = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    qw = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x3C   # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x41
    ia = np.rint(e4m3_lib(qa.numpy()) * 512).astype(np.int64)
    iw = np.rint(e4m3_lib(qw.numpy()) * 512).astype(np.int64)
    exact = ia @ iw.T                     # units of 2^-18
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    acc = oracle.scaled_mm_at(qa.numpy(), E4M3, np.ones((M, 3), np.float32), qw.numpy(),
                              np.ones((1, 3), np.float32), 128, 128, None,
                              ms.ravel(), ns.ravel())
    assert np.array_equal(acc, exact.ravel().astype(np.float64) * 2.0 ** -18)


def test_per_tensor_equals_constant_block_scales(oracle):
    a, w, scale, bias = synth.per_tensor_fp8_problem(M=11, N=224, K=512, seed=2)
    wq = bits_u8(w)
    f_pt, b_pt = oracle.scaled_mm(bits(a), BF16, None, wq, np.float32(0.01), 0, 0, bias.numpy())
    blocks = np.full((2, 4), 0.01, np.float32)
    f_bl, b_bl = oracle.scaled_mm(bits(a), BF16, None, wq, blocks, 128, 128, bias.numpy())
    assert np.allclose(f_pt, f_bl, rtol=1e-6, atol=0)
    # and with 1x128 weight blocks
    f_r, _ = oracle.scaled_mm(bits(a), BF16, None, wq, np.full((224, 4), 0.01, np.float32),
                              1, 128, bias.numpy())
    assert np.array_equal(f_r, f_bl)


def bits_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def test_identity_weight_reproduces_activation(oracle):
    K = 256
    qa = torch.randn(6, K, generator=torch.Generator().manual_seed(9)).to(torch.float8_e4m3fn)
    w = torch.zeros(K, K)
    w.fill_diagonal_(1.0)
    wq = bits_u8(w.to(torch.float8_e4m3fn))
    f, _ = oracle.scaled_mm(bits_u8(qa), E4M3, np.ones((6, 2), np.float32), wq,
                            np.ones((2, 2), np.float32), 128, 128)
    assert np.array_equal(f.astype(np.float64), e4m3_lib(bits_u8(qa)))


def test_one_hot_activation_selects_scaled_column(oracle):
    N, K = 256, 384
    wq, ws = synth.block_fp8_weight(N, K, 128, seed=4)
    a = torch.zeros(3, K)
    a[0, 5] = 1.0
    a[1, 200] = 2.0
    a[2, 383] = -0.5
    qa = bits_u8(a.to(torch.float8_e4m3fn))
    a_s = np.full((3, 3), 0.25, np.float32)
    f, _ = oracle.scaled_mm(qa, E4M3, a_s, bits_u8(wq), ws.numpy(), 128, 128)
    wd = e4m3_lib(bits_u8(wq))
    wsn = ws.numpy().astype(np.float64)
    for m, (k, v) in enumerate([(5, 1.0), (200, 2.0), (383, -0.5)]):
        col = wd[:, k] * wsn[np.arange(N) // 128, k // 128] * v * 0.25
        assert np.array_equal(f[m].astype(np.float64), col.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("block_n", [128, 1])
def test_block_gemm_matches_library_matmul_of_dequantised(oracle, block_n):
    """The pages' reference: dequantise both operands, then matmul (here a
    torch fp64 matmul; the oracle applies scales per 128-wide slice)."""
    M, N, K = 16, 256, 256
    g = torch.Generator().manual_seed(11)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    q, s = oracle.per_token_group_quant_fp8(bits(x), 128)
    wq, ws = synth.block_fp8_weight(N, K, block_n, seed=12)
    bias = torch.randn(N, generator=g).to(torch.bfloat16)
    f, b = oracle.scaled_mm(q, E4M3, s, bits_u8(wq), ws.numpy(), block_n, 128, bits(bias))
    a_deq = e4m3_lib(q) * np.repeat(s.astype(np.float64), 128, axis=1)
    w_deq = e4m3_lib(bits_u8(wq)) * np.repeat(np.repeat(ws.numpy().astype(np.float64),
                                                        block_n, axis=0), 128, axis=1)[:N]
    ref = torch.from_numpy(a_deq) @ torch.from_numpy(w_deq).T + bias.double()
    assert np.allclose(f, ref.numpy(), rtol=1e-6, atol=1e-6)
    # bf16 output is the library's rounding of the fp32 result
    assert np.array_equal(b, bits(torch.from_numpy(f).to(torch.bfloat16)))


def test_scale_layout_change_is_bit_identical(oracle):
    """Transposed-contiguous scale storage must not change a single bit
    ("[XPU] block-FP8 linear" numerical test, post-load layout, rtol=atol=0)."""
    M, N, K = 16, 256, 256
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
    q, s = oracle.per_token_group_quant_fp8(bits(x), 128)
    wq = bits_u8(torch.randn(N, K).to(torch.float8_e4m3fn))
    ws = (torch.rand(N // 128, K // 128, generator=torch.Generator().manual_seed(14)) + 0.1).numpy()
    f0, b0 = oracle.scaled_mm(q, E4M3, s, wq, ws, 128, 128)
    f1, b1 = oracle.scaled_mm(q, E4M3, s, wq, ws, 128, 128, w_scale_col_major=True)
    assert np.array_equal(f0, f1) and np.array_equal(b0, b1)


@pytest.mark.parametrize("M,N,K", [(1, 128, 512), (11, 224, 576), (97, 224, 576)])
def test_per_tensor_matches_page_reference_formula(oracle, M, N, K):
    """"[CPU] fp8_per_tensor_scaled_mm_cpu" test: ref = matmul(data.float(),
    weight.float().T) * scale + bias, then bf16 (torch fp64 here)."""
    a, w, scale, bias = synth.per_tensor_fp8_problem(M=M, N=N, K=K, seed=M)
    f, b = oracle.scaled_mm(bits(a), BF16, None, bits_u8(w), scale.numpy(), 0, 0, bias.numpy())
    ref = (a.double() @ w.double().T) * float(scale) + bias.double()
    assert np.allclose(f, ref.numpy(), rtol=1e-6, atol=1e-6)
    ref16 = ref.float().to(torch.bfloat16).float().numpy()
    got16 = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.allclose(got16, ref16, rtol=1e-2, atol=1e-2)
