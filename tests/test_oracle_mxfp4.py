"""Pins of the oracle's MXFP4 quantizer (the OCP MX conversion rule).

- a hand-derived block covering every tie and the saturation
  (tests/golden/mxfp4_ocp_rounding_block.txt);
- the shared-exponent rule at its edges (powers of two, just below them, an
  all-zero block, the lower clamp);
- brute force: each element decodes to a nearest point of its block's scaled
  E2M1 grid, ties to the even code;
- an independent implementation (the input generator's torch restatement of
  the same rule) gives the same values."""
import os

import numpy as np
import pytest
import torch

from mxfp4_quantized_gemm_token_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nibbles(packed):
    p = np.asarray(packed)
    return np.stack([p & 15, p >> 4], axis=-1).reshape(p.shape[0], -1)


def decode(packed, scales):
    nib = nibbles(packed)
    v = MAG[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    return v * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)


def test_golden_block(oracle):
    vals, codes = [], []
    with open(os.path.join(GOLDEN, "mxfp4_ocp_rounding_block.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v, c = line.split()[:2]
            vals.append(float(v))
            codes.append(int(c))
    assert len(vals) == 32
    packed, scales = oracle.mxfp4_quantize(np.array([vals], np.float32))
    assert scales.tolist() == [[127]]
    assert nibbles(packed)[0].tolist() == codes


@pytest.mark.parametrize("amax,byte", [(1.0, 125), (0.99, 124), (6.0, 127), (8.0, 128),
                                       (2.0 ** -130, 0), (0.0, 0), (3.0e38, 252)])
def test_shared_exponent_edges(oracle, amax, byte):
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = amax
    x[0, 6] = -amax / 3
    packed, scales = oracle.mxfp4_quantize(x)
    assert scales[0, 0] == byte
    if amax > 0:
        got = decode(packed, scales)[0]
        assert got[5] == pytest.approx(min(6.0, amax / 2.0 ** (byte - 127)) * 2.0 ** (byte - 127),
                                       rel=0.25)


def test_nearest_point_brute_force(oracle):
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(64, 256, generator=g) * torch.exp(torch.randn(64, 1, generator=g) * 3)).numpy()
    x[3, :32] = 0.0
    packed, scales = oracle.mxfp4_quantize(x)
    nib = nibbles(packed)
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            sc = 2.0 ** (int(scales[r, b]) - 127)
            amax = np.abs(x[r, b * 32:(b + 1) * 32]).max()
            if amax > 0:
                assert sc == 2.0 ** (np.floor(np.log2(np.float64(amax))) - 2)
            for i in range(32):
                v = float(x[r, b * 32 + i]) / sc
                code = int(nib[r, b * 32 + i])
                d = np.abs(np.abs(v) - MAG)
                best = d.min()
                assert d[code & 7] == best or (abs(v) > 6.0 and code & 7 == 7)
                if (d == best).sum() > 1 and abs(v) <= 6.0:
                    assert (code & 1) == 0                      # tie -> even code
                assert (code >> 3) == (1 if np.signbit(v) else 0)


def test_agrees_with_independent_torch_restatement(oracle):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(96, 2880, generator=g) * 0.05
    packed, scales = oracle.mxfp4_quantize(x.numpy())
    p2, s2 = synth._mx_quantize(x)
    assert np.array_equal(scales, s2.numpy())
    assert np.array_equal(decode(packed, scales), decode(p2.numpy(), s2.numpy()))
