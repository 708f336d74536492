"""Pins of the oracle's format codecs against things other than itself:
library casts (torch CPU), closed forms and the OCP table (golden file)."""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_decode_all_codes_match_library(oracle):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(lib)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    # closed-form anchors: max normal, min normal, min subnormal
    assert mine[0x7E] == 448.0 and mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9


def test_e2m1_decode_matches_ocp_table(oracle):
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            table[int(c)] = float(v)
    mine = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    for c in range(16):
        assert mine[c] == table[c]
        assert math.copysign(1.0, mine[c]) == math.copysign(1.0, table[c])


def test_ue8m0_decode_closed_form_and_library(oracle):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.ue8m0_decode(codes)
    for e in range(255):
        assert mine[e] == math.ldexp(1.0, e - 127)
    assert math.isnan(mine[255])
    lib = torch.from_numpy(codes).view(torch.float8_e8m0fnu).float().double().numpy()
    assert np.array_equal(mine[:255], lib[:255]) and np.isnan(lib[255])


def test_bf16_round_matches_library_at_every_tie_and_neighbour(oracle):
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    f = bits.view(np.float32)
    finite = np.isfinite(f)
    f = f[finite]
    lib = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # the oracle's scalar entry point on a deterministic sample, plus every tie
    idx = np.arange(0, f.size, 97)
    ties = np.nonzero((f.view(np.uint32) & 0xFFFF) == 0x8000)[0][::5]
    idx = np.unique(np.concatenate([idx, ties]))
    mine = oracle.bf16_from_f32(f[idx])
    assert np.array_equal(mine, lib[idx])


def _encode_check_range(oracle, exp_lo, exp_hi):
    """All fp32 bit patterns with exponent field in [exp_lo, exp_hi] and
    |x| <= 448, both signs: the oracle's encoder vs torch's CPU cast."""
    mant = np.arange(1 << 23, dtype=np.uint32)
    for ef in range(exp_lo, exp_hi + 1):
        for sign in (0, 1):
            bits = (np.uint32(sign) << np.uint32(31)) | (np.uint32(ef) << np.uint32(23)) | mant
            f = bits.view(np.float32)
            f = f[np.abs(f) <= 448.0]
            if f.size == 0:
                continue
            lib = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            mine = oracle.e4m3_encode(f)
            bad = np.nonzero(mine != lib)[0]
            assert bad.size == 0, (ef, sign, f[bad[:5]], mine[bad[:5]], lib[bad[:5]])


def test_e4m3_encode_matches_library_exhaustive(oracle):
    """Every fp32 pattern with 2^-10 <= |x| <= 448 (exponent fields 117..135):
    the whole range where the e4m3 result is not simply +-0."""
    _encode_check_range(oracle, 117, 135)


def test_e4m3_encode_tiny_and_signed_zero(oracle):
    rng = np.random.default_rng(0)
    tiny = (rng.random(200000) * 2.0 ** -10).astype(np.float32)
    f = np.concatenate([tiny, -tiny, np.float32([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10)])])
    lib = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(f), lib)
    assert oracle.e4m3_encode(np.float32([-0.0]))[0] == 0x80
    assert oracle.e4m3_encode(np.float32([448.0, -448.0])).tolist() == [0x7E, 0xFE]
