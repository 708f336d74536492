"""Helpers shared by the GPU parity tests: host copies as raw bits and the
tolerances the parity contract states.

bf16 outputs: |g - r| <= 1e-2 + 1e-2 |r| (rtol = atol = 1e-2 after bf16).
fp32 accumulator probe: |g - r| <= 1e-3 (|r| + 1e-2 max_n |r[m, :]|), i.e.
1e-3 relative with a row-relative floor so that cancellation near zero does
not fail a correct kernel.
"""
import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def bf16_values(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, np.float64)


def assert_bf16_close(got, ref_bits, rtol=1e-2, atol=1e-2, what="output"):
    g = _np(got)
    r = bf16_values(ref_bits) if ref_bits.dtype == np.uint16 else np.asarray(ref_bits, np.float64)
    bad = ~(np.abs(g - r) <= atol + rtol * np.abs(r))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d outside tolerance, e.g. at %s: got %s ref %s" % (
            what, bad.sum(), bad.size, idx.tolist(), g[tuple(idx.T)], r[tuple(idx.T)]))


def assert_probe_close(got, ref, rel=1e-3, floor=1e-2, what="fp32 accumulator"):
    g = _np(got)
    r = np.asarray(ref, np.float64)
    rowmax = np.abs(r).max(axis=-1, keepdims=True) if r.ndim == 2 else np.abs(r).max()
    bad = ~(np.abs(g - r) <= rel * (np.abs(r) + floor * rowmax))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d outside tolerance, e.g. at %s: got %s ref %s" % (
            what, bad.sum(), bad.size, idx.tolist(), g[tuple(idx.T)], r[tuple(idx.T)]))


def assert_sampled_close(got, ref, rowmax, rel=1e-3, floor=1e-2, what="sampled accumulator"):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    bad = ~(np.abs(g - r) <= rel * (np.abs(r) + floor * np.asarray(rowmax, np.float64)))
    if bad.any():
        i = np.nonzero(bad)[0][:5]
        raise AssertionError("%s: %d of %d outside tolerance, e.g. got %s ref %s" % (
            what, bad.sum(), bad.size, g[i], r[i]))
