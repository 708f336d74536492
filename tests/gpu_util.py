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


def moe_stage_probes(oracle, wtype, x_bits, ids, tw, expert, act, y, h, slots):
    """The two fp32 stage accumulators of the fused MoE at the given slots
    (slot = t*topk + k), each against the oracle's per-expert GEMM fed with
    the GPU's own stage input, at the fp32 accumulator tolerance:
        h[slot] = x[t] . W1[e]^T                 (before the bias)
        y[slot] = w[slot] * (act[slot] . W2[e]^T + b2[e])
    x_bits: bf16 bits [T, K]; ids / tw: [T, topk] (CPU); act, y, h: GPU
    checkpoints in slot order; expert(e) -> (w1, s1, w2, s2, b2) of expert e
    alone as numpy arrays with a leading dimension of one (b2 may be None)."""
    ids_f = np.asarray(ids).reshape(-1)
    tw_f = np.asarray(tw, np.float64).reshape(-1)
    topk = np.asarray(ids).shape[1]
    slots = np.asarray(sorted(slots), np.int64)
    sl_t = torch.from_numpy(slots).to(act.device)
    act_b = bits16(act[sl_t])
    h_g = h[sl_t].double().cpu().numpy()
    y_g = y[sl_t].double().cpu().numpy()
    h_r = np.empty_like(h_g)
    y_r = np.empty_like(y_g)
    for e in np.unique(ids_f[slots]):
        sel = np.nonzero(ids_f[slots] == e)[0]
        w1, s1, w2, s2, b2 = expert(int(e))
        h_r[sel] = oracle.expert_linear(x_bits[slots[sel] // topk], wtype, w1, s1, 0)
        z = oracle.expert_linear(act_b[sel], wtype, w2, s2, 0)
        if b2 is not None:
            z = z + np.asarray(b2, np.float64).reshape(1, -1)
        y_r[sel] = tw_f[slots[sel]].reshape(-1, 1) * z
    assert_probe_close(h_g, h_r, what="stage-1 accumulator h")
    assert_probe_close(y_g, y_r, what="stage-2 accumulator y")
