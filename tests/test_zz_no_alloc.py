"""mxq_fp8_scaled_mm_noalloc, the scaled GEMM for callers that cannot
allocate device memory (plugins handed only their buffers, frameworks whose
pools forbid raw cudaMalloc, serving loops that must not allocate after
start-up).  It keeps its split-K partials in a fixed array inside the library.

Called here through the C ABI and compared with mxq_fp8_scaled_mm (given a
workspace) on two calls in a row with different shapes and data, so a stale
array from the first call would show up in the second.  Both entry points run
the same split plan and reduce the partials in the same fixed order, so the
fp32 outputs must be bit-identical: that shows the split path really ran
from the library's array.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from mxfp4_quantized_gemm_token_gb300 import _lib, synth
from gpu_util import assert_bf16_close, bits16

pytestmark = pytest.mark.gpu

E4M3 = 3


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(lib, fn, q, s, w, ws, block_n, out, extra):
    M, K = q.shape
    N = w.shape[0]
    od = _lib.BF16 if out.dtype == torch.bfloat16 else _lib.F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [_p(q), E4M3, M, K, K, _p(s), s.stride(0), s.stride(1), _p(w), N, K, _p(ws), block_n,
            128, ws.stride(0), ws.stride(1), None, 0, _p(out), od, N]
    return getattr(lib, fn)(*(args + extra + [stream]))


def _problem(M, N, K, block_n, seed):
    import mxfp4_quantized_gemm_token_gb300 as mxq
    x = synth.activations(M, K, seed=seed, device="cuda")
    w, ws = synth.block_fp8_weight(N, K, block_n, seed=seed + 1, device="cuda")
    q, s = mxq.per_token_group_quant_fp8(x)
    return q, s, w, ws


def _need(lib, M, N, K, block_n):
    need = ctypes.c_size_t(0)
    assert lib.mxq_fp8_scaled_mm_workspace_size(M, N, K, E4M3, block_n, 128,
                                                ctypes.byref(need)) == 0
    return need.value


def _compare(lib, q, s, w, ws, bn, need):
    M, N = q.shape[0], w.shape[0]
    work = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    for dt in (torch.float32, torch.bfloat16):
        ref = torch.empty((M, N), dtype=dt, device="cuda")
        got = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        assert _call(lib, "mxq_fp8_scaled_mm", q, s, w, ws, bn, ref,
                     [_p(work) if need else None, need]) == 0, lib.mxq_last_error()
        assert _call(lib, "mxq_fp8_scaled_mm_noalloc", q, s, w, ws, bn, got, []) == 0, \
            lib.mxq_last_error()
        torch.cuda.synchronize()
        if dt == torch.float32:
            assert torch.equal(got, ref)
        else:
            assert_bf16_close(got, bits16(ref))


def test_noalloc_matches_workspace_entry_point_twice():
    lib = _lib.load()
    for (M, N, K, bn, seed) in [(8, 4096, 7168, 128, 1), (3, 2048, 4096, 1, 2)]:
        q, s, w, ws = _problem(M, N, K, bn, seed)
        need = _need(lib, M, N, K, bn)
        assert 0 < need <= _lib.NOALLOC_SCRATCH_BYTES      # this shape uses the scratch
        _compare(lib, q, s, w, ws, bn, need)


def test_noalloc_accepts_per_row_weight_scales_at_large_m():
    """[1, 128] weight scales at M = 512, N = 4608: the call's own plan needs
    no split here, so no scratch is needed and the shape is accepted."""
    lib = _lib.load()
    M, N, K = 512, 4608, 7168
    q, s, w, ws = _problem(M, N, K, 1, 5)
    need = _need(lib, M, N, K, 1)
    assert need <= _lib.NOALLOC_SCRATCH_BYTES
    _compare(lib, q, s, w, ws, 1, need)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    q, s, w, ws = _problem(128, 4096, 4096, 128, 3)
    out = torch.empty((128, 4096), dtype=torch.bfloat16, device="cuda")
    try:
        assert lib.mxq_set_option(_lib.OPT_SPLIT_K, 16) == 0     # 16 x 128 x 4096 x 4 B = 32 MiB
        rc = _call(lib, "mxq_fp8_scaled_mm_noalloc", q, s, w, ws, 128, out, [])
    finally:
        lib.mxq_set_option(_lib.OPT_SPLIT_K, 0)
    assert rc == _lib.ERR_UNSUPPORTED
    assert b"scratch" in lib.mxq_last_error()
