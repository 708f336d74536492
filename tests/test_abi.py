"""The C-ABI library builds, loads, and exports every symbol include/mxq.h
declares; host-side argument validation returns its documented status codes
before touching any device (these calls need no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from mxfp4_quantized_gemm_token_gb300 import _lib
    return _lib.load()


def test_header_declares_the_four_ops_and_helpers():
    names = declared_functions()
    for op in ("mxq_fp8_scaled_mm", "mxq_per_token_group_quant_fp8", "mxq_moe_align_block",
               "mxq_fused_experts"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    from mxfp4_quantized_gemm_token_gb300 import _lib
    names = declared_functions()
    assert sorted(_lib.EXPORTED) == names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_options_roundtrip(lib):
    from mxfp4_quantized_gemm_token_gb300 import _lib
    assert b"sm_103a" in lib.mxq_version()
    v = ctypes.c_int64()
    assert lib.mxq_get_option(_lib.OPT_WAIT_BUDGET_NS, ctypes.byref(v)) == 0
    old = v.value
    assert lib.mxq_set_option(_lib.OPT_WAIT_BUDGET_NS, 12345) == 0
    assert lib.mxq_get_option(_lib.OPT_WAIT_BUDGET_NS, ctypes.byref(v)) == 0 and v.value == 12345
    assert lib.mxq_set_option(_lib.OPT_WAIT_BUDGET_NS, old) == 0
    assert lib.mxq_set_option(99, 1) == _lib.ERR_INVALID_ARG
    assert lib.mxq_set_option(_lib.OPT_FORCE_PATH, 4) == _lib.ERR_INVALID_ARG
    assert b"FORCE_PATH" in lib.mxq_last_error()
    assert lib.mxq_set_option(_lib.OPT_FORCE_PATH, 3) == 0       # one path per layer
    assert lib.mxq_set_option(_lib.OPT_FORCE_PATH, 0) == 0
    assert lib.mxq_set_option(_lib.OPT_NORMAL_TILE, 160) == _lib.ERR_INVALID_ARG
    assert b"NORMAL_TILE" in lib.mxq_last_error()
    assert lib.mxq_get_option(_lib.OPT_PDL, ctypes.byref(v)) == 0 and v.value == 1   # default on
    assert lib.mxq_set_option(_lib.OPT_PDL, 2) == _lib.ERR_INVALID_ARG
    assert lib.mxq_set_option(_lib.OPT_PDL, 0) == 0
    assert lib.mxq_set_option(_lib.OPT_PDL, 1) == 0


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first


def mm(lib, **kw):
    a = dict(A=FAKE, a_dtype=3, M=4, K=256, lda=256, a_scale=FAKE, sa0=2, sa1=1, W=FAKE, N=128,
             ldw=256, w_scale=FAKE, block_n=128, block_k=128, sw0=2, sw1=1, bias=None,
             bias_dtype=0, out=FAKE, out_dtype=1, ldo=128, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.mxq_fp8_scaled_mm(*a.values())


def test_scaled_mm_rejects_unsupported_block_sizes(lib):
    from mxfp4_quantized_gemm_token_gb300 import _lib
    # MXFP8 [1, 32] and other shapes are refused like the page's block_size check
    for bn, bk in [(1, 32), (64, 64), (128, 64), (2, 128), (0, 128), (128, 0)]:
        assert mm(lib, block_n=bn, block_k=bk) == _lib.ERR_UNSUPPORTED
    assert b"block size" in lib.mxq_last_error()


def test_scaled_mm_argument_errors(lib):
    from mxfp4_quantized_gemm_token_gb300 import _lib
    assert mm(lib, M=0) == _lib.OK                      # empty problem: nothing to do
    assert mm(lib, N=0) == _lib.OK
    assert mm(lib, K=0) == _lib.ERR_INVALID_ARG
    assert mm(lib, M=-1) == _lib.ERR_INVALID_ARG
    assert mm(lib, A=None) == _lib.ERR_INVALID_ARG
    assert mm(lib, a_scale=None) == _lib.ERR_INVALID_ARG   # W8A8 needs group scales
    assert mm(lib, a_dtype=1) == _lib.ERR_INVALID_ARG      # bf16 A takes no scale
    assert mm(lib, a_dtype=7) == _lib.ERR_UNSUPPORTED
    assert mm(lib, out_dtype=3) == _lib.ERR_UNSUPPORTED
    assert mm(lib, lda=100) == _lib.ERR_INVALID_ARG
    assert mm(lib, bias=FAKE, bias_dtype=3) == _lib.ERR_UNSUPPORTED
    assert mm(lib, lda=264) == _lib.ERR_UNSUPPORTED         # row stride not 16-byte multiple
    assert mm(lib, W=ctypes.c_void_p((1 << 20) + 8)) == _lib.ERR_UNSUPPORTED


def test_workspace_query_and_noalloc_validate_before_any_device_work(lib):
    """The split-K workspace query takes the block size the call will get and
    refuses the same illegal ones; the allocation-free GEMM reports a bad
    argument as itself (not as a scratch-size problem), whatever the shape."""
    from mxfp4_quantized_gemm_token_gb300 import _lib
    sz = ctypes.c_size_t(7)
    q = lib.mxq_fp8_scaled_mm_workspace_size
    assert q(4, 128, 256, 3, 1, 32, ctypes.byref(sz)) == _lib.ERR_UNSUPPORTED     # MXFP8 [1, 32]
    assert q(4, 128, 256, 7, 128, 128, ctypes.byref(sz)) == _lib.ERR_UNSUPPORTED   # a_dtype
    assert q(4, 128, 0, 3, 128, 128, ctypes.byref(sz)) == _lib.ERR_INVALID_ARG
    assert q(4, 128, 256, 3, 128, 128, None) == _lib.ERR_INVALID_ARG
    na = lib.mxq_fp8_scaled_mm_noalloc
    base = [FAKE, 3, 4096, 4096, 4096, FAKE, 32, 1, FAKE, 4096, 4096, FAKE, 128, 128, 32, 1,
            None, 0, FAKE, 1, 4096]
    for i, v, st in [(0, None, _lib.ERR_INVALID_ARG), (5, None, _lib.ERR_INVALID_ARG),
                     (12, 2, _lib.ERR_UNSUPPORTED), (19, 3, _lib.ERR_UNSUPPORTED)]:
        args = list(base)
        args[i] = v
        assert na(*args, None) == st
        assert b"scratch" not in lib.mxq_last_error()


def test_prepack_argument_errors(lib):
    """The prepack size query and the prepack refuse what the GEMM refuses,
    and bad pointers, before any device work."""
    from mxfp4_quantized_gemm_token_gb300 import _lib
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    q = lib.mxq_prepacked_weight_size
    assert q(300, 200, 128, 128, ctypes.byref(wb), ctypes.byref(sb)) == _lib.OK
    assert wb.value == 3 * 2 * 16384 and sb.value == 3 * 2 * 4
    assert q(300, 200, 1, 128, ctypes.byref(wb), ctypes.byref(sb)) == _lib.OK
    assert sb.value == 300 * 2 * 4
    assert q(300, 200, 0, 0, ctypes.byref(wb), ctypes.byref(sb)) == _lib.OK and sb.value == 4
    assert q(300, 200, 1, 32, ctypes.byref(wb), ctypes.byref(sb)) == _lib.ERR_UNSUPPORTED
    assert q(300, 0, 128, 128, ctypes.byref(wb), ctypes.byref(sb)) == _lib.ERR_INVALID_ARG
    pk = lib.mxq_prepack_weight
    ALIGNED = ctypes.c_void_p(1 << 20)
    assert pk(None, 256, 256, 256, FAKE, 128, 128, 2, 1, ALIGNED, FAKE, None) == _lib.ERR_INVALID_ARG
    assert pk(FAKE, 256, 256, 256, FAKE, 64, 128, 2, 1, ALIGNED, FAKE, None) == _lib.ERR_UNSUPPORTED
    assert pk(FAKE, 256, 256, 200, FAKE, 128, 128, 2, 1, ALIGNED, FAKE, None) == _lib.ERR_UNSUPPORTED
    assert pk(FAKE, 256, 256, 256, FAKE, 128, 128, 2, 1, ctypes.c_void_p((1 << 20) + 16), FAKE,
              None) == _lib.ERR_INVALID_ARG                       # tiles not 256-byte aligned
    mmp = lib.mxq_fp8_scaled_mm_prepacked
    args = [FAKE, 3, 4, 256, 256, FAKE, 2, 1, ALIGNED, 128, FAKE, 128, 128, None, 0, FAKE, 1, 128,
            None, 0, None]
    bad = list(args)
    bad[11], bad[12] = 1, 32                                      # MXFP8 [1, 32]
    assert mmp(*bad) == _lib.ERR_UNSUPPORTED
    bad = list(args)
    bad[8] = ctypes.c_void_p((1 << 20) + 16)                      # tiles not 256-byte aligned
    assert mmp(*bad) == _lib.ERR_INVALID_ARG


def test_quant_align_moe_argument_errors(lib):
    from mxfp4_quantized_gemm_token_gb300 import _lib
    q = lib.mxq_per_token_group_quant_fp8
    assert q(FAKE, 0, 128, 128, 128, 1e-10, FAKE, FAKE, None) == _lib.OK
    assert q(None, 2, 128, 128, 128, 1e-10, FAKE, FAKE, None) == _lib.ERR_INVALID_ARG
    assert q(FAKE, 2, 128, 64, 128, 1e-10, FAKE, FAKE, None) == _lib.ERR_INVALID_ARG
    assert q(FAKE, 2, 128, 128, 12, 1e-10, FAKE, FAKE, None) == _lib.ERR_UNSUPPORTED
    assert q(FAKE, 2, 128, 128, 128, 0.0, FAKE, FAKE, None) == _lib.ERR_INVALID_ARG
    al = lib.mxq_moe_align_block
    assert al(FAKE, 4, 2, 8, 48, FAKE, FAKE, FAKE, FAKE, 100, None, 0, None) == _lib.ERR_UNSUPPORTED
    assert al(FAKE, 4, 2, 2000, 16, FAKE, FAKE, FAKE, FAKE, 100, None, 0, None) == _lib.ERR_UNSUPPORTED
    assert al(FAKE, 4, 2, 8, 16, FAKE, FAKE, FAKE, FAKE, 1, None, 0, None) == _lib.ERR_INVALID_ARG
    sz = ctypes.c_size_t()
    assert lib.mxq_fused_experts_workspace_size(4, 256, 8, 128, 2, 16, 1, ctypes.byref(sz)) == 0
    assert sz.value > 0
    # block_m 0 is the library's choice: 32 when T*topk <= 16*E, else 64; the
    # workspace query resolves it the same way the call does
    def ws(T, topk, E, bm):
        v = ctypes.c_size_t()
        assert lib.mxq_fused_experts_workspace_size(T, 7168, E, 2048, topk, bm, 1,
                                                    ctypes.byref(v)) == 0
        return v.value
    assert ws(256, 8, 256, 0) == ws(256, 8, 256, 32)       # 2048 slots <= 16 * 256
    assert ws(1024, 8, 256, 0) == ws(1024, 8, 256, 64)     # 8192 slots > 16 * 256
    assert ws(512, 4, 128, 0) == ws(512, 4, 128, 32)       # 2048 = 16 * 128
    assert ws(1024, 8, 256, 32) != ws(1024, 8, 256, 64)    # the two block sizes differ here
    assert lib.mxq_fused_experts_workspace_size(4, 256, 8, 128, 2, -1, 1,
                                                ctypes.byref(sz)) == _lib.ERR_INVALID_ARG
    fe = lib.mxq_fused_experts
    args = [FAKE, 4, 256, 256, 1, 8, 128, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, FAKE, 2, 16,
            FAKE, 256, FAKE, sz.value, None]
    bad = list(args)
    bad[16] = 24                                              # block_m
    assert fe(*bad) == _lib.ERR_UNSUPPORTED
    bad = list(args)
    bad[4] = 9                                                # wtype
    assert fe(*bad) == _lib.ERR_UNSUPPORTED
    bad = list(args)
    bad[15] = 9                                               # topk > E
    assert fe(*bad) == _lib.ERR_INVALID_ARG
    bad = list(args)
    bad[20] = 16                                              # workspace too small
    assert fe(*bad) == _lib.ERR_INVALID_ARG
    bad = list(args)
    bad[1] = 0                                                # no tokens
    assert fe(*bad) == _lib.OK


def test_binding_has_no_cpu_fallback():
    """Every op refuses CPU tensors before touching the library: there is no
    CPU path behind the binding (the oracle is test infrastructure only)."""
    import torch
    import mxfp4_quantized_gemm_token_gb300 as mxq
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    w = torch.zeros(128, 256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    ws = torch.ones(1, 2)
    with pytest.raises(ValueError, match="CUDA"):
        mxq.per_token_group_quant_fp8(x)
    with pytest.raises(ValueError, match="CUDA"):
        mxq.fp8_scaled_mm(x, w, torch.ones(()), None)
    with pytest.raises(ValueError, match="CUDA"):
        mxq.moe_align_block(torch.zeros(4, 2, dtype=torch.int32), 8, 16)
    w1 = torch.zeros(2, 256, 256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="CUDA"):
        mxq.fused_experts(x, w1, ws, w1, ws, torch.ones(4, 1), torch.zeros(4, 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="block sizes"):
        mxq.w8a8_block_fp8_linear(x, w, [1, 32], ws)      # MXFP8-style [1, 32] blocks
