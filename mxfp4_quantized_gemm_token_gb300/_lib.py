"""ctypes loader for libmxq.so (the C ABI declared in include/mxq.h).

There is no fallback: if the library cannot be built or loaded, every call
raises.  The library is built in-tree (``mxfp4_quantized_gemm_token_gb300/
libmxq.so``) by ``build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

# status codes and tags (mirror include/mxq.h)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(6)
BF16, F32, E4M3, E2M1X2, UE8M0 = 1, 2, 3, 4, 5
W_FP8_BLOCK128, W_MXFP4 = 1, 2
ACT_SILU, ACT_SWIGLU_CLAMP = 0, 1
(OPT_SMALL_M_MAX, OPT_FORCE_PATH, OPT_WAIT_BUDGET_NS, OPT_SPLIT_K, OPT_INJECT_STALL, OPT_NUM_SMS,
 OPT_TILE_N, OPT_NORMAL_TILE, OPT_PDL, OPT_FUSE_COMBINE, OPT_MOE_F16,
 OPT_FUSE_QUANT) = (1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12)

EXPORTED = [
    "mxq_last_error", "mxq_version", "mxq_set_option", "mxq_get_option", "mxq_sync_status",
    "mxq_per_token_group_quant_fp8", "mxq_fp8_scaled_mm", "mxq_fp8_scaled_mm_workspace_size",
    "mxq_moe_align_block", "mxq_fused_experts", "mxq_fused_experts_debug",
    "mxq_fused_experts_workspace_size", "mxq_fp8_scaled_mm_noalloc",
    "mxq_prepacked_weight_size", "mxq_prepack_weight", "mxq_fp8_scaled_mm_prepacked",
    "mxq_fp8_scaled_bmm", "mxq_quantize_mxfp4", "mxq_fused_experts_ex",
    "mxq_w8a8_block_fp8_linear", "mxq_w8a8_block_fp8_linear_workspace_size",
]

NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class MxqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("mxq status %d: %s" % (status, message))
        self.status = status


def _declare(lib):
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    F = ctypes.c_float
    st = ctypes.c_int32
    sig = {
        "mxq_last_error": (ctypes.c_char_p, []),
        "mxq_version": (ctypes.c_char_p, []),
        "mxq_set_option": (st, [I32, I64]),
        "mxq_get_option": (st, [I32, ctypes.POINTER(I64)]),
        "mxq_sync_status": (st, [P]),
        "mxq_per_token_group_quant_fp8": (st, [P, I64, I64, I64, I32, F, P, P, P]),
        "mxq_fp8_scaled_mm": (st, [P, I32, I64, I64, I64, P, I64, I64, P, I64, I64, P, I32, I32,
                                   I64, I64, P, I32, P, I32, I64, P, SZ, P]),
        "mxq_fp8_scaled_mm_noalloc": (st, [P, I32, I64, I64, I64, P, I64, I64, P, I64, I64, P,
                                           I32, I32, I64, I64, P, I32, P, I32, I64, P]),
        "mxq_fp8_scaled_mm_workspace_size": (st, [I64, I64, I64, I32, I32, I32,
                                                  ctypes.POINTER(SZ)]),
        "mxq_prepacked_weight_size": (st, [I64, I64, I32, I32, ctypes.POINTER(SZ),
                                           ctypes.POINTER(SZ)]),
        "mxq_prepack_weight": (st, [P, I64, I64, I64, P, I32, I32, I64, I64, P, P, P]),
        "mxq_fp8_scaled_mm_prepacked": (st, [P, I32, I64, I64, I64, P, I64, I64, P, I64, P, I32,
                                             I32, P, I32, P, I32, I64, P, SZ, P]),
        "mxq_fp8_scaled_bmm": (st, [I64, P, I32, I64, I64, I64, I64, P, I64, I64, I64, P, I64,
                                    I64, I64, P, I32, I32, I64, I64, I64, P, I32, I64, P, I32,
                                    I64, I64, P]),
        "mxq_quantize_mxfp4": (st, [P, I32, I64, I64, I64, P, P, P]),
        "mxq_w8a8_block_fp8_linear": (st, [P, I64, I64, I64, P, I64, I64, P, I32, I32, I64,
                                           I64, P, I32, P, I32, I64, P, SZ, P]),
        "mxq_w8a8_block_fp8_linear_workspace_size": (st, [I64, I64, I64, I32,
                                                          ctypes.POINTER(SZ)]),
        "mxq_moe_align_block": (st, [P, I64, I32, I32, I32, P, P, P, P, I64, P, SZ, P]),
        "mxq_fused_experts": (st, [P, I64, I64, I64, I32, I32, I64, P, P, P, P, P, P, P, P, I32,
                                   I32, P, I64, P, SZ, P]),
        "mxq_fused_experts_debug": (st, [P, I64, I64, I64, I32, I32, I64, P, P, P, P, P, P, P, P,
                                         I32, I32, P, I64, P, SZ, P, P, P, P]),
        "mxq_fused_experts_ex": (st, [P, I64, I64, I64, I32, I32, I64, P, P, P, P, P, P, P, P,
                                      I32, I32, I32, F, F, P, I64, P, SZ, P, P, P, P]),
        "mxq_fused_experts_workspace_size": (st, [I64, I64, I32, I64, I32, I32, I32,
                                                  ctypes.POINTER(SZ)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmxq.so (building it first if it does not exist)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError("libmxq.so is not built (run __graft_entry__.build())")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        _declare(lib)
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != OK:
        raise MxqError(status, load().mxq_last_error().decode(errors="replace"))
