"""ctypes shim over the plain C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product path (the CUDA
library and its Python binding) never imports this package, and this package
imports nothing from the product.

Every function takes and returns numpy arrays.  bf16 data travels as its raw
``uint16`` bit patterns and fp8 / packed fp4 / ue8m0 data as ``uint8`` codes,
so nothing here depends on how a framework would cast them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# dtype tags of the oracle (its own numbering; nothing is shared)
BF16, F32, E4M3 = 1, 2, 3
W_FP8_BLOCK128, W_MXFP4 = 1, 2


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP when available) if stale."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-lm"]
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base[:-1] + ["-fopenmp", "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0_decode.restype = ctypes.c_double
        lib.oracle_ue8m0_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_decode.restype = ctypes.c_double
        lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
        lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [P, I64, P]
        lib.oracle_per_token_group_quant_fp8.restype = None
        lib.oracle_per_token_group_quant_fp8.argtypes = [P, I64, I64, I64, I32,
                                                          ctypes.c_float, P, P]
        lib.oracle_scaled_mm.restype = None
        lib.oracle_scaled_mm.argtypes = [P, I32, I64, I64, I64, P, I64, I64, P, I64,
                                         I64, P, I32, I32, I64, I64, P, I32, P, P, I64]
        lib.oracle_scaled_mm_at.restype = None
        lib.oracle_scaled_mm_at.argtypes = [P, I32, I64, I64, P, I64, I64, P, I64, P,
                                            I32, I32, I64, I64, P, I32, P, P, I64, P]
        lib.oracle_moe_align.restype = I32
        lib.oracle_moe_align.argtypes = [P, I64, I32, I32, I32, P, P, P, P, I64]
        lib.oracle_fused_experts.restype = I32
        lib.oracle_fused_experts.argtypes = [P, I64, I64, I64, I32, I32, I64, P, P, P,
                                             P, P, P, P, P, I32, P, I64, P, P]
        lib.oracle_expert_linear.restype = None
        lib.oracle_expert_linear.argtypes = [P, I64, I64, I32, P, P, I64, I64, I64, P]
        lib.oracle_mxfp4_quantize.restype = None
        lib.oracle_mxfp4_quantize.argtypes = [P, I64, I64, I64, P, P]
        lib.oracle_fused_experts_act.restype = I32
        lib.oracle_fused_experts_act.argtypes = [P, I64, I64, I64, I32, I32, I64, P, P, P,
                                                 P, P, P, P, P, I32, I32, ctypes.c_double,
                                                 ctypes.c_double, P, I64, P, P]
        lib.oracle_max_threads.restype = I32
        lib.oracle_set_threads.argtypes = [I32]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    """Contiguous numpy array of the given dtype (no value conversion)."""
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------ codecs

def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e2m1_decode(nibbles) -> np.ndarray:
    lib = _load()
    c = np.asarray(nibbles, dtype=np.uint8)
    return np.array([lib.oracle_e2m1_decode(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def ue8m0_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_ue8m0_decode(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def bf16_round(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.oracle_bf16_round(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def bf16_from_f32(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.oracle_bf16_from_f32(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    v = _c(np.asarray(values, dtype=np.float32), np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


# ------------------------------------------------------------------ ops

def per_token_group_quant_fp8(x_bf16_bits, group: int = 128, eps: float = 1e-10):
    """x: uint16 bf16 bits [M, K] (any row stride via a 2-D view)."""
    lib = _load()
    x = np.asarray(x_bf16_bits)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("x must be a 2-D uint16 array of bf16 bits")
    M, K = x.shape
    x = np.ascontiguousarray(x)
    G = (K + group - 1) // group
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, G), dtype=np.float32)
    lib.oracle_per_token_group_quant_fp8(_ptr(x), M, K, K, group, eps, _ptr(q), _ptr(s))
    return q, s


def _mm_args(a, a_dtype, a_scale, w, w_scale, block_n, block_k, bias):
    a = np.ascontiguousarray(a)
    w = _c(w, np.uint8)
    M, K = a.shape
    N = w.shape[0]
    if a_scale is not None:
        a_scale = _c(a_scale, np.float32)
    w_scale = np.ascontiguousarray(np.asarray(w_scale, dtype=np.float32)).reshape(
        (1,) if np.asarray(w_scale).ndim == 0 else np.asarray(w_scale).shape)
    bias_dtype = 0
    if bias is not None:
        bias = np.ascontiguousarray(bias)
        bias_dtype = BF16 if bias.dtype == np.uint16 else F32
        if bias_dtype == F32:
            bias = _c(bias, np.float32)
    sw0 = w_scale.shape[1] if (block_k and w_scale.ndim == 2) else 0
    sa0 = a_scale.shape[1] if a_scale is not None else 0
    return a, M, K, a_scale, sa0, w, N, w_scale, sw0, bias, bias_dtype


def scaled_mm(a, a_dtype, a_scale, w, w_scale, block_n=0, block_k=0, bias=None,
              w_scale_col_major=False):
    """Dequantise-then-matmul in fp64.  Returns (out_f32 [M,N], out_bf16_bits).

    a: uint16 bf16 bits (a_dtype=BF16) or uint8 e4m3 codes (E4M3), [M, K];
    a_scale: float32 [M, ceil(K/128)] or None; w: uint8 e4m3 [N, K];
    w_scale: float32 scalar / [1] (per-tensor) or [ceil(N/block_n), ceil(K/128)];
    bias: float32 [N], uint16 bf16 bits [N], or None.
    """
    lib = _load()
    a, M, K, a_scale, sa0, w, N, w_scale, sw0, bias, bias_dtype = _mm_args(
        a, a_dtype, a_scale, w, w_scale, block_n, block_k, bias)
    sw1 = 1
    if w_scale_col_major and w_scale.ndim == 2:
        # same logical [rows, cols] scales stored transposed-contiguous
        rows = w_scale.shape[0]
        w_scale = np.ascontiguousarray(w_scale.T)
        sw0, sw1 = 1, rows
    out_f32 = np.empty((M, N), dtype=np.float32)
    out_bf16 = np.empty((M, N), dtype=np.uint16)
    lib.oracle_scaled_mm(_ptr(a), a_dtype, M, K, K, _ptr(a_scale), sa0, 1, _ptr(w), N, K,
                         _ptr(w_scale), block_n, block_k, sw0, sw1, _ptr(bias), bias_dtype,
                         _ptr(out_f32), _ptr(out_bf16), N)
    return out_f32, out_bf16


def scaled_mm_at(a, a_dtype, a_scale, w, w_scale, block_n, block_k, bias, ms, ns):
    """fp64 accumulators (bias included, before rounding) at pairs (ms[i], ns[i])."""
    lib = _load()
    a, M, K, a_scale, sa0, w, N, w_scale, sw0, bias, bias_dtype = _mm_args(
        a, a_dtype, a_scale, w, w_scale, block_n, block_k, bias)
    ms = _c(np.asarray(ms, dtype=np.int64), np.int64)
    ns = _c(np.asarray(ns, dtype=np.int64), np.int64)
    out = np.empty(ms.shape, dtype=np.float64)
    lib.oracle_scaled_mm_at(_ptr(a), a_dtype, K, K, _ptr(a_scale), sa0, 1, _ptr(w), K,
                            _ptr(w_scale), block_n, block_k, sw0, 1, _ptr(bias),
                            bias_dtype, _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


def align_capacity(S: int, E: int, block_m: int) -> int:
    """Upper bound on the number of expert blocks: ceil(S/BM) + min(E, S)."""
    return (S + block_m - 1) // block_m + min(E, S)


def moe_align(topk_ids, E: int, block_m: int, cap: int | None = None):
    """Returns (sorted_ids [cap*BM], expert_ids [cap], offsets [cap+1], num_blocks)."""
    lib = _load()
    ids = _c(np.asarray(topk_ids, dtype=np.int32), np.int32)
    T, topk = ids.shape
    S = T * topk
    if cap is None:
        cap = align_capacity(S, E, block_m)
    sorted_ids = np.empty(cap * block_m, dtype=np.int32)
    expert_ids = np.empty(cap, dtype=np.int32)
    offsets = np.empty(cap + 1, dtype=np.int32)
    nb = np.zeros(1, dtype=np.int32)
    rc = lib.oracle_moe_align(_ptr(ids), T, topk, E, block_m, _ptr(sorted_ids),
                              _ptr(expert_ids), _ptr(offsets), _ptr(nb), cap)
    if rc != 0:
        raise ValueError("oracle_moe_align failed with code %d" % rc)
    return sorted_ids, expert_ids, offsets, int(nb[0])


def fused_experts(hidden_bits, wtype, w1, w1_scale, b1, w2, w2_scale, b2,
                  topk_weights, topk_ids, N: int, checkpoints: bool = False,
                  activation: int = 0, alpha: float = 1.702, limit: float = 7.0):
    """Reference routed MoE.  Returns out bf16 bits [T, K] (and act, z).
    activation 0: SiLU-and-mul; 1: clamped SwiGLU (alpha, limit)."""
    lib = _load()
    x = _c(hidden_bits, np.uint16)
    T, K = x.shape
    w1 = _c(w1, np.uint8)
    w2 = _c(w2, np.uint8)
    E = w1.shape[0]
    if wtype == W_MXFP4:
        w1_scale = _c(w1_scale, np.uint8)
        w2_scale = _c(w2_scale, np.uint8)
    else:
        w1_scale = _c(w1_scale, np.float32)
        w2_scale = _c(w2_scale, np.float32)
    b1 = None if b1 is None else _c(b1, np.float32)
    b2 = None if b2 is None else _c(b2, np.float32)
    tw = _c(topk_weights, np.float32)
    ids = _c(np.asarray(topk_ids, dtype=np.int32), np.int32)
    topk = ids.shape[1]
    out = np.empty((T, K), dtype=np.uint16)
    act = np.empty((T * topk, N), dtype=np.uint16) if checkpoints else None
    z = np.empty((T * topk, K), dtype=np.float64) if checkpoints else None
    rc = lib.oracle_fused_experts_act(_ptr(x), T, K, K, wtype, E, N, _ptr(w1), _ptr(w1_scale),
                                      _ptr(b1), _ptr(w2), _ptr(w2_scale), _ptr(b2), _ptr(tw),
                                      _ptr(ids), topk, int(activation), float(alpha),
                                      float(limit), _ptr(out), K, _ptr(act), _ptr(z))
    if rc != 0:
        raise ValueError("oracle_fused_experts failed with code %d" % rc)
    if checkpoints:
        return out, act, z
    return out


def expert_linear(x_bits, wtype, w, w_scale, e: int):
    """One expert GEMM without bias, fp64: x [M, C] (bf16 bits) . W[e]^T.

    w: [E, R, C] e4m3 (w_scale fp32 [E, ceil(R/128), ceil(C/128)]) or
    [E, R, C/2] packed e2m1 (w_scale ue8m0 [E, R, C/32]).  Returns [M, R]."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    M, C = x.shape
    w = _c(w, np.uint8)
    R = w.shape[1]
    w_scale = _c(w_scale, np.uint8 if wtype == W_MXFP4 else np.float32)
    if not 0 <= e < w.shape[0]:
        raise ValueError("expert index out of range")
    out = np.empty((M, R), dtype=np.float64)
    lib.oracle_expert_linear(_ptr(x), M, C, wtype, _ptr(w), _ptr(w_scale), e, R, C, _ptr(out))
    return out


def mxfp4_quantize(x_f32):
    """OCP MX rule: fp32 [R, C] (C % 32 == 0) -> (packed e2m1 [R, C/2] uint8,
    ue8m0 scales [R, C/32] uint8)."""
    lib = _load()
    x = _c(np.asarray(x_f32, dtype=np.float32), np.float32)
    R, C = x.shape
    if C % 32 != 0:
        raise ValueError("C must be a multiple of 32")
    packed = np.zeros((R, C // 2), dtype=np.uint8)
    scales = np.empty((R, C // 32), dtype=np.uint8)
    lib.oracle_mxfp4_quantize(_ptr(x), R, C, C, _ptr(packed), _ptr(scales))
    return packed, scales


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))
