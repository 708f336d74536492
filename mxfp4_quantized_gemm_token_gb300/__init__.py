"""GB300-native weight-quantized scaled GEMM and routed fused MoE.

A thin PyTorch binding over libmxq (the C ABI in ``include/mxq.h``).  Torch
provides device memory and the current stream; every step of the hot path
runs in the library's CUDA kernels.  The functions here only marshal
arguments: shapes, strides, output/workspace allocation and the stream.

    per_token_group_quant_fp8(x, group=128, eps=1e-10) -> (q, scales)
    fp8_scaled_mm(a, w, w_scale, block_size, a_scale=None, bias=None, ...)
    w8a8_block_fp8_linear(input, weight, block_size, weight_scale, ...)
    moe_align_block(topk_ids, num_experts, block_m) -> (sorted_ids, expert_ids,
                                                        offsets, num_blocks)
    fused_experts(hidden, w1, w1_scale, w2, w2_scale, topk_weights, topk_ids, ...)
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import MxqError, check

__all__ = [
    "MxqError", "per_token_group_quant_fp8", "fp8_scaled_mm", "w8a8_block_fp8_linear",
    "PackedWeight", "prepack_weight", "fp8_scaled_bmm", "quantize_mxfp4",
    "fp8_per_tensor_linear", "moe_align_block", "fused_experts", "align_capacity",
    "set_option", "get_option", "sync_status", "W_FP8_BLOCK128", "W_MXFP4",
]

W_FP8_BLOCK128 = _lib.W_FP8_BLOCK128
W_MXFP4 = _lib.W_MXFP4


def _lib_handle():
    return _lib.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("mxq operates on CUDA tensors only (got a %s tensor)" % t.device)


def set_option(option: int, value: int) -> None:
    check(_lib_handle().mxq_set_option(option, int(value)))


def get_option(option: int) -> int:
    v = ctypes.c_int64(0)
    check(_lib_handle().mxq_get_option(option, ctypes.byref(v)))
    return int(v.value)


def sync_status(device=None) -> None:
    """Synchronize the current stream and raise if a kernel flagged an error."""
    device = device if device is not None else torch.cuda.current_device()
    check(_lib_handle().mxq_sync_status(_stream(device)))


# ------------------------------------------------------------ quantization

def per_token_group_quant_fp8(x: torch.Tensor, group: int = 128, eps: float = 1e-10):
    """bf16 [..., K] -> (e4m3 [..., K], fp32 scales [..., ceil(K/group)])."""
    _need_cuda(x)
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bf16")
    K = x.shape[-1]
    x2 = x.reshape(-1, K) if x.dim() != 2 else x
    if x2.stride(-1) != 1:
        x2 = x2.contiguous()
    M = x2.shape[0]
    G = -(-K // group)
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x.device)
    s = torch.empty((M, G), dtype=torch.float32, device=x.device)
    check(_lib_handle().mxq_per_token_group_quant_fp8(
        _ptr(x2), M, K, x2.stride(0), group, float(eps), _ptr(q), _ptr(s), _stream(x.device)))
    return q.view(*x.shape[:-1], K), s.view(*x.shape[:-1], G)


def quantize_mxfp4(w: torch.Tensor):
    """bf16 / fp32 [..., C] (C % 32 == 0) -> (packed e2m1x2 uint8 [..., C/2],
    ue8m0 uint8 [..., C/32]) by the OCP MX rule."""
    _need_cuda(w)
    if w.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("w must be bf16 or fp32")
    C = w.shape[-1]
    w2 = _as_rows(w)
    R = w2.shape[0]
    packed = torch.empty((R, C // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((R, max(C // 32, 1)), dtype=torch.uint8, device=w.device)
    check(_lib_handle().mxq_quantize_mxfp4(
        _ptr(w2), _lib.BF16 if w.dtype == torch.bfloat16 else _lib.F32, R, C, w2.stride(0),
        _ptr(packed), _ptr(scales), _stream(w.device)))
    return packed.view(*w.shape[:-1], C // 2), scales.view(*w.shape[:-1], C // 32)


# ------------------------------------------------------------- scaled GEMM

def _as_rows(t: torch.Tensor):
    """A 2-D view [rows, K] with unit inner stride (copies only if needed)."""
    K = t.shape[-1]
    t2 = t.reshape(-1, K)
    if t2.stride(-1) != 1:
        t2 = t2.contiguous()
    return t2


class PackedWeight:
    """An e4m3 weight [N, K] and its scales after mxq_prepack_weight: the
    tiles (uint8, 16384 bytes per 128 x 128 tile) and the K-block-major
    scales.  Pass it as ``w`` to fp8_scaled_mm / w8a8_block_fp8_linear."""

    def __init__(self, tiles, scales, N, K, block_size):
        self.tiles, self.scales, self.N, self.K = tiles, scales, N, K
        self.block_size = None if block_size is None else [int(b) for b in block_size]
        self.device = tiles.device

    @property
    def shape(self):
        return (self.N, self.K)


def prepack_weight(w, w_scale, block_size=None) -> PackedWeight:
    """Load-time relayout of an e4m3 weight [N, K] (any row stride with unit
    inner stride) and its scales (per-tensor, or [ceil(N/bn), ceil(K/128)]
    with any strides) into the tile layout the GEMM streams."""
    _need_cuda(w, w_scale)
    lib = _lib_handle()
    if w.stride(-1) != 1:
        w = w.contiguous()
    N, K = w.shape
    bn, bk = (0, 0) if block_size is None else (int(block_size[0]), int(block_size[1]))
    sw0 = sw1 = 0
    if block_size is not None:
        if w_scale.dim() != 2:
            raise ValueError("block weight scales must be 2-D")
        sw0, sw1 = w_scale.stride(0), w_scale.stride(1)
    elif w_scale.numel() != 1:
        raise ValueError("per-tensor scale must have one element")
    wb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    check(lib.mxq_prepacked_weight_size(N, K, bn, bk, ctypes.byref(wb), ctypes.byref(sb)))
    tiles = torch.empty(max(wb.value, 1), dtype=torch.uint8, device=w.device)
    scales = torch.empty(max(sb.value // 4, 1), dtype=torch.float32, device=w.device)
    check(lib.mxq_prepack_weight(_ptr(w), N, K, w.stride(0), _ptr(w_scale), bn, bk, sw0, sw1,
                                 _ptr(tiles), _ptr(scales), _stream(w.device)))
    return PackedWeight(tiles, scales, N, K, block_size)


def fp8_scaled_mm(a, w, w_scale, block_size=None, a_scale=None, bias=None,
                  out_dtype=torch.bfloat16, workspace=None):
    """out[..., N] = sum_k a[..., k] w[n, k] * scales (+ bias).

    a: e4m3 [..., K] with a_scale fp32 [..., ceil(K/128)] (W8A8), or bf16
    [..., K] with a_scale None (W8A16); w: e4m3 [N, K]; w_scale: fp32 0-d/[1]
    (per-tensor, block_size None) or [ceil(N/bn), ceil(K/128)] with
    block_size [bn, 128], bn in {1, 128}, any strides.
    w may also be a PackedWeight (prepack_weight), with w_scale None and the
    block_size it was packed with; the result is bit-identical.
    workspace: None (the library's split-K plan, sized by the workspace
    query and allocated here) or a caller buffer of at least that size; an
    empty buffer runs without split-K.
    """
    packed = isinstance(w, PackedWeight)
    if packed:
        if w_scale is not None:
            raise ValueError("a PackedWeight carries its scales: pass w_scale=None")
        if (block_size is None) != (w.block_size is None) or (
                block_size is not None and list(block_size) != w.block_size):
            raise ValueError("block_size %r does not match the packed weight's %r"
                             % (block_size, w.block_size))
        if a.shape[-1] != w.K:
            raise ValueError("K of the input (%d) and of the packed weight (%d) differ"
                             % (a.shape[-1], w.K))
        _need_cuda(a, w.tiles, a_scale, bias)
    else:
        _need_cuda(a, w, w_scale, a_scale, bias)
    lib = _lib_handle()
    K = a.shape[-1]
    a2 = _as_rows(a)
    M = a2.shape[0]
    if not packed and w.stride(-1) != 1:
        w = w.contiguous()
    N = w.N if packed else w.shape[0]
    if a.dtype == torch.float8_e4m3fn:
        a_dtype = _lib.E4M3
    elif a.dtype == torch.bfloat16:
        a_dtype = _lib.BF16
    else:
        raise TypeError("a must be float8_e4m3fn or bfloat16")
    sa0 = sa1 = 0
    if a_scale is not None:
        a_scale = a_scale.reshape(-1, a_scale.shape[-1])
        sa0, sa1 = a_scale.stride(0), a_scale.stride(1)
    if block_size is None:
        bn = bk = 0
        sw0 = sw1 = 0
        if not packed and w_scale.numel() != 1:
            raise ValueError("per-tensor scale must have one element")
    else:
        if not isinstance(block_size, (list, tuple)) or len(block_size) != 2:
            raise ValueError("block_size must be a two-element list, got %r" % (block_size,))
        bn, bk = int(block_size[0]), int(block_size[1])
        if not packed:
            if w_scale.dim() != 2:
                raise ValueError("block weight scales must be 2-D")
            sw0, sw1 = w_scale.stride(0), w_scale.stride(1)
    bias_dtype = 0
    if bias is not None:
        if bias.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("bias must be fp32 or bf16")
        bias_dtype = _lib.BF16 if bias.dtype == torch.bfloat16 else _lib.F32
        bias = bias.contiguous()
    od = _lib.BF16 if out_dtype == torch.bfloat16 else _lib.F32
    out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    ws_bytes = 0
    if workspace is None:
        sz = ctypes.c_size_t(0)
        check(lib.mxq_fp8_scaled_mm_workspace_size(M, N, K, a_dtype, bn, bk, ctypes.byref(sz)))
        if sz.value:
            workspace = torch.empty(sz.value, dtype=torch.uint8, device=a.device)
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    if packed:
        check(lib.mxq_fp8_scaled_mm_prepacked(
            _ptr(a2), a_dtype, M, K, a2.stride(0), _ptr(a_scale), sa0, sa1, _ptr(w.tiles), N,
            _ptr(w.scales), bn, bk, _ptr(bias), bias_dtype, _ptr(out), od, N,
            _ptr(workspace) if ws_bytes else None, ws_bytes, _stream(a.device)))
    else:
        check(lib.mxq_fp8_scaled_mm(
            _ptr(a2), a_dtype, M, K, a2.stride(0), _ptr(a_scale), sa0, sa1, _ptr(w), N,
            w.stride(0), _ptr(w_scale), bn, bk, sw0, sw1, _ptr(bias), bias_dtype, _ptr(out), od,
            N, _ptr(workspace) if ws_bytes else None, ws_bytes, _stream(a.device)))
    return out.view(*a.shape[:-1], N)


def fp8_scaled_bmm(a, w, w_scale, block_size=None, a_scale=None, bias=None,
                   out_dtype=torch.bfloat16):
    """Batched fp8_scaled_mm: out[b] = scaled_mm(a[b], w[b]) (+ bias[b]).

    a: [B, M, K] e4m3 (with a_scale [B, M, ceil(K/128)]) or bf16; w: e4m3
    [B, N, K]; w_scale: [B] / [B, 1] (per-tensor) or [B, ceil(N/bn),
    ceil(K/128)]; bias: None, [N] (shared) or [B, N].  One launch for the
    whole batch."""
    _need_cuda(a, w, w_scale, a_scale, bias)
    lib = _lib_handle()
    if a.dim() != 3 or w.dim() != 3 or a.shape[0] != w.shape[0] or a.shape[2] != w.shape[2]:
        raise ValueError("a must be [B, M, K] and w [B, N, K]")
    a, w = a.contiguous(), w.contiguous()
    B, M, K = a.shape
    N = w.shape[1]
    if a.dtype == torch.float8_e4m3fn:
        a_dtype = _lib.E4M3
    elif a.dtype == torch.bfloat16:
        a_dtype = _lib.BF16
    else:
        raise TypeError("a must be float8_e4m3fn or bfloat16")
    sa0 = sa1 = sab = 0
    if a_scale is not None:
        if a_scale.dim() != 3:
            raise ValueError("a_scale must be [B, M, ceil(K/128)]")
        sab, sa0, sa1 = a_scale.stride()
    if block_size is None:
        bn = bk = 0
        sw0 = sw1 = 0
        if w_scale.numel() != B:
            raise ValueError("per-tensor scales: one per batch")
        w_scale = w_scale.reshape(B).contiguous()
        swb = 1
    else:
        bn, bk = int(block_size[0]), int(block_size[1])
        if w_scale.dim() != 3:
            raise ValueError("block weight scales must be [B, ceil(N/bn), ceil(K/128)]")
        swb, sw0, sw1 = w_scale.stride()
    bias_dtype, bb = 0, 0
    if bias is not None:
        if bias.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("bias must be fp32 or bf16")
        bias_dtype = _lib.BF16 if bias.dtype == torch.bfloat16 else _lib.F32
        bias = bias.contiguous()
        bb = N if bias.dim() == 2 else 0
    od = _lib.BF16 if out_dtype == torch.bfloat16 else _lib.F32
    out = torch.empty((B, M, N), dtype=out_dtype, device=a.device)
    check(lib.mxq_fp8_scaled_bmm(
        B, _ptr(a), a_dtype, M, K, K, M * K, _ptr(a_scale), sa0, sa1, sab, _ptr(w), N, K, N * K,
        _ptr(w_scale), bn, bk, sw0, sw1, swb, _ptr(bias), bias_dtype, bb, _ptr(out), od, N, M * N,
        _stream(a.device)))
    return out


def w8a8_block_fp8_linear(input, weight, block_size, weight_scale, input_scale=None, bias=None):
    """Block-FP8 linear with the pages' semantics: quantize the input per
    1x128 group unless input_scale is given; output bf16 for a pre-quantized
    input, else input.dtype; batch dims restored.  weight may be a
    PackedWeight (prepack_weight), with weight_scale None."""
    if not isinstance(block_size, (list, tuple)) or len(block_size) != 2:
        raise ValueError("block_size must be a two-element list, got %r" % (block_size,))
    bn, bk = block_size
    if bk != 128 or bn not in (1, 128):
        raise ValueError("supported weight block sizes are [1, 128] and [128, 128], got %r"
                         % (list(block_size),))
    if input_scale is None and input.dtype == torch.bfloat16 and not isinstance(weight, PackedWeight):
        return _linear_bf16(input, weight, bn, weight_scale, bias)
    if input_scale is None:
        q, s = per_token_group_quant_fp8(input, bk)
        out_dtype = input.dtype
    else:
        q, s = input, input_scale
        out_dtype = torch.bfloat16
    return fp8_scaled_mm(q, weight, weight_scale, [bn, bk], a_scale=s, bias=bias,
                         out_dtype=out_dtype)


def _linear_bf16(x, w, bn, w_scale, bias):
    """mxq_w8a8_block_fp8_linear: quantization per 1 x 128 group and the W8A8
    GEMM in one call (fused into the GEMM for decode-size inputs)."""
    _need_cuda(x, w, w_scale, bias)
    lib = _lib_handle()
    K = x.shape[-1]
    x2 = _as_rows(x)
    M = x2.shape[0]
    if w.stride(-1) != 1:
        w = w.contiguous()
    N = w.shape[0]
    if w_scale.dim() != 2:
        raise ValueError("block weight scales must be 2-D")
    bias_dtype = 0
    if bias is not None:
        if bias.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("bias must be fp32 or bf16")
        bias_dtype = _lib.BF16 if bias.dtype == torch.bfloat16 else _lib.F32
        bias = bias.contiguous()
    out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    sz = ctypes.c_size_t(0)
    check(lib.mxq_w8a8_block_fp8_linear_workspace_size(M, N, K, bn, ctypes.byref(sz)))
    ws = torch.empty(sz.value, dtype=torch.uint8, device=x.device) if sz.value else None
    check(lib.mxq_w8a8_block_fp8_linear(
        _ptr(x2), M, K, x2.stride(0), _ptr(w), N, w.stride(0), _ptr(w_scale), bn, 128,
        w_scale.stride(0), w_scale.stride(1), _ptr(bias), bias_dtype, _ptr(out), _lib.BF16, N,
        _ptr(ws), sz.value, _stream(x.device)))
    return out.view(*x.shape[:-1], N)


def fp8_per_tensor_linear(x, weight, scale, bias=None):
    """W8A16 per-tensor linear: (x . weight^T) * scale (+ bias), bf16 out."""
    return fp8_scaled_mm(x, weight, scale.reshape(1), None, bias=bias)


# ---------------------------------------------------------------------- MoE

def align_capacity(S: int, E: int, block_m: int) -> int:
    return -(-S // block_m) + min(E, S)


def moe_align_block(topk_ids: torch.Tensor, num_experts: int, block_m: int, cap=None):
    _need_cuda(topk_ids)
    ids = topk_ids.to(torch.int32).contiguous()
    T, topk = ids.shape
    S = T * topk
    cap = align_capacity(S, num_experts, block_m) if cap is None else cap
    dev = ids.device
    sorted_ids = torch.empty(cap * block_m, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    offsets = torch.empty(cap + 1, dtype=torch.int32, device=dev)
    nb = torch.empty(1, dtype=torch.int32, device=dev)
    check(_lib_handle().mxq_moe_align_block(
        _ptr(ids), T, topk, num_experts, block_m, _ptr(sorted_ids), _ptr(expert_ids),
        _ptr(offsets), _ptr(nb), cap, None, 0, _stream(dev)))
    return sorted_ids, expert_ids, offsets, nb


def fused_experts(hidden, w1, w1_scale, w2, w2_scale, topk_weights, topk_ids,
                  wtype=W_FP8_BLOCK128, w1_bias=None, w2_bias=None, block_m: int = 0,
                  workspace=None, checkpoints: bool = False, activation: str = "silu",
                  alpha: float = 1.702, limit: float = 7.0):
    """Routed MoE: align, stage 1 (+ SiLU-and-mul), stage 2, top-k combine.

    block_m: tokens per expert block (16, 32, 64, 128), or 0 for the
    library's choice (32 when T*topk <= 16*E, else 64).
    checkpoints: also return, in slot order (t*topk + k), act (bf16 [S, N]),
    y = w * z (fp32 [S, K]) and the stage-1 accumulator h before the bias
    (fp32 [S, 2N]).
    activation: "silu" (silu(gate) * up) or "swiglu_clamp" (GPT-OSS style:
    min(gate, limit) * sigmoid(alpha * min(gate, limit)) *
    (clamp(up, -limit, limit) + 1)); gate = the first N rows of w1[e]."""
    if activation not in ("silu", "swiglu_clamp"):
        raise ValueError("activation must be 'silu' or 'swiglu_clamp'")
    _need_cuda(hidden, w1, w1_scale, w2, w2_scale, topk_weights, topk_ids, w1_bias, w2_bias)
    lib = _lib_handle()
    T, K = hidden.shape
    if hidden.stride(-1) != 1:
        hidden = hidden.contiguous()
    E = w1.shape[0]
    N = w1.shape[1] // 2
    topk = topk_ids.shape[1]
    ids = topk_ids.to(torch.int32).contiguous()
    tw = topk_weights.to(torch.float32).contiguous()
    w1, w2 = w1.contiguous(), w2.contiguous()
    w1_scale, w2_scale = w1_scale.contiguous(), w2_scale.contiguous()
    b1 = None if w1_bias is None else w1_bias.to(torch.float32).contiguous()
    b2 = None if w2_bias is None else w2_bias.to(torch.float32).contiguous()
    out = torch.empty((T, K), dtype=torch.bfloat16, device=hidden.device)
    sz = ctypes.c_size_t(0)
    check(lib.mxq_fused_experts_workspace_size(T, K, E, N, topk, block_m, wtype, ctypes.byref(sz)))
    if workspace is None or workspace.numel() * workspace.element_size() < sz.value:
        workspace = torch.empty(max(sz.value, 1), dtype=torch.uint8, device=hidden.device)
    args = [_ptr(hidden), T, K, hidden.stride(0), wtype, E, N, _ptr(w1), _ptr(w1_scale), _ptr(b1),
            _ptr(w2), _ptr(w2_scale), _ptr(b2), _ptr(tw), _ptr(ids), topk, block_m, _ptr(out), K,
            _ptr(workspace), workspace.numel() * workspace.element_size()]
    if activation != "silu":
        act = y = h = None
        if checkpoints:
            act = torch.empty((T * topk, N), dtype=torch.bfloat16, device=hidden.device)
            y = torch.empty((T * topk, K), dtype=torch.float32, device=hidden.device)
            h = torch.empty((T * topk, 2 * N), dtype=torch.float32, device=hidden.device)
        check(lib.mxq_fused_experts_ex(*args[:17], _lib.ACT_SWIGLU_CLAMP, float(alpha),
                                       float(limit), *args[17:], _ptr(act), _ptr(y), _ptr(h),
                                       _stream(hidden.device)))
        return (out, act, y, h) if checkpoints else out
    if checkpoints:
        act = torch.empty((T * topk, N), dtype=torch.bfloat16, device=hidden.device)
        y = torch.empty((T * topk, K), dtype=torch.float32, device=hidden.device)
        h = torch.empty((T * topk, 2 * N), dtype=torch.float32, device=hidden.device)
        check(lib.mxq_fused_experts_debug(*args, _ptr(act), _ptr(y), _ptr(h),
                                          _stream(hidden.device)))
        return out, act, y, h
    check(lib.mxq_fused_experts(*args, _stream(hidden.device)))
    return out
