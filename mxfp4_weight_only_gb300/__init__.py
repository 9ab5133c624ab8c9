"""Python binding of the GB300 A16W4 MoE library (argument marshalling only).

Each function checks tensor placement, dtypes and shapes, allocates outputs
and the workspace with PyTorch when the caller does not pass them, and calls
the C ABI of ``libmoe_a16w4.so`` (include/moe_a16w4.h) with raw device
pointers on the current CUDA stream.  Every computation runs in the
library's CUDA kernels; there is no fallback path.
"""

from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import (MOE_ACT_SWIGLU, MOE_AQ_FP8, MOE_AQ_MXFP4, MOE_AQ_NONE,  # noqa: F401
                      MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL, MOE_STATUS_BAD_INDEX,
                      MOE_STATUS_NAN_SCALE, MOE_STATUS_WAIT_TIMEOUT, MoeDims, MoeError, MoeOptions, use_checked)

__all__ = [
    "moe_workspace_bytes", "moe_a16w4_mxfp4", "moe_a16w4_int4g32", "requant_mxfp4_to_int4g32",
    "moe_route", "moe_router_topk", "moe_read_status", "moe_quantize_act", "dims", "MoeError",
]

_AQ = {None: MOE_AQ_NONE, "bf16": MOE_AQ_NONE, "mxfp4": MOE_AQ_MXFP4, "fp8": MOE_AQ_FP8}


def _lib():
    return _native.load()


def dims(E: int, H: int, I: int, topk: int, T: int, path: int = MOE_PATH_AUTO) -> MoeDims:
    return MoeDims(E, H, I, topk, T, MOE_ACT_SWIGLU, path)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def moe_workspace_bytes(d: MoeDims) -> int:
    return int(_lib().moe_workspace_bytes(ctypes.byref(d)))


def _workspace(d: MoeDims, workspace, device):
    need = moe_workspace_bytes(d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace


def _options(E, H, I, w13_bias, w2_bias, expert_map, router_weight_on_input, act_quant=None,
             w13_input_scale=1.0, w2_input_scale=1.0, swiglu_limit=None):
    """The optional inputs as a MoeOptions struct, or None when none is set."""
    aq = _AQ[act_quant]
    if (w13_bias is None and w2_bias is None and expert_map is None and not router_weight_on_input and not aq
            and swiglu_limit is None):
        return None
    if w13_bias is not None:
        _need(w13_bias, "w13_bias", torch.bfloat16, (E, 2 * I))
    if w2_bias is not None:
        _need(w2_bias, "w2_bias", torch.bfloat16, (E, H))
    G = 0
    if expert_map is not None:
        G = expert_map.shape[0]
        _need(expert_map, "expert_map", torch.int32, (G,))
    return MoeOptions(_ptr(w13_bias).value, _ptr(w2_bias).value, _ptr(expert_map).value, G,
                      1 if router_weight_on_input else 0, aq, float(w13_input_scale), float(w2_input_scale),
                      0.0 if swiglu_limit is None else float(swiglu_limit))


def _moe(fn_name, x, topk_ids, topk_w, w13, s13, w2, s2, out, workspace, path, stream, scale_dtype,
         w13_bias=None, w2_bias=None, expert_map=None, router_weight_on_input=False, act_quant=None,
         w13_input_scale=1.0, w2_input_scale=1.0, swiglu_limit=None):
    T, H = x.shape
    E, two_i, _ = w13.shape
    I = two_i // 2
    topk = topk_ids.shape[1]
    _need(x, "x", torch.bfloat16, (T, H))
    _need(topk_ids, "topk_ids", torch.int32, (T, topk))
    _need(topk_w, "topk_w", torch.float32, (T, topk))
    _need(w13, "w13", torch.uint8, (E, 2 * I, H // 2))
    _need(s13, "w13_scale", scale_dtype, (E, 2 * I, H // 32))
    _need(w2, "w2", torch.uint8, (E, H, I // 2))
    _need(s2, "w2_scale", scale_dtype, (E, H, I // 32))
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (T, H))
    d = dims(E, H, I, topk, T, path)
    workspace = _workspace(d, workspace, x.device)
    opt = _options(E, H, I, w13_bias, w2_bias, expert_map, router_weight_on_input, act_quant, w13_input_scale,
                   w2_input_scale, swiglu_limit)
    if opt is None:
        rc = getattr(_lib(), fn_name)(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(s13),
                                      _ptr(w2), _ptr(s2), _ptr(out), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    else:
        fn_name += "_ex"
        rc = getattr(_lib(), fn_name)(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(s13),
                                      _ptr(w2), _ptr(s2), ctypes.byref(opt), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(stream))
    _native.check(fn_name, rc)
    return out


def moe_a16w4_mxfp4(x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, out=None, workspace=None,
                    path: int = MOE_PATH_AUTO, stream=None, w13_bias=None, w2_bias=None, expert_map=None,
                    router_weight_on_input: bool = False, act_quant=None, w13_input_scale: float = 1.0,
                    w2_input_scale: float = 1.0, swiglu_limit=None):
    """Fused MoE on MXFP4 weights (uint8 packed E2M1 + uint8 E8M0 scales).

    Optional: ``w13_bias`` bf16 [E, 2I], ``w2_bias`` bf16 [E, H], ``expert_map``
    int32 [global experts] (topk_ids then hold global ids),
    ``router_weight_on_input``, and ``act_quant`` ("mxfp4": W4A4, "fp8": W4A8
    with the static ``w13_input_scale`` / ``w2_input_scale``), and
    ``swiglu_limit`` (gate_up outputs clamped to [-limit, limit] before the
    gating); any of them selects ``moe_a16w4_mxfp4_ex``."""
    return _moe("moe_a16w4_mxfp4", x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, out, workspace, path,
                stream, torch.uint8, w13_bias, w2_bias, expert_map, router_weight_on_input, act_quant,
                w13_input_scale, w2_input_scale, swiglu_limit)


def moe_a16w4_int4g32(x, topk_ids, topk_w, w13_q, w13_s, w2_q, w2_s, out=None, workspace=None,
                      path: int = MOE_PATH_AUTO, stream=None, w13_bias=None, w2_bias=None, expert_map=None,
                      router_weight_on_input: bool = False, act_quant=None, w13_input_scale: float = 1.0,
                      w2_input_scale: float = 1.0, swiglu_limit=None):
    """Fused MoE on int4_per_group_32 weights (uint8 packed int4 + float32 or bfloat16 group
    scales: bfloat16 selects ``moe_a16w4_int4g32_bf16s``); options as ``moe_a16w4_mxfp4``
    (the library rejects ``act_quant`` with int4 weights)."""
    bf16 = w13_s.dtype == torch.bfloat16
    return _moe("moe_a16w4_int4g32_bf16s" if bf16 else "moe_a16w4_int4g32", x, topk_ids, topk_w, w13_q, w13_s,
                w2_q, w2_s, out, workspace, path, stream, torch.bfloat16 if bf16 else torch.float32, w13_bias,
                w2_bias, expert_map, router_weight_on_input, act_quant, w13_input_scale, w2_input_scale,
                swiglu_limit)


def requant_mxfp4_to_int4g32(w, scale, out_q=None, out_s=None, experts_per_chunk: int = 8, stream=None,
                             scale_dtype=torch.float32):
    """Lossy MXFP4 -> int4_per_group_32 conversion; returns ``(q uint8, s)`` with ``s``
    float32, or bfloat16 (``scale_dtype=torch.bfloat16``: ``requant_mxfp4_to_int4g32_bf16s``)."""
    E, N, Kh = w.shape
    K = 2 * Kh
    if scale_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("scale_dtype must be torch.float32 or torch.bfloat16")
    _need(w, "w", torch.uint8, (E, N, Kh))
    _need(scale, "scale", torch.uint8, (E, N, K // 32))
    if out_q is None:
        out_q = torch.empty_like(w)
    if out_s is None:
        out_s = torch.empty((E, N, K // 32), dtype=scale_dtype, device=w.device)
    _need(out_q, "out_q", torch.uint8, (E, N, Kh))
    _need(out_s, "out_s", scale_dtype, (E, N, K // 32))
    fn = "requant_mxfp4_to_int4g32_bf16s" if scale_dtype == torch.bfloat16 else "requant_mxfp4_to_int4g32"
    rc = getattr(_lib(), fn)(E, N, K, _ptr(w), _ptr(scale), _ptr(out_q), _ptr(out_s), experts_per_chunk,
                             _stream(stream))
    _native.check(fn, rc)
    return out_q, out_s


def moe_route(topk_ids, E: int, stream=None):
    """Stable grouping of the pairs by expert: ``(counts, offsets, sorted_pair, pair_pos)``."""
    T, topk = topk_ids.shape
    _need(topk_ids, "topk_ids", torch.int32, (T, topk))
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(T * topk, dtype=torch.int32, device=dev)
    pos = torch.empty(T * topk, dtype=torch.int32, device=dev)
    d = dims(E, 64, 64, topk, T)
    rc = _lib().moe_route(ctypes.byref(d), _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(sp), _ptr(pos),
                          _stream(stream))
    _native.check("moe_route", rc)
    return counts, offsets, sp, pos


def moe_router_topk(logits, topk: int, renormalize: bool = True, stream=None):
    """Top-k routing from float32 router logits [T, G]: ``(ids int32 [T, topk], weights float32 [T, topk])``."""
    T, G = logits.shape
    _need(logits, "logits", torch.float32, (T, G))
    ids = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    rc = _lib().moe_router_topk(_ptr(logits), T, G, topk, 1 if renormalize else 0, _ptr(ids), _ptr(w),
                                _stream(stream))
    _native.check("moe_router_topk", rc)
    return ids, w


def moe_quantize_act(x, act_quant: str, scale: float = 1.0, stream=None):
    """Activation quantiser of the W4A4 / W4A8 schemes on rows x [rows, K]
    (bf16 or float32, K % 32 == 0).  "mxfp4": ``(packed uint8 [rows, K/2],
    scale bytes uint8 [rows, K/32])``; "fp8": ``(e4m3 codes uint8 [rows, K], None)``."""
    rows, K = x.shape
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, (rows, K))
    aq = _AQ[act_quant]
    if aq == MOE_AQ_MXFP4:
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
        qs = torch.empty((rows, K // 32), dtype=torch.uint8, device=x.device)
    else:
        q = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
        qs = None
    rc = _lib().moe_quantize_act(aq, _ptr(x), 1 if x.dtype == torch.float32 else 0, rows, K, float(scale), _ptr(q),
                                 _ptr(qs), _stream(stream))
    _native.check("moe_quantize_act", rc)
    return q, qs


def moe_read_status(d: MoeDims, workspace, stream=None) -> int:
    """Read and clear the device status word of a workspace (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    rc = _lib().moe_read_status(ctypes.byref(d), _ptr(workspace), ctypes.byref(v), _stream(stream))
    _native.check("moe_read_status", rc)
    return int(v.value)
