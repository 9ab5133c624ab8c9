"""ctypes view of ``libmoe_a16w4.so`` (declarations of include/moe_a16w4.h)."""

from __future__ import annotations

import ctypes
import os

from . import build as _build

MOE_OK = 0
ERRORS = {
    -1: "MOE_ERR_NULL",
    -2: "MOE_ERR_BAD_DIMS",
    -3: "MOE_ERR_ALIGN",
    -4: "MOE_ERR_UNSUPPORTED_ACT",
    -5: "MOE_ERR_WORKSPACE",
    -6: "MOE_ERR_CUDA",
    -7: "MOE_ERR_DEVICE",
}
MOE_ACT_SWIGLU = 0
MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL = 0, 1, 2
MOE_STATUS_WAIT_TIMEOUT, MOE_STATUS_BAD_INDEX, MOE_STATUS_NAN_SCALE = 0x1, 0x2, 0x4
MOE_AQ_NONE, MOE_AQ_MXFP4, MOE_AQ_FP8 = 0, 1, 2

# Every symbol the header declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class MoeDims(ctypes.Structure):
    _fields_ = [("E", _i32), ("H", _i32), ("I", _i32), ("topk", _i32), ("T", _i32), ("act", _i32), ("path", _i32)]


_DimsP = ctypes.POINTER(MoeDims)


class MoeOptions(ctypes.Structure):
    _fields_ = [("w13_bias", _vp), ("w2_bias", _vp), ("expert_map", _vp), ("global_num_experts", _i32),
                ("router_weight_on_input", _i32), ("act_quant", _i32), ("w13_input_scale", ctypes.c_float),
                ("w2_input_scale", ctypes.c_float), ("swiglu_limit", ctypes.c_float)]


_OptP = ctypes.POINTER(MoeOptions)

SIGNATURES = {
    "moe_workspace_bytes": (ctypes.c_size_t, [_DimsP]),
    "moe_a16w4_mxfp4": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "moe_a16w4_int4g32": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "moe_a16w4_mxfp4_ex": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _OptP, _vp, _vp,
                                          ctypes.c_size_t, _vp]),
    "moe_a16w4_int4g32_ex": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _OptP, _vp, _vp,
                                            ctypes.c_size_t, _vp]),
    "requant_mxfp4_to_int4g32": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp]),
    "requant_mxfp4_to_int4g32_bf16s": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp]),
    "moe_a16w4_int4g32_bf16s": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                               ctypes.c_size_t, _vp]),
    "moe_a16w4_int4g32_bf16s_ex": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _OptP, _vp, _vp,
                                                  ctypes.c_size_t, _vp]),
    "moe_route": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_router_topk": (ctypes.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_read_status": (ctypes.c_int, [_DimsP, _vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "moe_set_wait_limit": (ctypes.c_int, [ctypes.c_uint64, _i32]),
    "moe_a16w4_mxfp4_noalloc": (ctypes.c_int, [_DimsP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_noalloc_read_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _vp]),
    "moe_quantize_act": (ctypes.c_int, [_i32, _vp, _i32, ctypes.c_int64, _i32, ctypes.c_float, _vp, _vp, _vp]),
    "moe_set_timing_events": (ctypes.c_int, [ctypes.POINTER(_vp), _i32]),
    "moe_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_abi_version": (ctypes.c_int, []),
}

_libs = {}
_use_checked = False


def load(path: str | None = None, checked: bool | None = None) -> ctypes.CDLL:
    """Load the library (built in-tree).  Raises if it has not been built.

    ``checked`` selects the bounds-checked build (``libmoe_a16w4_check.so``);
    by default the one chosen with ``use_checked`` (the regular build unless
    changed)."""
    if checked is None:
        checked = _use_checked
    key = path or checked
    if key in _libs:
        return _libs[key]
    path = path or _build.lib_path(checked)
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m mxfp4_weight_only_gb300.build` "
            "(there is no fallback implementation)"
        )
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _libs[key] = lib
    return lib


def use_checked(on: bool) -> None:
    """Route the package's calls to the bounds-checked build (True) or the
    regular one (False)."""
    global _use_checked
    _use_checked = bool(on)


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load().moe_error_string(code).decode()
        super().__init__(f"{fn} failed: {ERRORS.get(code, code)} ({msg})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != MOE_OK:
        raise MoeError(fn, code)
